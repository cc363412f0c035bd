"""Window + landmark sparse attention forward on GB300 (sm_103a).

The CUDA kernels live in ``libmsa.so`` (C ABI: ``include/msa.h``); the
binding and the user-facing calls are loaded on first use, so importing the
package (e.g. for ``workloads``) does not require the library.  Once used,
a missing library raises ImportError: there is no CPU fallback.
"""
from .workloads import WORKLOADS, Workload, generate, sample_rows  # noqa: F401

__all__ = ["WORKLOADS", "Workload", "generate", "sample_rows", "msa_attention",
           "ring_attention", "band_attention", "topk_attention", "compressed_attention", "landmarks",
           "msa_attention_backward", "msa_attention_trainable", "msa_attention_host",
           "compressed_attention_backward",
           "SparseLandmarkAttention", "binding"]


def __getattr__(name):
    if name in ("msa_attention", "ring_attention", "band_attention", "topk_attention",
                "compressed_attention", "landmarks", "msa_attention_backward",
                "msa_attention_trainable", "msa_attention_host", "SparseLandmarkAttention",
                "compressed_attention_backward"):
        from . import api
        return getattr(api, name)
    if name == "binding":
        from . import _binding
        return _binding
    raise AttributeError(name)
