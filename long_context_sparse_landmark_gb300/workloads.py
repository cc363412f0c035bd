"""Seeded synthetic workloads (shapes and input generators only).

This module holds no attention arithmetic: it names the workloads the
library is measured and checked on, draws their Q/K/V from a seeded
generator, and picks the sampled rows that large parity checks evaluate.
Both the CUDA path's tests/benchmark and the CPU oracle's tests read their
inputs from here, and from nothing else.

Shapes follow the pages: a 70B-style layer has 64 query heads, 8 KV heads of
dimension 128 ("Training at 1M+ Token Context", memory paragraph), and the
million-token Flash-MSA setting uses a 4096-token window and 512 landmarks
("Scaling GPU Cluster for Million Token Context", section "Why Sparse
Attention Changes the Game").  Values are i.i.d. N(0,1); no dataset is used.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n: int              # tokens (batch 1)
    Hq: int             # query heads
    Hkv: int            # key/value heads (GQA groups)
    d: int              # head dimension
    window: int         # w: keys i-w < j <= i
    G: int              # landmarks (0 = none)
    dtype: str          # "f32" or "bf16" (Q, K, V storage)
    outliers: bool = False   # 1% of K rows get one N(0, variance 2) bias each
    ring_chunks: int = 0     # > 0: KV split into this many contiguous chunks
    seed: int = 0
    band_block: int = 0      # > 0: block-band mask (blocks of this size) instead
    band_half: int = 0       #      of window + landmarks; half-width in blocks
    top_k: int = 0           # > 0: window + the top_k landmark-scored key blocks
                             #      of each 128-row query block (G blocks)
    global_every: int = 0    # > 0: rows c*global_every - 1 are global query rows
                             #      (attend every key j <= i); G gives the
                             #      compression tokens of the other rows

    def global_rows(self):
        """Positions of the global query rows (ascending), as a list."""
        if self.global_every <= 0:
            return []
        return list(range(self.global_every - 1, self.n, self.global_every))

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def block(self) -> int:
        return self.n // self.G if self.G > 0 else 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_n(self, n: int, **kw) -> "Workload":
        fields = dict(self.__dict__)
        fields.update(n=n, **kw)
        return Workload(**fields)


WORKLOADS = {
    # Small fp32 case: 2048 tokens, 4 query heads on 1 KV head, d=64,
    # w=256, 16 landmarks (blocks of 128).
    "pr1_2k": Workload("pr1_2k", 2048, 4, 1, 64, 256, 16, "f32"),
    # 32K tokens, 8 query heads on 1 KV head, w=4096, 512 landmarks
    # (blocks of 64), large-score outliers on 1% of K rows.
    "32k_outliers": Workload("32k_outliers", 32768, 8, 1, 128, 4096, 512,
                             "bf16", outliers=True),
    # One 70B-style layer at 128K tokens: 64 query heads, 8 KV heads.
    "128k_70b_layer": Workload("128k_70b_layer", 131072, 64, 8, 128, 4096,
                               512, "bf16"),
    # Million-token layer: 64/8 heads, w=4096, 512 landmarks (blocks of 2048).
    "1m_70b_layer": Workload("1m_70b_layer", 1048576, 64, 8, 128, 4096, 512,
                             "bf16"),
    # Ring-round emulation: full causal attention (w = n, no landmarks) with
    # the KV sequence split into 8 contiguous chunks of 16384 tokens.
    "ring_128k": Workload("ring_128k", 131072, 32, 8, 128, 131072, 0, "bf16",
                          ring_chunks=8),
    # Block-band mask of the 70B-style layer at 128K tokens: 128-token
    # blocks, each attending the 8 blocks on either side (16 neighbours).
    "band_128k": Workload("band_128k", 131072, 64, 8, 128, 1, 0, "bf16",
                          band_block=128, band_half=8),
    # Top-k block selection on the 70B-style layer at 128K tokens: 256-token
    # chunks (512 blocks), the 50 best-scoring ones per query block plus a
    # 1024-token window ("Million Token Context Window Optimization: What
    # Actually Works", section "The indexing game: smarter context
    # management").
    "topk_128k": Workload("topk_128k", 131072, 64, 8, 128, 1024, 512, "bf16",
                          top_k=50),
    # Compression tokens + global rows on the 70B-style layer at 128K tokens:
    # 4096-token window, one compression token per 32-token sub-block (256
    # per 8192-token chunk, G = 4096), and the last row of every 8192-token
    # chunk a global row attending all earlier keys ("Training at 1M+ Token
    # Context", Block-Sparse Flash Attention paragraph).
    "compress_128k": Workload("compress_128k", 131072, 64, 8, 128, 4096, 4096, "bf16",
                              global_every=8192),
}


def generate(wl: Workload, device="cpu", seed: int | None = None,
             chunk: int = 65536):
    """Draw Q [n,Hq,d], K [n,Hkv,d], V [n,Hkv,d] for a workload.

    One generator seeded with ``seed`` (default ``wl.seed``) draws fp32
    N(0,1) values for Q, then K, then V, each in chunks of ``chunk`` tokens;
    for ``outliers`` it then picks round(0.01 n) positions with ``randperm``
    and adds one N(0, variance 2) scalar per picked position to every K
    element of that token; finally values are rounded to the storage dtype
    (round to nearest even).  The same seed on the same device type gives
    the same bits.
    """
    seed = wl.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    out_dt = wl.torch_dtype

    def draw(H, keep_f32=False):
        t = torch.empty((wl.n, H, wl.d), dtype=torch.float32 if keep_f32 else out_dt,
                        device=device)
        for s in range(0, wl.n, chunk):
            e = min(wl.n, s + chunk)
            x = torch.randn((e - s, H, wl.d), generator=gen, dtype=torch.float32,
                            device=device)
            t[s:e].copy_(x)
        return t

    q = draw(wl.Hq)
    k32 = draw(wl.Hkv, keep_f32=True)
    v = draw(wl.Hkv)
    if wl.outliers:
        m = int(round(0.01 * wl.n))
        idx = torch.randperm(wl.n, generator=gen, device=device)[:m]
        bias = torch.randn((m,), generator=gen, dtype=torch.float32,
                           device=device) * math.sqrt(2.0)
        k32[idx] += bias.view(m, 1, 1)
    k = k32.to(out_dt)
    del k32
    return q, k, v


def sample_rows(wl: Workload, count: int = 2048, seed: int = 1) -> torch.Tensor:
    """A fixed, sorted set of row indices for sampled parity checks.

    Rows 0-63 and the last 64; rows around the window edge; for eight
    landmarks the two rows where the visible-landmark count steps; for ring
    workloads the rows beside every chunk boundary; the rest uniform from
    ``seed``.
    """
    n, w = wl.n, wl.window
    picked = set(range(min(64, n))) | set(range(max(0, n - 64), n))
    picked |= {r for r in range(w - 2, w + 3) if 0 <= r < n}
    if wl.G > 0:
        B = wl.block
        for l in range(0, wl.G, max(1, wl.G // 8)):
            for r in (w - 1 + l * B - 1, w - 1 + l * B):
                if 0 <= r < n:
                    picked.add(r)
    if wl.ring_chunks > 0:
        c = n // wl.ring_chunks
        for p in range(1, wl.ring_chunks):
            for r in (p * c - 1, p * c, p * c + 1):
                if 0 <= r < n:
                    picked.add(r)
    gen = torch.Generator().manual_seed(seed)
    while len(picked) < min(count, n):
        extra = torch.randint(0, n, (count,), generator=gen).tolist()
        for r in extra:
            if len(picked) >= min(count, n):
                break
            picked.add(int(r))
    return torch.tensor(sorted(picked), dtype=torch.int64)


def to_numpy_bits(t: torch.Tensor):
    """Host numpy view of a tensor: float32 as is, bf16 as uint16 bit patterns."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")
