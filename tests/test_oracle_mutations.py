"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the C oracle (text substitution;
the real source is not touched), compiles it, points the oracle module at
the copy, and runs a battery of the pin checks: at least one must fail.  The
unmodified oracle passes the same battery.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "msa_oracle.c")

MUTATIONS = [
    ("window edge off by one", "int64_t j_lo = i - window + 1;", "int64_t j_lo = i - window;"),
    ("future key attended", "int64_t j_hi = i;", "int64_t j_hi = i + 1;"),
    ("straddling block visible", "if ((l + 1) * B <= pos - window + 1) count = l + 1;",
     "if (l * B <= pos - window + 1) count = l + 1;"),
    ("landmark dropped from the denominator",
     "double p = exp(s_lm[l] - m);\n                    denom += p;",
     "double p = exp(s_lm[l] - m);"),
    ("landmark score unscaled", "s_lm[l] = scale * dot;", "s_lm[l] = dot;"),
    ("interleaved GQA mapping", "const int c = h / group;", "const int c = h % Hkv;"),
    ("lse without the max shift", "lse[(int64_t)h * n_rows + r] = m + log(denom);",
     "lse[(int64_t)h * n_rows + r] = log(denom);"),
    ("block sum not divided by B", "out[l * row + e] = s / (double)B;",
     "out[l * row + e] = s / (double)(B + 1);"),
    ("value read from K", "o[e] += p * oracle_load(v, voff + e, dtype);",
     "o[e] += p * oracle_load(k, voff + e, dtype);"),
    ("merge weight without the total", "const double wgt = exp(l - total);",
     "const double wgt = exp(l - mx);"),
    ("chunk offset ignored", "int64_t koff = ((j_lo + t - kv_start) * Hkv + c) * (int64_t)d;",
     "int64_t koff = ((j_lo + t) * Hkv + c) * (int64_t)d;"),
    ("backward: D not subtracted", "const double ds = p * (dp - Di);",
     "const double ds = p * dp;"),
    ("backward: dK unscaled", "gk[e] += scale * ds * oracle_load(q, qoff + e, dtype);",
     "gk[e] += ds * oracle_load(q, qoff + e, dtype);"),
    ("backward: dV weighted by dS", "gv[e] += p * oracle_load(dout, qoff + e, dtype);",
     "gv[e] += ds * oracle_load(dout, qoff + e, dtype);"),
    ("backward: last row of a key's window dropped",
     "const int64_t i_hi = j + window - 1 < n - 1 ? j + window - 1 : n - 1;",
     "const int64_t i_hi = j + window - 2 < n - 1 ? j + window - 2 : n - 1;"),
    ("backward: first row seeing a landmark skipped",
     "for (int64_t i = (l + 1) * B + window - 1; i < n; ++i)",
     "for (int64_t i = (l + 1) * B + window; i < n; ++i)"),
    ("backward: landmark gradient not divided by B",
     "dk[j * row_kv + e] += dk_lm[l * row_kv + e] / (double)B;",
     "dk[j * row_kv + e] += dk_lm[l * row_kv + e];"),
]


def battery(mod):
    """Run the pin checks against `mod`; return the names that failed."""
    checks = {
        "bruteforce 16/4/3": lambda: P.test_p1_bruteforce(mod, 16, 4, 3),
        "bruteforce 64/8/9": lambda: P.test_p1_bruteforce(mod, 64, 8, 9),
        "bruteforce 48/6/1": lambda: P.test_p1_bruteforce(mod, 48, 6, 1),
        "causal sdpa": lambda: P.test_p2_causal_special_case(mod, 33, 4, 2, 8),
        "merge of chunks": lambda: P.test_p3_merge_of_chunks_equals_single_pass(mod, 5),
        "empty parts": lambda: P.test_p3_empty_parts(mod),
        "convexity": lambda: P.test_p4_weights_are_a_convex_combination(mod, 16, 4, 3),
        "uniform weights": lambda: P.test_p5a_zero_keys_give_uniform_weights(mod, 64, 8, 9),
        "block centres": lambda: P.test_p5c_position_keys_give_block_centres(mod, 64, 8),
        "count via K=0": lambda: P.test_p6_oracle_count_via_zero_keys(mod),
        "bwd autograd 16/4/3": lambda: P.test_bwd_matches_dense_autograd(mod, 16, 4, 3),
        "bwd autograd 40/5/13": lambda: P.test_bwd_matches_dense_autograd(mod, 40, 5, 13),
        "bwd identities": lambda: P.test_bwd_sum_identities(mod),
    }
    failed = []
    for name, fn in checks.items():
        try:
            fn()
        except (AssertionError, ValueError):
            failed.append(name)
    return failed


@pytest.fixture
def swap_lib():
    saved = oracle._lib
    yield
    oracle._lib = saved


def _compile(src_text, tmp_path, tag):
    c = tmp_path / f"mut_{tag}.c"
    so = tmp_path / f"mut_{tag}.so"
    c.write_text(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", "-o", str(so), str(c), "-lm"], check=True)
    return oracle._configure(ctypes.CDLL(str(so)))


def test_unmodified_oracle_passes_the_battery(swap_lib):
    oracle._load()
    assert battery(oracle) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(swap_lib, tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, f"pattern for '{name}' not found"
    # The first occurrence is in the path the mistake names.
    lib = _compile(text.replace(old, new, 1), tmp_path, abs(hash(name)) % 10**8)
    oracle._lib = lib
    failed = battery(oracle)
    assert failed, f"no pin caught: {name}"
