"""Write attended_counts.json: attended-set sizes per head for each workload.

Calls only the CPU oracle.  With K = 0 every score is 0, so the oracle's lse
for a row is ln |attended set| and exp(lse) recovers the count; summing over
rows gives the per-head totals, which fix the useful-FLOP numerator
4 * d * Hq * total of every throughput figure.

Run from the repository root:  python tests/golden/make_counts.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from long_context_sparse_landmark_gb300.workloads import WORKLOADS  # noqa: E402


def main():
    per_head = {}
    for name, wl in WORKLOADS.items():
        q = np.ones((wl.n, 1, 1), dtype=np.float32)
        k = np.zeros((wl.n, 1, 1), dtype=np.float32)
        if wl.band_block > 0:
            _, lse = oracle.attn_band(q, k, k, wl.band_block, wl.band_half, 1.0)
        elif wl.global_every > 0:
            _, lse = oracle.attn_compressed(q, k, k, wl.window, wl.block, wl.global_rows(), 1.0)
        elif wl.top_k > 0:
            # every score 0: the count does not depend on which blocks win
            scores = oracle.block_scores(q, k, wl.G, wl.window)
            sel, cnt = oracle.select_top_k(scores, wl.top_k)
            _, lse = oracle.attn_select(q, k, k, wl.window, wl.G, sel, cnt, 1.0)
        else:
            _, lse = oracle.attn(q, k, k, wl.window, wl.G, 1.0)
        counts = np.rint(np.exp(lse[0])).astype(np.int64)
        per_head[name] = int(counts.sum())
        print(name, per_head[name], flush=True)
    out = {
        "what": ("sum over rows of |attended set| per head (window + visible landmarks, "
                 "the block band, window + selected blocks, or window + compression tokens "
                 "and global rows)"),
        "written_by": "tests/golden/make_counts.py (CPU oracle, K = 0 so lse = ln count)",
        "per_head": per_head,
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)),
                           "attended_counts.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
