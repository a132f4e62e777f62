"""The benchmark's algorithmic byte count, on the CPU, against a per-head-step loop.

bench.py's `achieved` GB/s divides these bytes by the decode time, so the count
is pinned here to the per-head-step formula written out term by term: with n
rows kept before the append and evicted slot e, an evicting step reads the n+1
keys (2D bytes each), writes the n-e keys that move, reads and writes the n+1
scores, reads the n+1 Gumbel values and moves n-e Gumbel values and positions;
a step within budget reads the n+1 keys, writes the new key, reads and writes
the n+1 scores and writes the new row's Gumbel value and position.
"""
import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _loop_count(D, prefill, budgets, ev):
    T, B, L, H = ev.shape
    total = 0
    for t in range(T):
        p = prefill + t
        for b in range(B):
            for l in range(L):
                n = min(p, budgets[l])
                for h in range(H):
                    e = int(ev[t, b, l, h])
                    if e >= 0:
                        total += (n + 1) * 2 * D + (n - e) * 2 * D + 8 * (n + 1) + 4 * (n + 1) + 12 * (n - e)
                    else:
                        total += (n + 1) * 2 * D + 2 * D + 8 * (n + 1) + 8
    return total


@pytest.mark.parametrize("D, prefill, budgets", [(128, 0, [5, 3]), (64, 7, [6, 4, 9]), (128, 20, [8])])
def test_algorithmic_bytes_match_the_per_step_formula(D, prefill, budgets):
    import bench
    rng = np.random.default_rng(D + prefill)
    T, B, H, L = 12, 2, 3, len(budgets)
    ev = np.full((T, B, L, H), -1, dtype=np.int32)
    for t in range(T):
        for l in range(L):
            n = min(prefill + t, budgets[l])
            if n + 1 > budgets[l]:                      # over budget: some slot 0..n goes
                ev[t, :, l, :] = rng.integers(0, n + 1, size=(B, H))
    wl = SimpleNamespace(head_dim=D, prefill=prefill)
    got = bench.algorithmic_bytes(wl, budgets, torch.from_numpy(ev))
    assert got == _loop_count(D, prefill, budgets, ev)
