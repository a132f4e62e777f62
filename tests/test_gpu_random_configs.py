"""Seeded random small configurations, every row against the oracle.

The hand-picked cases cover the edges one at a time; these draws combine them:
head_dim 64 or 128, 1-3 layers / heads / batch rows, sinks 0-5, a recent window
or none, cumulative or current-step scores, bulk or sequential prompts, constant
or annealed tau, and budgets and prompt lengths placed on and around the
64-row tile boundaries of the decode step and the 128-row blocks of the prompt
scorer.

The counts and the seed can be raised for a longer soak without changing the
defaults: KVEVICT_RANDOM_SMALL / KVEVICT_RANDOM_MEDIUM (cases of each kind)
and KVEVICT_RANDOM_SEED (small cases use it, medium cases it + 1).
"""
import os

import numpy as np
import pytest

from workloads import Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from test_gpu_parity import all_rows, assert_same_run, compare_rows, run_gpu, sampled_rows  # noqa: E402

_EDGES = [1, 2, 63, 64, 65, 127, 128, 129, 191, 192]


def _draw(i, rng, orc):
    while True:
        D = int(rng.choice([64, 128]))
        L, H, B = (int(x) for x in rng.integers(1, 4, size=3))
        n_sink = int(rng.integers(0, 6))
        recent = int(rng.choice([0, 0, int(rng.integers(1, 6))]))
        floor = n_sink + recent + 1
        avg = int(rng.choice([int(rng.integers(floor + 1, 200)), max(floor + 1, int(rng.choice(_EDGES)))]))
        beta = float(rng.choice([1.0, 1.5, 2.5]))
        budgets = orc.budgets(L, avg, n_sink, beta)
        if min(budgets) < floor:
            continue
        prefill = int(rng.choice([0, int(rng.integers(1, 300)), int(rng.choice(_EDGES))]))
        decode = int(rng.integers(5, 120))
        mode = int(rng.integers(0, 2))
        prefill_mode = int(rng.integers(0, 2)) if prefill else 0
        tau_init = float(np.round(rng.uniform(0, 2), 3))
        tau_end = float(np.round(rng.uniform(0, 2), 3))
        anneal = int(rng.choice([0, int(rng.integers(1, 300))]))
        return Workload(f"random_{i}", batch=B, n_layers=L, n_kv_heads=H, head_dim=D,
                        avg_budget=avg, beta=beta, n_sink=n_sink, tau_init=tau_init,
                        tau_end=tau_end, anneal_steps=anneal,
                        rope_theta=float(rng.choice([10000.0, 500000.0])),
                        gumbel_seed=int(rng.integers(0, 2 ** 32)), key_seed=1000 + i,
                        prefill=prefill, decode=decode, recent=recent, score_mode=mode,
                        prefill_mode=prefill_mode)


_SEED = os.environ.get("KVEVICT_RANDOM_SEED")
_N_SMALL = int(os.environ.get("KVEVICT_RANDOM_SMALL", "32"))
_N_MEDIUM = int(os.environ.get("KVEVICT_RANDOM_MEDIUM", "8"))


def _cases(n=_N_SMALL, seed=int(_SEED) if _SEED else 2026):
    import oracle as orc
    rng = np.random.default_rng(seed)
    return [_draw(i, rng, orc) for i in range(n)]


@pytest.mark.parametrize("wl", _cases(), ids=lambda w: w.name)
def test_random_config_all_rows(wl):
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    import oracle as orc
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rows = all_rows(wl)
    res = run_gpu(kvx, wgpu, wl, rows, segments=[wl.decode // 2])
    compare_rows(orc, wl, rows, *res)
    # the streaming decode kernel gives the same run bit for bit (the library's
    # choice above is the resident one wherever the rows fit)
    assert_same_run(res, run_gpu(kvx, wgpu, wl, rows, segments=[wl.decode // 2], decode_kernel=1))


def _medium_cases(n=_N_MEDIUM, seed=int(_SEED) + 1 if _SEED else 4051):
    """More rows than the decode step runs CTAs (up to 2 per SM), budgets of several
    tiles: every CTA claims several rows per step, of mixed lengths."""
    import oracle as orc
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        while True:
            D = int(rng.choice([64, 128]))
            B, L, H = int(rng.integers(2, 9)), int(rng.integers(2, 9)), int(rng.integers(4, 17))
            if B * L * H < 320:
                continue
            n_sink = int(rng.integers(0, 6))
            recent = int(rng.choice([0, int(rng.integers(1, 9))]))
            avg = int(rng.integers(150, 700))
            beta = float(rng.choice([1.0, 1.6, 2.2]))
            if min(orc.budgets(L, avg, n_sink, beta)) < n_sink + recent + 1:
                continue
            break
        out.append(Workload(f"random_medium_{i}", batch=B, n_layers=L, n_kv_heads=H, head_dim=D,
                            avg_budget=avg, beta=beta, n_sink=n_sink,
                            tau_init=float(np.round(rng.uniform(0, 2), 3)),
                            tau_end=float(np.round(rng.uniform(0, 2), 3)),
                            anneal_steps=int(rng.choice([0, int(rng.integers(100, 1200))])),
                            rope_theta=500000.0, gumbel_seed=int(rng.integers(0, 2 ** 32)),
                            key_seed=2000 + i, prefill=int(rng.integers(0, 900)),
                            decode=int(rng.integers(40, 160)), recent=recent,
                            score_mode=int(rng.integers(0, 2)), prefill_mode=int(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("wl", _medium_cases(), ids=lambda w: w.name)
def test_random_medium_config_sampled_rows(wl):
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    import oracle as orc
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rows = sampled_rows(wl, k=12, seed=5)
    res = run_gpu(kvx, wgpu, wl, rows, segments=[wl.decode // 2])
    compare_rows(orc, wl, rows, *res)
    assert_same_run(res, run_gpu(kvx, wgpu, wl, rows, segments=[wl.decode // 2], decode_kernel=1))
