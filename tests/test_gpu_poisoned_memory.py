"""Parity with every byte of fresh device memory set to NaN first.

cudaMalloc does not clear memory, so the cache arena, the prompt scratch and
the Gumbel table start with whatever an earlier allocation left there. These
tests fill a large block with 0xFF bytes (NaN as fp16 and as f32, -1 as i32),
hand it back to the driver, then create the handle and run the workload, so
that the library's allocations very likely land on poisoned pages. A kernel
that read a row, score or table entry it never wrote would turn a cache
row's scores into NaN and fail parity (or raise the bad-index error word).
"""
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from test_gpu_parity import all_rows, compare_rows, run_gpu, sampled_rows  # noqa: E402

CASES = [
    Workload("poison_pyramid_anneal", batch=2, n_layers=3, n_kv_heads=2, head_dim=128,
             avg_budget=24, beta=2.0, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=40,
             rope_theta=10000.0, gumbel_seed=7, key_seed=51, prefill=37, decode=60),
    Workload("poison_sequential_tova", batch=1, n_layers=2, n_kv_heads=2, head_dim=64,
             avg_budget=20, beta=1.0, n_sink=2, tau_init=0.0, tau_end=0.0, anneal_steps=0,
             rope_theta=10000.0, gumbel_seed=0, key_seed=52, prefill=50, decode=30, recent=2,
             score_mode=1, prefill_mode=1),
    Workload("poison_long_rows_mixed", batch=8, n_layers=2, n_kv_heads=32, head_dim=64,
             avg_budget=2048, beta=1.5, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=3200,
             rope_theta=500000.0, gumbel_seed=22, key_seed=53, prefill=3100, decode=24),
    workloads.KEYFORMER_3B,
]


def _poison(gib=8):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.synchronize()
    free = torch.cuda.mem_get_info()[0]
    n = min(gib << 30, free // 2)
    block = torch.full((n // 2,), -1, dtype=torch.int16, device="cuda")   # every byte 0xFF
    torch.cuda.synchronize()
    del block
    torch.cuda.empty_cache()                                              # back to the driver


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_parity_on_poisoned_memory(wl):
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    import oracle as orc
    _poison()
    heads = wl.batch * wl.n_layers * wl.n_kv_heads
    rows = all_rows(wl) if heads <= 16 else sampled_rows(wl, k=8, seed=3)
    res = run_gpu(kvx, wgpu, wl, rows, segments=[wl.decode // 2])
    reps = compare_rows(orc, wl, rows, *res)
    assert sum(r.evictions for r in reps.values()) > 0
