"""Maximum sizes and zero-length calls, against the oracle.

- The longest prompt the library takes (KVEVICT_MAX_PREFILL = 16384 tokens)
  with head_dim 128 and a budget of 8000 rows: 128 scorer blocks per row, the
  bulk selection's largest sort, and decode rows whose metadata takes the
  whole shared-memory ring.
- head_dim 64 with a budget of 4080 rows, near the largest metadata stride
  the ring holds at that width (4092).
- A sequential prompt of 6000 tokens: 3000-odd decode steps inside the prompt,
  all in one launch, with a pyramid whose rows take both metadata layouts.
- Calls of length zero (a prompt of 0 tokens, 0 decode steps) change nothing.
"""
import numpy as np
import pytest

from workloads import Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from test_gpu_parity import all_rows, compare_rows, run_gpu  # noqa: E402

CASES = [
    Workload("max_prefill_d128", batch=1, n_layers=1, n_kv_heads=2, head_dim=128,
             avg_budget=8000, beta=1.0, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=16500,
             rope_theta=500000.0, gumbel_seed=71, key_seed=71, prefill=16384, decode=8),
    Workload("max_budget_d64", batch=1, n_layers=1, n_kv_heads=2, head_dim=64,
             avg_budget=4080, beta=1.0, n_sink=4, tau_init=0.5, tau_end=0.5, anneal_steps=0,
             rope_theta=10000.0, gumbel_seed=72, key_seed=72, prefill=4200, decode=16, recent=8),
    Workload("long_sequential_prompt", batch=1, n_layers=2, n_kv_heads=1, head_dim=64,
             avg_budget=2000, beta=1.5, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=6100,
             rope_theta=500000.0, gumbel_seed=73, key_seed=73, prefill=6000, decode=12,
             prefill_mode=1),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_max_sizes_all_rows(wl):
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    import oracle as orc
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rows = all_rows(wl)
    res = run_gpu(kvx, wgpu, wl, rows, segments=[wl.decode // 2])
    reps = compare_rows(orc, wl, rows, *res)
    assert sum(r.evictions for r in reps.values()) > 0


def test_zero_length_calls_change_nothing():
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = Workload("zero_lengths", batch=1, n_layers=2, n_kv_heads=2, head_dim=128, avg_budget=16,
                  beta=1.0, n_sink=4, tau_init=1.0, tau_end=1.0, anneal_steps=0,
                  rope_theta=10000.0, gumbel_seed=5, key_seed=74, prefill=20, decode=30)
    pre, dec = wgpu.device_inputs(wl)
    rows = all_rows(wl)

    a = kvx.from_workload(wl)
    a.prefill(pre[:, :, :, :0])    # a prompt of 0 tokens
    assert a.next_pos == 0
    a.decode(dec[:0])              # 0 decode steps
    assert a.next_pos == 0
    a.decode(dec)
    a.decode(dec[:0])
    assert a.next_pos == wl.decode
    got = {r: a.read_state(*r) for r in rows}
    a.close()

    b = kvx.from_workload(wl)
    b.decode(dec)
    want = {r: b.read_state(*r) for r in rows}
    b.close()
    for r in rows:
        for x, y in zip(got[r], want[r]):
            assert np.array_equal(x, y), f"row {r}"
