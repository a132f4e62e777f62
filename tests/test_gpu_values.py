"""Value rows on the CUDA path against the oracle carrying the same value rows.

Page "veloxquant_mlx.quantizers.keyformer module": KeyformerState.values holds
one fp16 value row per kept token, keyformer_update appends it with its key and
moves it with the key when an earlier row is evicted (step 3), and
keyformer_get_kv returns keys and values together. A value row is never
rotated. Each case runs a value-carrying handle and replays every row on the
oracle with the same value rows: eviction logs and positions as in the key-only
parity, value rows bit-exact. The decisions must also equal a key-only run's
(values never influence them).
"""
import numpy as np
import pytest

from workloads import Workload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CASES = [
    Workload("values_bulk", batch=2, n_layers=2, n_kv_heads=2, head_dim=128, avg_budget=30,
             beta=1.5, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=80, rope_theta=500000.0,
             gumbel_seed=3, key_seed=40, prefill=70, decode=90),
    Workload("values_sequential_tova", batch=1, n_layers=2, n_kv_heads=3, head_dim=64,
             avg_budget=20, beta=1.0, n_sink=2, tau_init=0.0, tau_end=0.0, anneal_steps=0,
             rope_theta=10000.0, gumbel_seed=0, key_seed=41, prefill=45, decode=60, recent=2,
             score_mode=1, prefill_mode=1),
    Workload("values_decode_only", batch=1, n_layers=1, n_kv_heads=4, head_dim=128,
             avg_budget=40, beta=1.0, n_sink=4, tau_init=2.0, tau_end=2.0, anneal_steps=0,
             rope_theta=500000.0, gumbel_seed=9, key_seed=42, prefill=0, decode=200),
]


def _random_cases(k=8):
    """Seeded random small configurations (as in the random-configuration parity
    tests) long enough that every layer evicts several times."""
    import oracle as orc
    from test_gpu_random_configs import _cases
    out = []
    for w in _cases(n=64, seed=77):
        if w.prefill + w.decode > max(orc.budgets(w.n_layers, w.avg_budget, w.n_sink, w.beta)) + 5:
            out.append(w.scaled(name=w.name + "_values"))
        if len(out) == k:
            break
    return out


@pytest.fixture(scope="module")
def kvx():
    import kv_cache_attention_02_gb300 as k
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    k.lib()
    return k


@pytest.fixture(scope="module")
def wgpu():
    from workloads import gpu
    gpu.lib()
    return gpu


@pytest.mark.parametrize("wl", CASES + _random_cases(), ids=lambda w: w.name)
@pytest.mark.parametrize("path", ["multi", "step"])
def test_values_match_oracle(kvx, wgpu, orc, wl, path):
    from test_gpu_parity import all_rows, compare_rows, run_gpu
    rows = all_rows(wl)
    seg = [wl.decode // 3]
    res = run_gpu(kvx, wgpu, wl, rows, segments=seg, mode=path, with_values=True)
    reps = compare_rows(orc, wl, rows, *res, with_values=True)
    assert sum(r.evictions for r in reps.values()) > 0
    moved = sum(int(np.sum(st[3] != np.arange(len(st[3])))) for st in res[2].values())
    assert moved > 0
    # the same decisions, bit for bit, as a key-only handle run the same way (a
    # launch boundary and the checkpoint reads, which apply the pending
    # compaction, change which threads sum which rows, so the scores of runs
    # cut differently may differ in the last bit)
    plain = run_gpu(kvx, wgpu, wl, rows, segments=seg, mode=path)
    assert np.array_equal(plain[1], res[1])
    if res[4] is not None:
        assert np.array_equal(plain[4], res[4])
    for r in rows:
        for x, y in zip(plain[2][r], res[2][r][:4]):
            assert np.array_equal(x, y)
