"""The allocation-free prompt scorer (kvevict_prefill_scores_noalloc).

It exists for callers that cannot call cudaMalloc -- an engine that owns the
whole device heap through its own pool, or a latency-bound loop that cannot
take cudaMalloc's implicit synchronisation -- and keeps its working memory in
a fixed device array inside the library. Its output must equal the scores the
allocating path (kvevict_prefill) gives the same prompt before any eviction,
call after call, although every call reuses the same array.

This file sorts last so that a run stopping at its first failure has already
run every other test.
"""
import numpy as np
import pytest

from workloads import Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

RTOL = 1e-4   # the score tolerance of the parity tests (relative)


def _prompt(S, D, B, L, H, key_seed):
    return Workload("noalloc", batch=B, n_layers=L, n_kv_heads=H, head_dim=D, avg_budget=S + 8,
                    beta=1.0, n_sink=4, tau_init=0.0, tau_end=0.0, anneal_steps=0,
                    rope_theta=500000.0, gumbel_seed=0, key_seed=key_seed, prefill=S, decode=1)


def _allocating_scores(kvx, wl, pre):
    """Scores after kvevict_prefill with every budget above S (nothing evicted)."""
    h = kvx.from_workload(wl)
    h.prefill(pre)
    out = np.stack([h.read_state(b, l, hh)[1]
                    for b in range(wl.batch) for l in range(wl.n_layers)
                    for hh in range(wl.n_kv_heads)])
    h.close()
    return out


def test_noalloc_scores_match_prefill_call_after_call():
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cases = [_prompt(300, 128, 2, 2, 4, key_seed=31),   # several 64-token tiles, ragged tail
             _prompt(77, 64, 1, 3, 2, key_seed=32),     # other head_dim and shape
             _prompt(300, 128, 2, 2, 4, key_seed=33)]   # first shape again, new keys
    inputs = []
    for wl in cases:
        pre, _ = wgpu.device_inputs(wl)
        heads = wl.batch * wl.n_layers * wl.n_kv_heads
        out = torch.full((heads, wl.prefill), float("nan"), dtype=torch.float32, device="cuda")
        inputs.append((wl, pre, out, _allocating_scores(kvx, wl, pre)))
    torch.cuda.synchronize()

    free_before = None
    for i, (wl, pre, out, want) in enumerate(inputs):
        heads = wl.batch * wl.n_layers * wl.n_kv_heads
        keys = pre.view(heads, wl.prefill, wl.head_dim)
        kvx.prefill_scores_noalloc(keys, out)
        torch.cuda.synchronize()
        if i == 0:
            free_before = torch.cuda.mem_get_info()[0]   # after the first call's set-up
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), f"call {i}: output not fully written"
        np.testing.assert_allclose(got, want, rtol=RTOL, atol=0, err_msg=f"call {i}")
    assert torch.cuda.mem_get_info()[0] == free_before, "a later call took device memory"


@pytest.mark.parametrize("S,D,heads,key_seed", [(300, 128, 3, 34), (77, 64, 2, 35)])
def test_noalloc_scores_match_oracle(orc, S, D, heads, key_seed):
    """Raw column sums of the causal softmax against the fp64 oracle's, entry
    by entry, for each head_dim (several 128-row tiles and a ragged tail)."""
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = _prompt(S, D, 1, 1, heads, key_seed=key_seed)
    pre, _ = wgpu.device_inputs(wl)
    keys = pre.view(heads, S, D)
    out = torch.full((heads, S), float("nan"), dtype=torch.float32, device="cuda")
    for _ in range(2):   # two calls in a row, the second over the first's scratch
        kvx.prefill_scores_noalloc(keys, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        for h in range(heads):
            want = orc.prefill_colsum(wl.head_keys(0, 0, h, 0, S))
            np.testing.assert_allclose(got[h], want, rtol=RTOL, atol=0, err_msg=f"head {h}")


def test_noalloc_timeout_is_reported_as_nan():
    """A bounded wait that runs out cannot reach the return code; the call then
    writes NaN to every score instead, and the next call is unaffected (its
    error word starts cleared). The wait is made to run out by the library's
    test hook, which leaves one copy unissued: nothing faults or hangs."""
    import time
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = _prompt(200, 128, 1, 1, 2, key_seed=36)
    pre, _ = wgpu.device_inputs(wl)
    keys = pre.view(2, 200, 128)
    good = torch.zeros((2, 200), dtype=torch.float32, device="cuda")
    kvx.prefill_scores_noalloc(keys, good)
    torch.cuda.synchronize()
    out = torch.zeros((2, 200), dtype=torch.float32, device="cuda")
    assert kvx.lib().kvevict_test_stall_next_step(None) == kvx.OK
    t0 = time.time()
    kvx.prefill_scores_noalloc(keys, out)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert torch.isnan(out).all(), "a timed-out call must leave only NaN"
    assert 0.5 < elapsed < 10.0, f"the stalled call took {elapsed:.1f} s"
    kvx.prefill_scores_noalloc(keys, out)
    torch.cuda.synchronize()
    assert torch.equal(out, good)


def test_noalloc_rejects_sizes_beyond_the_fixed_scratch():
    import kv_cache_attention_02_gb300 as kvx
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    heads, S, D = 1024, 4096, 128   # 2 * 1024 * 4096 floats > 4,194,304
    keys = torch.zeros((heads, 1, D), dtype=torch.float16, device="cuda")
    lib = kvx.lib()
    rc = lib.kvevict_prefill_scores_noalloc(keys.data_ptr(), heads, S, D, keys.data_ptr(), None)
    assert rc == kvx.ERR_INVALID_ARG
    assert "scratch" in kvx.last_error()
