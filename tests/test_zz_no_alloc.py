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

RTOL, ATOL = 1e-4, 1e-6   # the score tolerance of the parity tests


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
        np.testing.assert_allclose(got, want, rtol=RTOL, atol=ATOL, err_msg=f"call {i}")
    assert torch.cuda.mem_get_info()[0] == free_before, "a later call took device memory"


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
