"""The failure path of the decode step, with no fault: a wait that runs out.

Every wait in the kernels is bounded (4 s of %globaltimer); when one runs
out the kernel sets the handle's error word and its CTAs leave their loops,
so the GPU context stays usable. kvevict_test_stall_next_step makes the next
decode launch skip one copy, leaving a barrier that nothing completes. The
tests check that the error reaches the host as DEVICE_CHECK ("bounded wait
ran out") within seconds, that the same context still runs other work, and
that after kvevict_reset the handle reproduces a fresh handle's results bit
for bit.
"""
import time

import numpy as np
import pytest

from workloads import Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

WL = Workload("stall", batch=2, n_layers=2, n_kv_heads=2, head_dim=128, avg_budget=100,
              beta=1.5, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=150,
              rope_theta=500000.0, gumbel_seed=1234, key_seed=61, prefill=200, decode=20)


def _rows(wl):
    return [(b, l, h) for b in range(wl.batch) for l in range(wl.n_layers)
            for h in range(wl.n_kv_heads)]


def _run(kvx, h, pre, dec):
    ev = torch.full((WL.decode, WL.batch, WL.n_layers, WL.n_kv_heads), -7, dtype=torch.int32,
                    device="cuda")
    h.prefill(pre)
    h.decode(dec, ev)
    states = {r: h.read_state(*r) for r in _rows(WL)}
    h.check()
    return ev.cpu().numpy(), states


def test_wait_that_runs_out_is_reported_and_the_handle_recovers():
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pre, dec = wgpu.device_inputs(WL)
    h = kvx.from_workload(WL)
    h.prefill(pre)
    h.test_stall_next_step()
    t0 = time.perf_counter()
    h.step(dec[0])
    with pytest.raises(kvx.KVEvictError) as err:
        h.check()
    elapsed = time.perf_counter() - t0
    assert err.value.code == kvx.ERR_DEVICE_CHECK
    assert "bounded wait ran out" in str(err.value)
    assert elapsed < 10.0, f"the stalled launch took {elapsed:.1f} s"
    with pytest.raises(kvx.KVEvictError):   # the error word stays set until a reset
        h.read_state(0, 0, 0)

    # the context still runs work: a fresh handle, then the reset one, match
    ref = kvx.from_workload(WL)
    want_ev, want = _run(kvx, ref, pre, dec)
    ref.close()
    h.reset()
    got_ev, got = _run(kvx, h, pre, dec)
    h.close()
    assert np.array_equal(got_ev, want_ev)
    for r in _rows(WL):
        for x, y in zip(got[r], want[r]):
            assert np.array_equal(x, y), f"row {r}"


def test_stall_hook_is_one_shot():
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pre, dec = wgpu.device_inputs(WL)
    h = kvx.from_workload(WL)
    h.prefill(pre)
    h.test_stall_next_step()
    h.step(dec[0])
    with pytest.raises(kvx.KVEvictError):
        h.check()
    h.reset()
    h.prefill(pre)
    h.decode(dec)          # no hook armed now: runs clean
    h.check()
    h.close()


def test_prompt_scorer_wait_that_runs_out_is_reported():
    """The same for the tensor-core prompt scorer: with a null handle the hook
    makes the next scorer launch leave one copy unissued, so the MMA issuer's
    bounded wait runs out; the prompt's handle reports DEVICE_CHECK and, after
    a reset, reproduces a fresh handle's results."""
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pre, dec = wgpu.device_inputs(WL)
    h = kvx.from_workload(WL)
    assert kvx.lib().kvevict_test_stall_next_step(None) == kvx.OK
    t0 = time.perf_counter()
    h.prefill(pre)
    with pytest.raises(kvx.KVEvictError) as err:
        h.check()
    elapsed = time.perf_counter() - t0
    assert err.value.code == kvx.ERR_DEVICE_CHECK
    assert elapsed < 10.0, f"the stalled prompt took {elapsed:.1f} s"
    ref = kvx.from_workload(WL)
    want_ev, want = _run(kvx, ref, pre, dec)
    ref.close()
    h.reset()
    got_ev, got = _run(kvx, h, pre, dec)
    h.close()
    assert np.array_equal(got_ev, want_ev)
    for r in _rows(WL):
        for x, y in zip(got[r], want[r]):
            assert np.array_equal(x, y), f"row {r}"


def test_resident_decode_wait_that_runs_out_is_reported():
    """The same for the resident decode step (a call of several steps on rows
    that fit in shared memory): the hook leaves the first CTA's row load
    unissued, its consumers' bounded wait runs out, the helper warp leaves its
    loop on the abort flag, and the handle reports DEVICE_CHECK and recovers
    after a reset."""
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pre, dec = wgpu.device_inputs(WL)
    h = kvx.from_workload(WL)
    assert h.decode_kernel_for(WL.decode) == kvx.DECODE_RESIDENT
    h.prefill(pre)
    h.test_stall_next_step()
    t0 = time.perf_counter()
    h.decode(dec)
    with pytest.raises(kvx.KVEvictError) as err:
        h.check()
    elapsed = time.perf_counter() - t0
    assert err.value.code == kvx.ERR_DEVICE_CHECK
    assert elapsed < 10.0, f"the stalled launch took {elapsed:.1f} s"
    ref = kvx.from_workload(WL)
    want_ev, want = _run(kvx, ref, pre, dec)
    ref.close()
    h.reset()
    got_ev, got = _run(kvx, h, pre, dec)
    h.close()
    assert np.array_equal(got_ev, want_ev)
    for r in _rows(WL):
        for x, y in zip(got[r], want[r]):
            assert np.array_equal(x, y), f"row {r}"
