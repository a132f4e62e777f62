"""Checkpoint and resume (kvevict_save_state / kvevict_load_state).

The pages keep the cache state in an object returned by each call (page
"veloxquant_mlx.quantizers.keyformer module", KeyformerState); a snapshot is
that state copied to the host. A run that is saved part-way, loaded into a
fresh handle and continued must match the uninterrupted run bit for bit: the
eviction log of the remaining steps and every row's keys, scores, Gumbel values
and positions (values too, for a value-carrying cache). A snapshot taken right
after a step still has that step's compaction pending; saving applies it first,
which the next step would otherwise do, so the results are the same.
Snapshots that do not fit the handle are refused and leave it unchanged.
"""
import numpy as np
import pytest

from workloads import Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from test_gpu_parity import all_rows  # noqa: E402

WL = Workload("ckpt", batch=2, n_layers=3, n_kv_heads=2, head_dim=128, avg_budget=40, beta=1.5,
              n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=90, rope_theta=500000.0,
              gumbel_seed=99, key_seed=81, prefill=57, decode=70, recent=2)
WL64 = Workload("ckpt_d64_values", batch=1, n_layers=2, n_kv_heads=3, head_dim=64, avg_budget=30,
                beta=1.5, n_sink=2, tau_init=0.5, tau_end=0.5, anneal_steps=0, rope_theta=10000.0,
                gumbel_seed=5, key_seed=82, prefill=45, decode=50)


def _state(h, wl, values=False):
    out = {}
    for r in all_rows(wl):
        st = list(h.read_state(*r))
        if values:
            st.append(h.read_values(*r))
        out[r] = st
    return out


def _same(a, b):
    for r in a:
        for x, y in zip(a[r], b[r]):
            assert np.array_equal(x, y), f"row {r}"


def _values(dec, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(dec.shape, generator=g, device="cuda").to(torch.float16)


@pytest.mark.parametrize("wl,values", [(WL, False), (WL64, True)], ids=["keys", "values_d64"])
@pytest.mark.parametrize("cut", [0, 1, 23])
def test_resume_equals_uninterrupted(wl, values, cut):
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pre, dec = wgpu.device_inputs(wl)
    vpre = _values(pre, 1) if values else None
    vdec = _values(dec, 2) if values else None
    T = wl.decode
    shape = (T - cut, wl.batch, wl.n_layers, wl.n_kv_heads)

    def start(h):
        if values:
            h.prefill(pre, values=vpre)
            if cut:
                h.decode(dec[:cut], values=vdec[:cut])
        else:
            h.prefill(pre)
            if cut:
                h.decode(dec[:cut])

    def finish(h):
        ev = torch.full(shape, -7, dtype=torch.int32, device="cuda")
        if values:
            h.decode(dec[cut:], ev, values=vdec[cut:])
        else:
            h.decode(dec[cut:], ev)
        return ev.cpu().numpy()

    a = kvx.from_workload(wl, with_values=values)
    start(a)
    snap = a.save_state()
    assert snap.size == a.state_bytes()
    ev_a = finish(a)
    want = _state(a, wl, values)

    b = kvx.from_workload(wl, with_values=values)
    b.load_state(snap)
    assert b.next_pos == wl.prefill + cut
    ev_b = finish(b)
    assert np.array_equal(ev_a, ev_b)
    _same(want, _state(b, wl, values))
    b.check()

    a.reset()                        # the same handle, loaded again
    a.load_state(snap)
    ev_c = finish(a)
    assert np.array_equal(ev_a, ev_c)
    _same(want, _state(a, wl, values))
    a.close()
    b.close()


def test_mismatched_or_corrupt_snapshot_is_refused():
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pre, dec = wgpu.device_inputs(WL)
    a = kvx.from_workload(WL)
    a.prefill(pre)
    a.decode(dec[:10])
    snap = a.save_state()

    b = kvx.from_workload(WL)
    b.prefill(pre)                   # b's own state, which a refused load must leave alone
    before = _state(b, WL)
    for bad in (snap[:100], snap[:-1]):
        with pytest.raises(kvx.KVEvictError) as err:
            b.load_state(bad)
        assert err.value.code == kvx.ERR_INVALID_ARG
    garbled = snap.copy()
    garbled[:8] = 0
    with pytest.raises(kvx.KVEvictError) as err:
        b.load_state(garbled)
    assert "not a kvevict snapshot" in str(err.value)
    assert b.next_pos == WL.prefill
    _same(before, _state(b, WL))

    for field, value in (("gumbel_seed", 100), ("avg_budget", 41), ("recent", 1), ("tau_end", 2.5),
                         ("rope_theta", 10000.0)):
        other = kvx.from_workload(WL.scaled(**{field: value}))
        with pytest.raises(kvx.KVEvictError) as err:
            other.load_state(snap)
        assert err.value.code == kvx.ERR_INVALID_ARG, field
        assert other.next_pos == 0
        other.close()
    a.close()
    b.close()


def test_empty_snapshot_allows_a_prompt():
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pre, dec = wgpu.device_inputs(WL)
    a = kvx.from_workload(WL)
    snap = a.save_state()            # nothing in it yet
    b = kvx.from_workload(WL)
    b.prefill(pre)
    b.load_state(snap)               # back to empty
    assert b.next_pos == 0
    b.prefill(pre)
    b.decode(dec)
    a.prefill(pre)
    a.decode(dec)
    _same(_state(a, WL), _state(b, WL))
    a.close()
    b.close()
