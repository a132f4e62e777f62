"""CUDA path vs the fp64 oracle, through the C ABI, on seeded synthetic keys.

Small configurations compare every cache row over the whole run (several TMA
tiles, ragged tails, every edge case the method has); the five full-size
workloads run exactly as the benchmark launches them (prompt, then one launch
of all decode steps) and compare, over the whole run, every row of
keyformer_llama3.2-3b and at least one row of every layer of the others.
"""
import concurrent.futures as cf
import json
import os

import numpy as np
import pytest

import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


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


def head_params(orc, wl, l, h):
    budgets = orc.budgets(wl.n_layers, wl.avg_budget, wl.n_sink, wl.beta)
    return orc.HeadParams(D=wl.head_dim, budget=budgets[l], n_sink=wl.n_sink, layer=l, head=h,
                          tau_init=wl.tau_init, tau_end=wl.tau_end, anneal_steps=wl.anneal_steps,
                          theta=wl.rope_theta, seed=wl.gumbel_seed, recent=wl.recent,
                          mode=wl.score_mode, prefill_mode=wl.prefill_mode)


def value_workload(wl):
    """The value rows fed alongside wl's keys: any distinct fp16 payload; the
    key generator with another seed gives one, on the host and the device."""
    return wl.scaled(key_seed=wl.key_seed + 1000)


def run_gpu(kvx, wgpu, wl, rows, segments=None, mode="multi", with_values=False, decode_kernel=0):
    """Run the workload on the GPU; read back the sampled rows (with their
    value rows, as a fifth element, on a value-carrying handle). decode_kernel:
    0 the library's choice, 1 the streaming step, 2 the shared-memory-resident
    step."""
    h = kvx.from_workload(wl, with_values=with_values, decode_kernel=decode_kernel)
    pre, dec = wgpu.device_inputs(wl)
    vpre, vdec = wgpu.device_inputs(value_workload(wl)) if with_values else (None, None)

    def read(r):
        st = h.read_state(*r)
        return st + (h.read_values(*r),) if with_values else st

    after_prefill = {}
    pev = None
    if pre is not None:
        if wl.prefill_mode == 1:
            pev = torch.full((wl.prefill, wl.batch, wl.n_layers, wl.n_kv_heads), -7,
                             dtype=torch.int32, device="cuda")
        h.prefill(pre, pev, values=vpre)
        after_prefill = {r: read(r) for r in rows}
    T = wl.decode
    ev = torch.full((T, wl.batch, wl.n_layers, wl.n_kv_heads), -7, dtype=torch.int32, device="cuda")
    bounds = sorted(set([0, T] + list(segments or [])))
    checkpoints = {r: {} for r in rows}
    for t0, t1 in zip(bounds, bounds[1:]):
        if mode == "multi":
            h.decode(dec[t0:t1], ev[t0:t1], values=vdec[t0:t1] if with_values else None)
        else:
            for t in range(t0, t1):
                h.step(dec[t], ev[t], v_new=vdec[t] if with_values else None)
        if t1 != T:
            for r in rows:
                checkpoints[r][t1] = read(r)
    final = {r: read(r) for r in rows}
    h.check()
    evh = ev.cpu().numpy()
    pevh = pev.cpu().numpy() if pev is not None else None
    h.close()
    del pre, dec, ev, vpre, vdec
    torch.cuda.empty_cache()
    return after_prefill, evh, final, checkpoints, pevh


def compare_rows(orc, wl, rows, after_prefill, evh, final, checkpoints, pevh=None, threads=None,
                 with_values=False):
    """Replay each row on the oracle (threads: the oracle's C calls release the
    interpreter lock) and require every row to agree."""
    import parity
    vwl = value_workload(wl) if with_values else None

    def one(r):
        b, l, hh = r
        keys = wl.head_keys(b, l, hh, 0, wl.positions)
        vals = None
        if with_values:
            v = vwl.head_keys(b, l, hh, 0, wl.positions)
            vals = (v[: wl.prefill] if wl.prefill else None, v[wl.prefill:])
        prm = head_params(orc, wl, l, hh)
        return r, parity.run_row(orc, prm, keys[: wl.prefill] if wl.prefill else None,
                                 keys[wl.prefill:], evh[:, b, l, hh], after_prefill.get(r), final[r],
                                 checkpoints.get(r),
                                 pevh[:, b, l, hh] if pevh is not None else None, values=vals)

    threads = threads or min(16, os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        reports = dict(ex.map(one, rows))
    bad = {r: rep.failures for r, rep in reports.items() if not rep.ok()}
    assert not bad, f"{wl.name}: {bad}"
    return reports


def all_rows(wl):
    return [(b, l, h) for b in range(wl.batch) for l in range(wl.n_layers)
            for h in range(wl.n_kv_heads)]


def sampled_rows(wl, k=6, seed=0):
    rng = np.random.default_rng(seed)
    rows = {(0, 0, 0), (wl.batch - 1, wl.n_layers - 1, wl.n_kv_heads - 1),
            (wl.batch // 2, wl.n_layers // 2, min(1, wl.n_kv_heads - 1))}
    while len(rows) < k:
        rows.add((int(rng.integers(wl.batch)), int(rng.integers(wl.n_layers)),
                  int(rng.integers(wl.n_kv_heads))))
    return sorted(rows)


SMALL = [
    Workload("pyramid_anneal_ragged", batch=2, n_layers=3, n_kv_heads=2, head_dim=128,
             avg_budget=24, beta=2.0, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=40,
             rope_theta=10000.0, gumbel_seed=7, key_seed=3, prefill=37, decode=60),
    Workload("d64_no_sinks", batch=1, n_layers=2, n_kv_heads=3, head_dim=64, avg_budget=9,
             beta=1.0, n_sink=0, tau_init=0.0, tau_end=0.0, anneal_steps=0, rope_theta=10000.0,
             gumbel_seed=0, key_seed=5, prefill=0, decode=50),
    Workload("budget_sinks_plus_one", batch=1, n_layers=1, n_kv_heads=2, head_dim=128,
             avg_budget=5, beta=1.0, n_sink=4, tau_init=0.5, tau_end=0.5, anneal_steps=0,
             rope_theta=500000.0, gumbel_seed=11, key_seed=6, prefill=3, decode=30),
    Workload("prefill_equals_budget", batch=1, n_layers=1, n_kv_heads=2, head_dim=64,
             avg_budget=16, beta=1.0, n_sink=4, tau_init=0.0, tau_end=0.0, anneal_steps=0,
             rope_theta=10000.0, gumbel_seed=0, key_seed=7, prefill=16, decode=20),
    Workload("multi_tile_bulk", batch=1, n_layers=2, n_kv_heads=2, head_dim=128, avg_budget=100,
             beta=1.5, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=150,
             rope_theta=500000.0, gumbel_seed=1234, key_seed=8, prefill=200, decode=150),
    Workload("late_riser_small", batch=1, n_layers=2, n_kv_heads=2, head_dim=128, avg_budget=48,
             beta=1.0, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=300,
             rope_theta=500000.0, gumbel_seed=3, key_seed=9, prefill=0, decode=300,
             late_riser=True),
    workloads.TINY_H2O,
    Workload("recent_window", batch=1, n_layers=2, n_kv_heads=2, head_dim=128, avg_budget=24,
             beta=1.0, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=60, rope_theta=500000.0,
             gumbel_seed=5, key_seed=10, prefill=40, decode=60, recent=5),
    Workload("tova_prompt", batch=2, n_layers=2, n_kv_heads=2, head_dim=64, avg_budget=16,
             beta=1.0, n_sink=2, tau_init=0.0, tau_end=0.0, anneal_steps=0, rope_theta=10000.0,
             gumbel_seed=0, key_seed=11, prefill=30, decode=50, score_mode=1),
    Workload("tova_recent_gumbel", batch=1, n_layers=1, n_kv_heads=3, head_dim=128,
             avg_budget=20, beta=1.0, n_sink=4, tau_init=0.5, tau_end=0.5, anneal_steps=0,
             rope_theta=500000.0, gumbel_seed=12, key_seed=12, prefill=0, decode=80, recent=3,
             score_mode=1),
    Workload("sequential_prompt_pyramid", batch=2, n_layers=3, n_kv_heads=2, head_dim=128,
             avg_budget=40, beta=1.8, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=100,
             rope_theta=500000.0, gumbel_seed=13, key_seed=13, prefill=90, decode=40,
             prefill_mode=1),
    Workload("sequential_prompt_tova_recent", batch=1, n_layers=2, n_kv_heads=2, head_dim=64,
             avg_budget=20, beta=1.0, n_sink=2, tau_init=0.0, tau_end=0.0, anneal_steps=0,
             rope_theta=10000.0, gumbel_seed=0, key_seed=14, prefill=50, decode=30, recent=2,
             score_mode=1, prefill_mode=1),
    # rows long enough (661 keys) that one resident CTA fills an SM's shared
    # memory: the resident step then runs its sixteen-warp form
    Workload("long_rows_sixteen_warps", batch=1, n_layers=2, n_kv_heads=2, head_dim=128,
             avg_budget=600, beta=1.1, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=900,
             rope_theta=500000.0, gumbel_seed=31, key_seed=31, prefill=700, decode=200),
]


_SLOT_KINDS = {"first": 0, "last": 0, "mid": 0}


KERNELS = {"stream": 1, "resident": 2}


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_small_all_rows(kvx, wgpu, orc, wl, kernel):
    rows = all_rows(wl)
    seg = [wl.decode // 3]
    res = run_gpu(kvx, wgpu, wl, rows, segments=seg, decode_kernel=KERNELS[kernel])
    reps = compare_rows(orc, wl, rows, *res)
    assert sum(r.evictions for r in reps.values()) > 0
    for r in reps.values():
        _SLOT_KINDS["first"] += r.evicted_first
        _SLOT_KINDS["last"] += r.evicted_last
        _SLOT_KINDS["mid"] += r.evicted_mid


def test_small_runs_evicted_first_mid_and_last_slots():
    """Across the small configurations the decode step evicted (in agreement
    with the oracle) the first candidate slot n_sink, the last candidate slot
    and slots in between."""
    if sum(_SLOT_KINDS.values()) == 0:
        pytest.skip("run together with test_small_all_rows")
    assert all(v > 0 for v in _SLOT_KINDS.values()), _SLOT_KINDS


def assert_same_run(a, b):
    """Two run_gpu results agree bit for bit: eviction logs, prompt logs and
    every read-back state (prompt, checkpoints, final)."""
    assert np.array_equal(a[1], b[1])
    if a[4] is not None or b[4] is not None:
        assert np.array_equal(a[4], b[4])
    for k in (0, 2):
        assert a[k].keys() == b[k].keys()
        for r in a[k]:
            for x, y in zip(a[k][r], b[k][r]):
                assert np.array_equal(x, y), f"row {r}"
    for r in a[3]:
        assert a[3][r].keys() == b[3][r].keys()
        for t in a[3][r]:
            for x, y in zip(a[3][r][t], b[3][r][t]):
                assert np.array_equal(x, y), f"row {r} after step {t}"


def test_step_path_equals_multistep_path(kvx, wgpu):
    # one launch of every step (the resident kernel) against one launch per
    # step (the streaming kernel): the two kernels visit rows in the same
    # order and agree bit for bit
    wl = SMALL[0]
    rows = all_rows(wl)
    a = run_gpu(kvx, wgpu, wl, rows, mode="multi")
    b = run_gpu(kvx, wgpu, wl, rows, mode="step")
    assert_same_run(a, b)


@pytest.mark.parametrize("wl", [w for w in SMALL if w.decode >= 8][:6] + [SMALL[-1], workloads.LATE_RISER_ANNEAL.scaled(
    name="late_riser_short", batch=2, n_layers=3, decode=600)], ids=lambda w: w.name)
def test_resident_kernel_equals_streaming_kernel(kvx, wgpu, wl):
    """The shared-memory-resident decode step and the streaming one give the
    same eviction logs, keys, scores, Gumbel values and positions, bit for bit,
    with checkpoints cutting the run into several calls."""
    rows = all_rows(wl)
    seg = [1, wl.decode // 3, wl.decode // 3 + 5]
    a = run_gpu(kvx, wgpu, wl, rows, segments=seg, decode_kernel=KERNELS["stream"])
    b = run_gpu(kvx, wgpu, wl, rows, segments=seg, decode_kernel=KERNELS["resident"])
    assert_same_run(a, b)


def test_batched_equals_single_row(kvx, wgpu):
    # keyformer page, keyformer_update_batched: the batched step equals the
    # per-row loop bit for bit. tau = 0 so the Gumbel hash (which keys on the
    # layer and head index) cannot differ between the two layouts.
    wl = Workload("batched", batch=2, n_layers=1, n_kv_heads=3, head_dim=128, avg_budget=40,
                  beta=1.0, n_sink=4, tau_init=0.0, tau_end=0.0, anneal_steps=0,
                  rope_theta=10000.0, gumbel_seed=0, key_seed=21, prefill=50, decode=80)
    pre, dec = wgpu.device_inputs(wl)
    h = kvx.from_workload(wl)
    h.prefill(pre)
    ev = torch.zeros((wl.decode, 2, 1, 3), dtype=torch.int32, device="cuda")
    h.decode(dec, ev)
    full = {(b, hh): h.read_state(b, 0, hh) for b in range(2) for hh in range(3)}
    h.close()
    for b in range(2):
        for hh in range(3):
            one = kvx.KVEvict(batch=1, n_layers=1, n_kv_heads=1, head_dim=128, avg_budget=40,
                              n_sink=4, rope_theta=10000.0, max_prefill=50)
            one.prefill(pre[b:b + 1, :, hh:hh + 1].contiguous())
            ev1 = torch.zeros((wl.decode, 1, 1, 1), dtype=torch.int32, device="cuda")
            one.decode(dec[:, b:b + 1, :, hh:hh + 1].contiguous(), ev1)
            st = one.read_state(0, 0, 0)
            one.close()
            assert np.array_equal(ev1.cpu().numpy()[:, 0, 0, 0], ev.cpu().numpy()[:, b, 0, hh])
            # keys, scores and positions; the frozen Gumbel values themselves
            # are keyed on the head index and differ by design
            for i in (0, 1, 3):
                assert np.array_equal(st[i], full[(b, hh)][i])


# run_host: the inputs come from host memory. Page-locked buffers are moved by
# the library's kernels (the prompt staged by a copy kernel, the decode keys
# read in place), pageable ones by cudaMemcpyAsync chunks that overlap compute;
# a page-locked buffer that does not start on a 16-byte boundary is staged by
# the copy kernel with narrower words. pyramidkv is large enough for several
# chunks of each (the staging buffers hold 256 MiB).
RUN_HOST_CASES = ["multi_tile_bulk", "tova_prompt", "sequential_prompt_pyramid", "d64_no_sinks",
                  "pyramidkv"]
RUN_HOST_MEMORY = [(n, "pinned") for n in RUN_HOST_CASES] + [(n, "pageable") for n in RUN_HOST_CASES] + [
    ("multi_tile_bulk", "pinned_prompt_pageable_decode"), ("tova_prompt", "pageable_prompt_pinned_decode"),
    ("multi_tile_bulk", "pinned_misaligned"), ("d64_no_sinks", "pinned_misaligned")]


def _host_copy(t, pinned, offset_elems=0):
    """A contiguous host copy of t, page-locked or not, starting offset_elems
    elements into its allocation."""
    flat = torch.empty(t.numel() + offset_elems, dtype=t.dtype, pin_memory=pinned)
    view = flat[offset_elems:].view(t.shape)
    view.copy_(t.cpu() if t.is_cuda else t)
    return view


@pytest.mark.parametrize("name,memory", RUN_HOST_MEMORY, ids=[f"{n}-{m}" for n, m in RUN_HOST_MEMORY])
def test_run_host_equals_device_path(kvx, wgpu, name, memory):
    wl = next((w for w in SMALL if w.name == name), None) or workloads.ALL[name]
    pre, dec = wgpu.device_inputs(wl)
    rows = all_rows(wl)
    h = kvx.from_workload(wl)
    if pre is not None:
        h.prefill(pre)
    ev = torch.zeros((wl.decode, wl.batch, wl.n_layers, wl.n_kv_heads), dtype=torch.int32,
                     device="cuda")
    h.decode(dec, ev)
    want = {r: h.read_state(*r) for r in rows}
    h.close()
    pin_pre = memory in ("pinned", "pinned_prompt_pageable_decode", "pinned_misaligned")
    pin_dec = memory in ("pinned", "pageable_prompt_pinned_decode", "pinned_misaligned")
    off = 1 if memory == "pinned_misaligned" else 0   # 2 bytes for keys, 4 for the slots
    h2 = kvx.from_workload(wl)
    pre_h = _host_copy(pre, pin_pre, off) if pre is not None else None
    dec_h = _host_copy(dec, pin_dec, off)
    ev_h = _host_copy(torch.full(tuple(ev.shape), -9, dtype=torch.int32), pin_dec, off)
    h2.run_host(pre_h, dec_h, ev_h)
    assert np.array_equal(ev_h.numpy(), ev.cpu().numpy())
    for r in rows:
        for x, y in zip(h2.read_state(*r), want[r]):
            assert np.array_equal(x, y)
    h2.close()
    del pre, dec
    torch.cuda.empty_cache()


def test_misaligned_device_keys_are_rejected(kvx, wgpu):
    wl = SMALL[0]
    pre, dec = wgpu.device_inputs(wl)
    h = kvx.from_workload(wl)
    shifted = lambda t: torch.empty(t.numel() + 8, dtype=t.dtype, device="cuda")[1:1 + t.numel()].view(t.shape)
    with pytest.raises(kvx.KVEvictError) as err:
        h.prefill(shifted(pre))
    assert err.value.code == kvx.ERR_INVALID_ARG and "16-byte" in str(err.value)
    h.prefill(pre)
    for call in (lambda: h.decode(shifted(dec)), lambda: h.step(shifted(dec[0]))):
        with pytest.raises(kvx.KVEvictError) as err:
            call()
        assert err.value.code == kvx.ERR_INVALID_ARG
    assert h.next_pos == wl.prefill   # nothing ran
    h.decode(dec)
    h.check()
    h.close()


def test_reset_replays_identically(kvx, wgpu):
    wl = SMALL[0]
    pre, dec = wgpu.device_inputs(wl)
    h = kvx.from_workload(wl)
    outs = []
    for _ in range(2):
        h.reset()
        h.prefill(pre)
        ev = torch.zeros((wl.decode, wl.batch, wl.n_layers, wl.n_kv_heads), dtype=torch.int32,
                         device="cuda")
        h.decode(dec, ev)
        outs.append((ev.cpu().numpy(), [h.read_state(*r) for r in all_rows(wl)]))
    h.close()
    assert np.array_equal(outs[0][0], outs[1][0])
    for s0, s1 in zip(outs[0][1], outs[1][1]):
        for x, y in zip(s0, s1):
            assert np.array_equal(x, y)


def test_decode_kernel_choice(kvx):
    """The automatic choice: the resident step for calls of 4+ steps when the
    rows fit in one wave, or two at two CTAs an SM; the streaming step
    otherwise (long rows, value rows, short calls)."""
    cases = [(workloads.TINY_H2O, 256, kvx.DECODE_RESIDENT),
             (workloads.LATE_RISER_ANNEAL, 4096, kvx.DECODE_RESIDENT),
             (workloads.KEYFORMER_3B, 2048, kvx.DECODE_STREAM),   # 513-key rows: 1 CTA an SM, 2 waves
             (workloads.PYRAMIDKV, 2048, kvx.DECODE_STREAM),      # budget 1019: too long to be resident
             (workloads.TINY_H2O, 3, kvx.DECODE_STREAM),          # a short call
             (workloads.TINY_H2O, 1, kvx.DECODE_STREAM)]
    for wl, T, want in cases:
        h = kvx.from_workload(wl.scaled(prefill=0))
        assert h.decode_kernel_for(T) == want, (wl.name, T)
        h.close()
    h = kvx.from_workload(workloads.TINY_H2O, with_values=True)
    assert h.decode_kernel_for(256) == kvx.DECODE_STREAM
    h.close()
    h = kvx.from_workload(workloads.TINY_H2O, decode_kernel=kvx.DECODE_RESIDENT)
    assert h.decode_kernel_for(1) == kvx.DECODE_RESIDENT
    h.close()
    with pytest.raises(kvx.KVEvictError) as err:   # rows too long to be resident
        kvx.from_workload(workloads.PYRAMIDKV.scaled(prefill=0), decode_kernel=kvx.DECODE_RESIDENT)
    assert err.value.code == kvx.ERR_INVALID_ARG


def test_state_errors(kvx, wgpu):
    wl = SMALL[3]
    pre, dec = wgpu.device_inputs(wl)
    h = kvx.from_workload(wl)
    h.step(dec[0])
    with pytest.raises(kvx.KVEvictError) as ei:
        h.prefill(pre)
    assert ei.value.code == kvx.ERR_BAD_STATE
    with pytest.raises(kvx.KVEvictError) as ei:
        h.read_state(0, 5, 0)
    assert ei.value.code == kvx.ERR_INVALID_ARG
    h.close()


@pytest.mark.parametrize("wl", list(workloads.ALL.values()), ids=lambda w: w.name)
def test_gpu_keygen_matches_host(wgpu, wl):
    rows = sampled_rows(wl, k=4, seed=1)
    pre, dec = wgpu.device_inputs(wl)
    for b, l, h in rows:
        want = wl.head_keys(b, l, h, 0, wl.positions)
        got = np.concatenate(
            ([pre[b, l, h].cpu().numpy().view(np.uint16)] if pre is not None else [])
            + [dec[:, b, l, h].cpu().numpy().view(np.uint16)])
        assert np.array_equal(got, want)
    del pre, dec
    torch.cuda.empty_cache()


# More rows than the decode step runs CTAs (two per SM at most), so every CTA
# claims several rows in turn; rows of one CTA differ in budget and so in tile
# count. Rows longer than one ring stage per metadata array (budget above 2044
# at head_dim 64, above 4092 at head_dim 128) take the whole ring for their
# metadata, and the mixed case alternates the two layouts within a launch.
MANY_ROWS = [
    Workload("many_rows_per_cta", batch=4, n_layers=4, n_kv_heads=40, head_dim=64,
             avg_budget=24, beta=2.0, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=50,
             rope_theta=10000.0, gumbel_seed=21, key_seed=21, prefill=30, decode=50),
    Workload("long_rows_mixed_d64", batch=8, n_layers=2, n_kv_heads=32, head_dim=64,
             avg_budget=2048, beta=1.5, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=3200,
             rope_theta=500000.0, gumbel_seed=22, key_seed=22, prefill=3100, decode=24),
    Workload("long_rows_d128", batch=4, n_layers=2, n_kv_heads=40, head_dim=128,
             avg_budget=4200, beta=1.0, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=4300,
             rope_theta=500000.0, gumbel_seed=23, key_seed=23, prefill=4250, decode=16),
]


@pytest.mark.parametrize("wl", MANY_ROWS, ids=lambda w: w.name)
def test_many_rows_sampled(kvx, wgpu, orc, wl):
    rows = sampled_rows(wl, k=24 if wl.avg_budget < 1000 else 6, seed=1)
    res = run_gpu(kvx, wgpu, wl, rows, segments=[wl.decode // 2])
    reps = compare_rows(orc, wl, rows, *res, threads=8)
    assert sum(r.evictions for r in reps.values()) > 0


FULL = [workloads.KEYFORMER_3B, workloads.PYRAMIDKV, workloads.LATE_RISER_TAU0,
        workloads.LATE_RISER_ANNEAL, workloads.LARGE_CONTEXT]


def full_size_rows(wl):
    """The rows the full-size parity replays on the oracle: all of them when
    there are at most 256 (keyformer_llama3.2-3b's 224); otherwise every layer
    (each has its own budget, so its own tile count and metadata layout),
    with the batch and head indices varied from layer to layer: one row per
    layer from 32 layers up (pyramidkv, large_context), four per layer below
    (the late-riser runs: 64 rows), plus the first and last row."""
    if wl.n_heads <= 256:
        return all_rows(wl)
    per_layer = 1 if wl.n_layers >= 32 else max(1, 64 // wl.n_layers)
    rows = {(0, 0, 0), (wl.batch - 1, wl.n_layers - 1, wl.n_kv_heads - 1)}
    for l in range(wl.n_layers):
        for k in range(per_layer):
            rows.add(((5 * l + 3 * k + 1) % wl.batch, l, (3 * l + 2 * k + 1) % wl.n_kv_heads))
    return sorted(rows)


def _report(name, reps):
    import parity
    summary = dict(workload=name, **parity.summarise(reps.values()))
    print("PARITY " + json.dumps(summary))
    return summary


@pytest.mark.parametrize("wl", FULL, ids=lambda w: w.name)
def test_full_size_rows(kvx, wgpu, orc, wl):
    rows = full_size_rows(wl)
    res = run_gpu(kvx, wgpu, wl, rows, segments=[wl.decode // 2])
    reps = compare_rows(orc, wl, rows, *res)
    summary = _report(wl.name, reps)
    assert summary["evictions"] > 0
    assert len({l for _, l, _ in rows}) == wl.n_layers


@pytest.mark.parametrize("wl", [workloads.KEYFORMER_3B, workloads.LATE_RISER_ANNEAL], ids=lambda w: w.name)
def test_full_size_streaming_kernel(kvx, wgpu, wl):
    """Where the library picks the resident decode kernel at full size, the
    streaming kernel gives the same run bit for bit (sampled rows)."""
    rows = sampled_rows(wl, k=16, seed=4)
    a = run_gpu(kvx, wgpu, wl, rows, segments=[wl.decode // 2], decode_kernel=KERNELS["stream"])
    b = run_gpu(kvx, wgpu, wl, rows, segments=[wl.decode // 2], decode_kernel=KERNELS["resident"])
    assert_same_run(a, b)


def test_full_size_value_rows(kvx, wgpu, orc):
    """keyformer_llama3.2-3b with value rows: 64 seeded rows (of 224) replayed
    on the oracle carrying the same value rows; value rows bit-exact."""
    wl = workloads.KEYFORMER_3B
    rows = sampled_rows(wl, k=64, seed=3)
    res = run_gpu(kvx, wgpu, wl, rows, segments=[wl.decode // 2], with_values=True)
    reps = compare_rows(orc, wl, rows, *res, with_values=True)
    summary = _report(wl.name + "+values", reps)
    assert summary["evictions"] > 0
