"""Value rows move with their keys (keyformer page, KeyformerState.values;
keyformer_update step 3: survivors keep their temporal order) and are never
rotated, so the value rows a cache row keeps are exactly the input value rows
of its kept positions, in slot order. The positions themselves are checked
against the oracle by the parity tests; here the values are checked bit for
bit against that closed form, and the decisions against a key-only run."""
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


@pytest.mark.parametrize("wl", CASES + _random_cases(), ids=lambda w: w.name)
@pytest.mark.parametrize("path", ["multi", "step"])
def test_values_follow_positions(wl, path):
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pre, dec = wgpu.device_inputs(wl)
    vwl = wl.scaled(key_seed=wl.key_seed + 1000)        # any distinct fp16 payload
    vpre, vdec = wgpu.device_inputs(vwl)
    shape = (wl.decode, wl.batch, wl.n_layers, wl.n_kv_heads)
    runs = {}
    for with_values in (False, True):
        h = kvx.from_workload(wl, with_values=with_values)
        ev = torch.full(shape, -7, dtype=torch.int32, device="cuda")
        pev = None
        if pre is not None:
            pev = torch.full((wl.prefill,) + shape[1:], -7, dtype=torch.int32, device="cuda")
            h.prefill(pre, pev, values=vpre)
        if path == "multi":
            h.decode(dec, ev, values=vdec)
        else:
            for t in range(wl.decode):
                h.step(dec[t], ev[t], v_new=vdec[t])
        rows = [(b, l, hh) for b in range(wl.batch) for l in range(wl.n_layers)
                for hh in range(wl.n_kv_heads)]
        st = {r: h.read_state(*r) for r in rows}
        vals = {r: h.read_values(*r) for r in rows} if with_values else None
        runs[with_values] = (ev.cpu().numpy(), pev.cpu().numpy() if pev is not None else None, st,
                             vals)
        h.close()
    ev0, pev0, st0, _ = runs[False]
    ev1, pev1, st1, vals = runs[True]
    assert np.array_equal(ev0, ev1)
    if pev0 is not None:
        assert np.array_equal(pev0, pev1)
    vin_dec = vdec.cpu().numpy().view(np.uint16)
    vin_pre = vpre.cpu().numpy().view(np.uint16) if vpre is not None else None
    moved = 0
    for r, (K, sc, g, pos) in st1.items():
        for x, y in zip(st0[r], st1[r]):
            assert np.array_equal(x, y)
        b, l, hh = r
        allv = np.concatenate(([vin_pre[b, l, hh]] if vin_pre is not None else [])
                              + [vin_dec[:, b, l, hh]])
        assert np.array_equal(vals[r], allv[pos]), f"row {r}"
        moved += int(np.sum(pos != np.arange(len(pos))))
    assert moved > 0
