"""Pins for the oracle's value rows.

Page "veloxquant_mlx.quantizers.keyformer module": KeyformerState.values holds
one fp16 value row per kept token; keyformer_update appends each token's key
and value together (step 2) and, on an eviction, the survivors after the
evicted token shift down by one (step 3); keyformer_get_kv returns keys and
values together. A value row carries no position, so the RoPE remap of step 3
touches keys only.

That fixes the kept values without reference to how the oracle moves them:
after any sequence of steps, the value row in slot j is, bit for bit, the
input value row of the token whose original position is positions[j]. Every
value row fed in below is distinct and encodes its own position, so a row
moved to the wrong slot, left behind, rotated or taken from the wrong input
fails that check.
"""
import numpy as np
import pytest


def _params(orc, **kw):
    base = dict(D=64, budget=12, n_sink=4, layer=0, head=0, tau_init=0.0, tau_end=0.0,
                anneal_steps=0, theta=1e4, seed=0)
    base.update(kw)
    return orc.HeadParams(**base)


def _marked_values(T, D, p0=0):
    """Distinct finite fp16 rows: row t's entries spell out position p0 + t."""
    p = np.arange(p0, p0 + T, dtype=np.int64)[:, None]
    d = np.arange(D, dtype=np.int64)[None, :]
    bits = (p * 131 + d * 7 + 1) % 0x7800     # below the fp16 infinity pattern 0x7C00
    return bits.astype(np.uint16)


def _keys(rng, T, D):
    return rng.standard_normal((T, D)).astype(np.float16).view(np.uint16)


def _check(head, vin):
    K, sc, g, pos = head.state()
    V = head.values()
    assert V.shape == K.shape
    assert np.array_equal(V, vin[pos]), "value rows do not follow their keys' positions"
    return pos


@pytest.mark.parametrize("kw", [
    dict(),                                                         # plain H2O rule
    dict(D=128, budget=9, n_sink=2, tau_init=1.0, tau_end=2.0, anneal_steps=40, theta=5e5, seed=3),
    dict(budget=10, recent=3),                                      # trailing protected window
    dict(budget=8, mode=1),                                         # TOVA-adapted scores
    dict(budget=6, n_sink=4, tau_init=2.0, tau_end=2.0, seed=5),   # two evictable rows
])
def test_decode_values_follow_positions(orc, kw):
    rng = np.random.default_rng(1)
    prm = _params(orc, **kw)
    T = 70
    keys = _keys(rng, T, prm.D)
    vin = _marked_values(T, prm.D)
    head = orc.OracleHead(prm, values=True)
    moved = 0
    for t in range(T):
        e = head.step(keys[t], vin[t])
        pos = _check(head, vin)
        moved += int(e >= 0 and e < head.n)
    assert moved > 0
    # a keys-only head takes the same decisions and ends with the same keys
    plain = orc.OracleHead(prm)
    for t in range(T):
        plain.step(keys[t])
    for x, y in zip(plain.state(), head.state()):
        assert np.array_equal(x, y)
    # the keys that moved were re-rotated; their values were not touched
    K = head.state()[0]
    assert not np.array_equal(K, keys[pos])


@pytest.mark.parametrize("prefill_mode", [0, 1])
@pytest.mark.parametrize("S,budget", [(40, 16), (16, 16), (10, 16)])
def test_prompt_values_follow_positions(orc, prefill_mode, S, budget):
    rng = np.random.default_rng(2)
    prm = _params(orc, D=128, budget=budget, n_sink=4, tau_init=1.0, tau_end=2.0, anneal_steps=60,
                  theta=5e5, seed=9, prefill_mode=prefill_mode)
    T = 30
    keys = _keys(rng, S + T, prm.D)
    vin = _marked_values(S + T, prm.D)
    head = orc.OracleHead(prm, values=True)
    head.prefill(keys[:S], vin[:S])
    pos = _check(head, vin)
    assert len(pos) == min(S, budget)
    for t in range(T):
        head.step(keys[S + t], vin[S + t])
        _check(head, vin)


def test_value_helpers_hand_case(orc):
    """Slot-level behaviour on a 5-row state: evicting slot 1 moves rows 2..4
    down by one, unchanged; a prompt mask keeps the unmasked rows in order."""
    D = 64
    V = np.zeros((6, D), np.uint16)
    rows = _marked_values(6, D)
    for n in range(5):
        orc.lib().orc_values_append(D, n, orc._p(V), orc._p(np.ascontiguousarray(rows[n])))
    assert np.array_equal(V[:5], rows[:5])
    n = orc.lib().orc_values_evict(D, 5, orc._p(V), 1)
    assert n == 4
    assert np.array_equal(V[:4], rows[[0, 2, 3, 4]])
    mask = np.array([0, 1, 1, 0, 0, 1], np.uint8)
    out = np.zeros((6, D), np.uint16)
    kept = orc.lib().orc_values_prefill_apply(6, D, orc._p(rows), orc._p(mask), orc._p(out))
    assert kept == 3
    assert np.array_equal(out[:3], rows[[0, 3, 4]])
