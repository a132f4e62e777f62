"""Pins for the oracle's decode step, eviction and prefill scoring.

Sources: page "veloxquant_mlx.quantizers.keyformer module" (keyformer_update
steps 1-3, THE HONESTY CRUX, the tau = 0 ablation recovering H2O exactly) and
page "PyramidKV -- Layer-Adaptive Budget Attention-Mass Eviction" ("How it
works", "Evidence": single-token bootstrap, budget never exceeded, budget + 1
-> exactly budget, sinks always present, n_sink = 0, non-negative scores,
determinism).
"""
import math

import numpy as np
import pytest
from scipy.special import softmax


def _params(orc, D=64, budget=12, n_sink=4, tau_init=0.0, tau_end=0.0, A=0, theta=1e4, seed=0,
            layer=0, head=0, recent=0, mode=0):
    return orc.HeadParams(D=D, budget=budget, n_sink=n_sink, layer=layer, head=head,
                          tau_init=tau_init, tau_end=tau_end, anneal_steps=A, theta=theta, seed=seed,
                          recent=recent, mode=mode)


def _keys(rng, T, D, scale=1.0):
    return (rng.standard_normal((T, D)) * scale).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------- brute force
class Brute:
    """Tiny-input brute force written from the definition with numpy/scipy."""

    def __init__(self, orc, prm):
        self.orc, self.prm = orc, prm
        self.rows = []  # [key bits, score, g, pos]
        D = prm.D
        w = [prm.theta ** (-(2.0 * i) / D) for i in range(D // 2)]
        self.c = np.array([math.cos(-x) for x in w], np.float32)
        self.s = np.array([math.sin(-x) for x in w], np.float32)

    def rot(self, bits):
        D = bits.size
        v = bits.view(np.float16).astype(np.float32)
        a, b = v[: D // 2], v[D // 2:]
        x = np.float32(a * self.c) - np.float32(b * self.s)
        y = np.float32(a * self.s) + np.float32(b * self.c)
        return np.concatenate([x, y]).astype(np.float16).view(np.uint16)

    def step(self, k, p):
        prm = self.prm
        g = float(self.orc.gumbel(prm.seed, prm.layer, prm.head, p, 1)[0])
        self.rows.append([k.copy(), 0.0, g, p])
        K = np.stack([r[0] for r in self.rows]).view(np.float16).astype(np.float64)
        attn = softmax(K @ k.view(np.float16).astype(np.float64) / math.sqrt(prm.D))
        for r, a in zip(self.rows, attn):
            r[1] = a if prm.mode == 1 else r[1] + a
        if len(self.rows) <= prm.budget:
            return -1
        if prm.anneal_steps > 0 and prm.tau_init != prm.tau_end:
            tau = prm.tau_init + min(p, prm.anneal_steps) * (prm.tau_end - prm.tau_init) / prm.anneal_steps
        else:
            tau = prm.tau_init
        cand = [(r[1] + tau * r[2], j) for j, r in enumerate(self.rows)
                if prm.n_sink <= j < len(self.rows) - prm.recent]
        e = min(cand)[1]
        del self.rows[e]
        for r in self.rows[e:]:
            r[0] = self.rot(r[0])
        return e


@pytest.mark.parametrize("D,budget,n_sink,tau_init,tau_end,A,theta,recent,mode", [
    (64, 12, 4, 0.0, 0.0, 0, 1e4, 0, 0),
    (64, 5, 4, 0.0, 0.0, 0, 1e4, 0, 0),        # budget = n_sink + 1
    (64, 8, 0, 0.0, 0.0, 0, 1e4, 0, 0),        # no sinks
    (128, 16, 4, 1.0, 2.0, 30, 5e5, 0, 0),     # annealed Gumbel regulariser
    (128, 9, 2, 0.5, 0.5, 0, 5e5, 0, 0),       # constant tau
    (64, 12, 4, 0.0, 0.0, 0, 1e4, 3, 0),       # trailing protected window
    (64, 8, 2, 0.0, 0.0, 0, 1e4, 5, 0),        # budget = n_sink + recent + 1
    (64, 12, 4, 0.0, 0.0, 0, 1e4, 0, 1),       # TOVA-adapted (current-step scores)
    (128, 10, 2, 1.0, 2.0, 30, 5e5, 2, 1),     # TOVA + Gumbel + recent window
])
def test_brute_force_tiny(orc, D, budget, n_sink, tau_init, tau_end, A, theta, recent, mode):
    rng = np.random.default_rng(budget * 7 + n_sink + 13 * recent + 101 * mode)
    prm = _params(orc, D=D, budget=budget, n_sink=n_sink, tau_init=tau_init, tau_end=tau_end, A=A,
                  theta=theta, seed=42, layer=1, head=3, recent=recent, mode=mode)
    head, brute = orc.OracleHead(prm), Brute(orc, prm)
    keys = _keys(rng, 40, D)
    for p in range(40):
        e_o = head.step(keys[p])
        e_b = brute.step(keys[p], p)
        assert e_o == e_b, f"step {p}"
        K, sc, g, pos = head.state()
        assert np.array_equal(K, np.stack([r[0] for r in brute.rows]))
        assert np.array_equal(pos, np.array([r[3] for r in brute.rows]))
        np.testing.assert_allclose(sc, [r[1] for r in brute.rows], rtol=1e-12, atol=1e-15)


def test_bootstrap_single_token(orc):
    head = orc.OracleHead(_params(orc))
    head.step(_keys(np.random.default_rng(0), 1, 64)[0])
    K, sc, g, pos = head.state()
    assert head.n == 1 and sc[0] == 1.0 and pos[0] == 0


def test_invariants_stress(orc):
    rng = np.random.default_rng(3)
    for n_sink, budget, tau in [(4, 12, 0.0), (0, 6, 0.0), (4, 10, 1.5)]:
        prm = _params(orc, D=64, budget=budget, n_sink=n_sink, tau_init=tau, tau_end=tau, seed=5)
        head = orc.OracleHead(prm)
        keys = _keys(rng, 60, 64)
        seen = set()
        total = 0.0
        for p in range(60):
            before = head.score[: head.n].sum()
            head.accumulate(keys[p])
            total += 1.0
            # each step adds exactly 1.0 of attention mass before eviction
            assert abs(head.score[: head.n].sum() - (before + 1.0)) < 1e-12
            if head.over_budget():
                assert head.n == budget + 1
                e = head.select()
                gone = int(head.pos[e])
                head.evict(e)
                assert head.n == budget  # budget + 1 -> exactly budget
                seen.add(gone)
            assert head.n <= budget
            K, sc, g, pos = head.state()
            assert np.all(sc >= 0)
            assert list(pos[:n_sink]) == list(range(min(n_sink, head.n)))   # sinks stay
            assert np.all(np.diff(pos) > 0)                                  # temporal order
            assert set(pos.tolist()).isdisjoint(seen)
            assert set(pos.tolist()) | seen == set(range(p + 1))
        # determinism
        head2 = orc.OracleHead(prm)
        for p in range(60):
            head2.step(keys[p])
        for a, b in zip(head.state(), head2.state()):
            assert np.array_equal(a, b)


def test_tau_zero_is_h2o_for_any_seed(orc):
    # keyformer page: tau_init = tau_end = 0 removes the noise and recovers
    # H2O-adapted exactly -- the Gumbel values then cannot matter.
    rng = np.random.default_rng(4)
    keys = _keys(rng, 80, 64)
    runs = []
    for seed in (0, 1, 999):
        head = orc.OracleHead(_params(orc, budget=10, seed=seed))
        ev = [head.step(k) for k in keys]
        K, sc, g, pos = head.state()
        runs.append((ev, K, sc, pos))
    for r in runs[1:]:
        assert r[0] == runs[0][0]
        for a, b in zip(r[1:], runs[0][1:]):
            assert np.array_equal(a, b)
    # and a large tau makes the noise decide differently
    head = orc.OracleHead(_params(orc, budget=10, seed=0, tau_init=5.0, tau_end=5.0))
    assert [head.step(k) for k in keys] != runs[0][0]


def test_orthogonal_keys_closed_form(orc):
    # One-hot keys c*e_d: every cross logit is 0, the self logit is c^2/sqrt(D).
    # With i rows stored, token i pays E/(E+i) to itself and 1/(E+i) to each
    # older row (E = exp(c^2/sqrt(D))), so row j's score after step t is
    # E/(E+j) + sum_{i=j+1..t} 1/(E+i). The new row is part of its own softmax.
    D, c = 64, 2.0
    prm = _params(orc, D=D, budget=40)
    head = orc.OracleHead(prm)
    E = math.exp(c * c / math.sqrt(D))
    T = 30
    for i in range(T):
        k = np.zeros(D, np.float16)
        k[i] = c
        head.step(k.view(np.uint16))
    want = [E / (E + j) + sum(1.0 / (E + i) for i in range(j + 1, T)) for j in range(T)]
    np.testing.assert_allclose(head.state()[1], want, rtol=1e-13)


def test_argmin_rules_hand_cases(orc):
    prm = _params(orc, D=64, budget=7, n_sink=4)
    head = orc.OracleHead(prm)
    head.n = 8
    head.score[:8] = [0.0, 0.0, 0.0, 0.0, 0.3, 0.1, 0.1, 0.7]  # sinks hold the lowest scores
    head.g[:8] = 0.0
    head.next_pos = 8
    assert head.select() == 5          # tie between slots 5 and 6 -> lowest slot
    head.prm = _params(orc, D=64, budget=7, n_sink=0)
    assert head.select() == 0          # no sinks: slot 0 is evictable
    head.prm = _params(orc, D=64, budget=7, n_sink=4, tau_init=2.0, tau_end=2.0)
    head.g[:8] = [0, 0, 0, 0, 0.0, 0.5, 0.2, -0.4]
    # r = [.., 0.3, 1.1, 0.5, -0.1] -> slot 7
    assert head.select() == 7


def test_evict_shifts_and_rerotates(orc):
    rng = np.random.default_rng(6)
    prm = _params(orc, D=128, budget=6, n_sink=2, theta=5e5)
    head = orc.OracleHead(prm)
    keys = _keys(rng, 7, 128)
    for k in keys:
        head.accumulate(k)
    before = head.state()
    head.evict(3)
    K, sc, g, pos = head.state()
    c, s = orc.rope_consts(5e5, 128, -1)
    assert np.array_equal(K[:3], before[0][:3])
    for j in range(3, 6):
        assert np.array_equal(K[j], orc.rotate_row(before[0][j + 1], c, s))
    assert list(pos) == [0, 1, 2, 4, 5, 6]
    assert np.array_equal(sc, np.delete(before[1], 3))


# ---------------------------------------------------------------- prefill
def test_prefill_colsum_equals_steps_and_matrix_form(orc):
    rng = np.random.default_rng(7)
    for D, S in [(64, 1), (64, 37), (128, 130)]:
        keys = _keys(rng, S, D)
        col = orc.prefill_colsum(keys)
        head = orc.OracleHead(_params(orc, D=D, budget=S + 1))
        for k in keys:
            head.step(k)
        np.testing.assert_allclose(col, head.state()[1], rtol=1e-12)
        Kf = keys.view(np.float16).astype(np.float64)
        G = Kf @ Kf.T / math.sqrt(D)
        G[np.triu_indices(S, 1)] = -np.inf
        P = softmax(G, axis=1)
        np.testing.assert_allclose(col, P.sum(axis=0), rtol=1e-12)
        assert abs(col.sum() - S) < 1e-9


def test_prefill_bulk_select_and_apply(orc):
    prm = _params(orc, D=64, budget=6, n_sink=2, theta=1e4)
    head = orc.OracleHead(prm)
    r = np.array([0.0, 0.0, 0.5, 0.2, 0.2, 0.9, 0.1, 0.8, 0.3, 0.6])
    mask = head.prefill_select(r)
    # evict 4 of the non-sink rows: 0.1 (6), 0.2 (3), 0.2 (4), 0.3 (8); sinks kept
    assert list(np.nonzero(mask)[0]) == [3, 4, 6, 8]
    rng = np.random.default_rng(8)
    keys = _keys(rng, 10, 64)
    colsum = np.arange(10, dtype=np.float64)
    g = np.arange(10, dtype=np.float32) / 10
    head.prefill_apply(keys, colsum, g, mask)
    K, sc, gg, pos = head.state()
    assert list(pos) == [0, 1, 2, 5, 7, 9]
    assert list(sc) == [0, 1, 2, 5, 7, 9]
    for new, old in enumerate(pos):
        if new == old:
            assert np.array_equal(K[new], keys[old])
        else:
            c, s = orc.rope_consts(1e4, 64, new - old)
            assert np.array_equal(K[new], orc.rotate_row(keys[old], c, s))


def test_prefill_within_budget_keeps_all(orc):
    rng = np.random.default_rng(9)
    keys = _keys(rng, 20, 64)
    head = orc.OracleHead(_params(orc, budget=32))
    mask = head.prefill(keys)
    assert mask.sum() == 0
    K, sc, g, pos = head.state()
    assert np.array_equal(K, keys) and list(pos) == list(range(20))


def test_c_driver_matches_stepwise(orc):
    rng = np.random.default_rng(10)
    prms = [_params(orc, D=64, budget=b, n_sink=ns, tau_init=ti, tau_end=te, A=A, seed=11,
                    layer=l, head=h)
            for b, ns, ti, te, A, l, h in [(16, 4, 0.0, 0.0, 0, 0, 0), (12, 2, 1.0, 2.0, 50, 3, 1),
                                            (24, 4, 1.0, 1.0, 0, 2, 7)]]
    S, T = 20, 50
    pk = np.stack([_keys(rng, S, 64) for _ in prms])
    dk = np.stack([_keys(rng, T, 64) for _ in prms])
    ev, n, K, sc, g, pos, used = orc.run_heads(prms, pk, dk, n_threads=2)
    for i, prm in enumerate(prms):
        head = orc.OracleHead(prm)
        head.prefill(pk[i])
        evs = [head.step(k) for k in dk[i]]
        assert evs == list(ev[i])
        Kh, sch, gh, posh = head.state()
        assert n[i] == head.n
        assert np.array_equal(K[i, : head.n], Kh) and np.array_equal(pos[i, : head.n], posh)
        assert np.array_equal(sc[i, : head.n], sch) and np.array_equal(g[i, : head.n], gh)


# ---------------------------------------------------------------- recent window / TOVA
def test_recent_window_protects_the_newest_rows(orc):
    # keyformer page, KeyformerState.recent: a trailing protected window
    rng = np.random.default_rng(11)
    for recent, n_sink, budget in [(3, 4, 12), (5, 0, 7), (1, 2, 4)]:
        head = orc.OracleHead(_params(orc, budget=budget, n_sink=n_sink, recent=recent,
                                      tau_init=1.0, tau_end=1.0, seed=3))
        keys = _keys(rng, 80, 64)
        for p in range(80):
            n_before = head.n
            e = head.step(keys[p])
            if e >= 0:
                assert n_sink <= e < n_before + 1 - recent
            K, sc, g, pos = head.state()
            newest = list(range(max(0, p + 1 - recent), p + 1))
            assert set(newest) <= set(pos.tolist())
            assert head.n <= budget


def test_recent_zero_is_the_plain_rule(orc):
    rng = np.random.default_rng(12)
    keys = _keys(rng, 60, 64)
    a = orc.OracleHead(_params(orc, budget=10, tau_init=1.0, tau_end=1.0, seed=9))
    b = orc.OracleHead(_params(orc, budget=10, tau_init=1.0, tau_end=1.0, seed=9, recent=0))
    assert [a.step(k) for k in keys] == [b.step(k) for k in keys]


def test_tova_closed_form_orthogonal_keys(orc):
    # PyramidKV page, method table: TOVA-adapted scores each row by the current
    # step's attention weight. With one-hot keys the step over i+1 rows gives
    # the newest row E/(E+i) and every older row 1/(E+i).
    D, c = 64, 2.0
    head = orc.OracleHead(_params(orc, D=D, budget=40, mode=1))
    E = math.exp(c * c / math.sqrt(D))
    for i in range(30):
        k = np.zeros(D, np.float16)
        k[i] = c
        head.step(k.view(np.uint16))
        sc = head.state()[1]
        np.testing.assert_allclose(sc[:-1], 1.0 / (E + i), rtol=1e-13)
        np.testing.assert_allclose(sc[-1], E / (E + i), rtol=1e-13)


def test_tova_scores_are_one_distribution(orc):
    rng = np.random.default_rng(13)
    head = orc.OracleHead(_params(orc, budget=10, mode=1))
    for k in _keys(rng, 50, 64):
        head.accumulate(k)
        assert abs(head.score[: head.n].sum() - 1.0) < 1e-12
        assert np.all(head.score[: head.n] >= 0)
        if head.over_budget():
            head.evict(head.select())


def test_tova_prompt_scores_are_the_last_softmax_row(orc):
    rng = np.random.default_rng(14)
    for D, S in [(64, 1), (64, 33), (128, 130)]:
        keys = _keys(rng, S, D)
        Kf = keys.view(np.float16).astype(np.float64)
        want = softmax(Kf @ Kf[-1] / math.sqrt(D))
        np.testing.assert_allclose(orc.prefill_lastrow(keys), want, rtol=1e-12)
        # and equal to one decode step over the first S-1 rows
        head = orc.OracleHead(_params(orc, D=D, budget=S + 1, mode=1))
        for k in keys:
            head.step(k)
        np.testing.assert_allclose(head.state()[1], want, rtol=1e-12)


def test_prefill_select_respects_recent(orc):
    head = orc.OracleHead(_params(orc, budget=6, n_sink=2, recent=2))
    r = np.array([0.0, 0.0, 0.5, 0.2, 0.2, 0.9, 0.1, 0.8, 0.0, 0.0])  # last two lowest but protected
    mask = head.prefill_select(r)
    # 4 of the rows 2..7 go: 0.1 (6), 0.2 (3), 0.2 (4), 0.5 (2); rows 8, 9 are protected
    assert list(np.nonzero(mask)[0]) == [2, 3, 4, 6]


# ---------------------------------------------------------------- sequential prompt
def test_sequential_prompt_c_driver_matches_stepwise(orc):
    # keyformer page, keyformer_update: "For each of the S incoming tokens" the
    # three steps run in turn, so a prompt longer than the budget evicts inside it
    rng = np.random.default_rng(21)
    prms = [_params(orc, D=64, budget=b, n_sink=ns, tau_init=ti, tau_end=te, A=A, seed=7,
                    layer=l, head=h, recent=rc, mode=m)
            for b, ns, ti, te, A, l, h, rc, m in [(10, 4, 0.0, 0.0, 0, 0, 0, 0, 0),
                                                   (8, 2, 1.0, 2.0, 40, 1, 1, 2, 0),
                                                   (12, 4, 0.5, 0.5, 0, 2, 3, 0, 1)]]
    for p in prms:
        p.prefill_mode = 1
    S, T = 30, 25
    pk = np.stack([_keys(rng, S, 64) for _ in prms])
    dk = np.stack([_keys(rng, T, 64) for _ in prms])
    ev, n, K, sc, g, pos, used = orc.run_heads(prms, pk, dk, n_threads=2)
    for i, prm in enumerate(prms):
        head = orc.OracleHead(prm)
        prompt_ev = head.prefill(pk[i])
        assert (prompt_ev >= 0).sum() == S - prm.budget     # one eviction per token past the budget
        evs = [head.step(k) for k in dk[i]]
        assert evs == list(ev[i])
        Kh, sch, gh, posh = head.state()
        assert np.array_equal(K[i, : head.n], Kh) and np.array_equal(pos[i, : head.n], posh)
        assert np.array_equal(sc[i, : head.n], sch)


def test_sequential_equals_bulk_when_the_prompt_fits(orc):
    rng = np.random.default_rng(22)
    keys = _keys(rng, 20, 64)
    a = orc.OracleHead(_params(orc, budget=24, tau_init=1.0, tau_end=1.0, seed=2))
    b = orc.OracleHead(_params(orc, budget=24, tau_init=1.0, tau_end=1.0, seed=2))
    b.prm.prefill_mode = 1
    a.prefill(keys)
    b.prefill(keys)
    sa, sb = a.state(), b.state()
    for x, y in ((sa[0], sb[0]), (sa[3], sb[3]), (sa[2], sb[2])):
        assert np.array_equal(x, y)
    np.testing.assert_allclose(sa[1], sb[1], rtol=1e-12)
