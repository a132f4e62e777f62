"""Lockstep comparison of the CUDA path against the fp64 oracle, one cache row
at a time. Test infrastructure (used by the GPU tests and ``smoke()``).

Agreement rules (the eviction step's parity definition):
  * the evicted slot of every step and the positions[] array are bit-exact
    integers, except at steps where the oracle's two lowest regularised scores
    differ by less than ``TIE_REL`` relative: those are ties, counted, and the
    CUDA path's pick must then be one of the tied rows;
  * scores match within 1e-4 relative;
  * survivor keys match within 1 fp16 ULP (the fp32 re-rotation is specified
    op by op, so they are expected bit-exact);
  * Gumbel values are bit-equal, up to counted 1-ULP double-rounding outliers.

At a tie where the two picks differ, both are correct answers of the method up
to rounding; the driver then applies the CUDA path's (validated) pick to the
oracle state so the two stay comparable for the rest of the run. The oracle
itself never reads CUDA output: the choice is made here, after checking it
against the oracle's own tie set.

"Relative" is relative to |r| (the plain reading): the CUDA path may pick
another row only when it lies within TIE_REL * |r| of the oracle's lowest.
For information a wider set is counted as well, whose tolerance scales with
the magnitude of the terms forming r = score + tau*g (|r| + |score| +
|tau*g|, the rounding a near-cancellation of score against tau*g carries):
``ties`` counts the steps that are ties under that wider rule, ``ties_plain``
those that are ties under the plain rule, and a divergence that only the
wider rule would admit is a failure (``tie_divergences_wide_only`` stays 0).

Value rows (a value-carrying cache) are compared bit for bit: they are moved,
never computed.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

TIE_REL = 1e-5
SCORE_RTOL = 1e-4


@dataclass
class RowReport:
    steps: int = 0
    evictions: int = 0
    evicted_first: int = 0        # evictions of the first candidate slot (n_sink)
    evicted_last: int = 0         # evictions of the last candidate slot (the new row when recent = 0)
    evicted_mid: int = 0          # evictions strictly between them
    ties: int = 0                 # steps whose two lowest r are within TIE_REL (wide rule)
    ties_plain: int = 0           # ... of which also within TIE_REL * |r| (plain rule)
    tie_divergences: int = 0      # ties where the CUDA path picked another tied row
    tie_divergences_wide_only: int = 0   # ... at a step that is a tie under the wide rule only
    prefill_tie: bool = False
    prefill_tie_wide_only: bool = False
    gumbel_ulp_outliers: int = 0
    max_key_ulp: int = 0
    max_score_rel: float = 0.0
    failures: list = field(default_factory=list)

    def ok(self) -> bool:
        return not self.failures


def _scale(head, j: int, tau: float) -> float:
    return abs(head.r[j]) + abs(head.score[j]) + abs(tau * float(head.g[j]))


def _tie_set(head, tau: float, n_sink: int, recent: int = 0, plain: bool = False) -> tuple[list[int], float]:
    """Rows whose r is within the tie tolerance of the lowest (lowest first).
    plain: the tolerance is TIE_REL * |r| instead of the wide rule's scale."""
    n = head.n
    r = head.r[:n]
    cand = np.arange(n_sink, n - recent)
    order = cand[np.argsort(r[cand], kind="stable")]
    best = int(order[0])
    ties = [best]
    gap = np.inf
    for j in order[1:]:
        j = int(j)
        if plain:
            tol = TIE_REL * max(abs(r[best]), abs(r[j]))
        else:
            tol = TIE_REL * max(_scale(head, best, tau), _scale(head, j, tau))
        d = r[j] - r[best]
        if len(ties) == 1:
            gap = d
        if d <= tol:
            ties.append(j)
        else:
            break
    return ties, gap


def ulp_diff_f16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in fp16 ULPs between two arrays of fp16 bit patterns."""
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + (x & 0x7FFF))
    return np.abs(key(a) - key(b))


def compare_state(rep: RowReport, where: str, orc_state, gpu_state):
    """States are (keys, scores, gumbel, positions) or, on a value-carrying
    cache, (keys, scores, gumbel, positions, values)."""
    oK, osc, og, opos = orc_state[:4]
    gK, gsc, gg, gpos = gpu_state[:4]
    if len(orc_state) != len(gpu_state):
        rep.failures.append(f"{where}: one side carries value rows, the other does not")
        return
    if len(opos) != len(gpos):
        rep.failures.append(f"{where}: kept {len(gpos)} rows, oracle {len(opos)}")
        return
    if not np.array_equal(opos, gpos):
        bad = int(np.nonzero(opos != gpos)[0][0])
        rep.failures.append(f"{where}: positions differ first at slot {bad}: gpu {gpos[bad]} "
                            f"oracle {opos[bad]}")
        return
    if len(opos):
        u = ulp_diff_f16(oK, gK)
        rep.max_key_ulp = max(rep.max_key_ulp, int(u.max()))
        if u.max() > 1:
            rep.failures.append(f"{where}: keys differ by {int(u.max())} fp16 ULP")
        err = np.abs(gsc.astype(np.float64) - osc)
        rep.max_score_rel = max(rep.max_score_rel,
                                float((err / np.maximum(np.abs(osc), 1e-12)).max()))
        bad = err > SCORE_RTOL * np.abs(osc)
        if bad.any():
            j = int(np.nonzero(bad)[0][0])
            rep.failures.append(f"{where}: score slot {j}: gpu {gsc[j]!r} oracle {osc[j]!r}")
        gdiff = np.abs(og.view(np.int32).astype(np.int64) - gg.view(np.int32).astype(np.int64))
        rep.gumbel_ulp_outliers += int((gdiff == 1).sum())
        if (gdiff > 1).any():
            rep.failures.append(f"{where}: gumbel values differ by more than 1 ULP")
        if len(orc_state) == 5:
            oV, gV = orc_state[4], gpu_state[4]
            if oV.shape != gV.shape or not np.array_equal(oV, gV):
                rep.failures.append(f"{where}: value rows differ")


def _state(head):
    st = head.state()
    return st + (head.values(),) if head.V is not None else st


def _replay_steps(orc, prm, head, keys, gpu_ev, rep, what, checkpoints=None, values=None):
    for t in range(int(keys.shape[0])):
        head.accumulate(keys[t], None if values is None else values[t])
        rep.steps += 1
        eg = int(gpu_ev[t])
        if not head.over_budget():
            if eg != -1:
                rep.failures.append(f"{what} {t}: gpu evicted {eg} within budget")
                return
            continue
        rep.evictions += 1
        tau = orc.tau(prm.tau_init, prm.tau_end, prm.anneal_steps, head.next_pos - 1)
        head.regularised()
        ties, gap = _tie_set(head, tau, prm.n_sink, prm.recent)
        plain = ties   # the plain rule's set is a prefix of the wide rule's
        if len(ties) > 1:
            rep.ties += 1
            plain = _tie_set(head, tau, prm.n_sink, prm.recent, plain=True)[0]
            if len(plain) > 1:
                rep.ties_plain += 1
        e = ties[0]
        if eg != e:
            if eg in plain:
                rep.tie_divergences += 1
                e = eg
            elif eg in ties:
                rep.tie_divergences_wide_only += 1
                rep.failures.append(
                    f"{what} {t} (pos {head.next_pos - 1}): gpu evicted {eg} (r={head.r[eg]}), "
                    f"oracle {e} (r={head.r[e]}): a tie only under the wider rule")
                return
            else:
                rep.failures.append(
                    f"{what} {t} (pos {head.next_pos - 1}): gpu evicted {eg} "
                    f"(r={head.r[eg] if 0 <= eg < head.n else None}), oracle {e} (r={head.r[e]}), "
                    f"ties {ties}")
                return
        last = head.n - 1 - prm.recent
        if e == prm.n_sink:
            rep.evicted_first += 1
        elif e == last:
            rep.evicted_last += 1
        else:
            rep.evicted_mid += 1
        head.evict(e)
        if checkpoints and (t + 1) in checkpoints:
            compare_state(rep, f"after step {t + 1}", _state(head), checkpoints[t + 1])
            if rep.failures:
                return


def run_row(orc, prm, prefill_keys, decode_keys, gpu_ev, gpu_after_prefill=None,
            gpu_final=None, checkpoints=None, gpu_prompt_ev=None, values=None) -> RowReport:
    """Replay one cache row on the oracle and compare it with the CUDA path.

    gpu_ev: int32 [T] evicted slots the CUDA path reported per decode step.
    gpu_after_prefill / gpu_final: (keys, scores, gumbel, positions[, values])
    read back from the CUDA path after the prompt and at the end. checkpoints:
    optional {step_index: state} read back after that many decode steps.
    values: (prompt value rows [S, D] or None, decode value rows [T, D]) for a
    value-carrying cache; the oracle then carries them too.
    """
    rep = RowReport()
    head = orc.OracleHead(prm, values=values is not None)
    pre_v, dec_v = values if values is not None else (None, None)
    S = 0 if prefill_keys is None else int(prefill_keys.shape[0])
    if S > 0 and getattr(prm, "prefill_mode", 0) == 1:
        # one step per prompt token: replay them like decode steps against the
        # CUDA path's prompt eviction log, then compare the state
        if gpu_prompt_ev is None:
            rep.failures.append("sequential prompt needs the CUDA path's prompt eviction log")
            return rep
        _replay_steps(orc, prm, head, prefill_keys, gpu_prompt_ev, rep, "prompt step", values=pre_v)
        if rep.failures:
            return rep
        if gpu_after_prefill is not None:
            compare_state(rep, "after prefill", _state(head), gpu_after_prefill)
            if rep.failures:
                return rep
        S = 0   # the prompt is done
    if S > 0:
        colsum, g, r = head.prefill_scores(prefill_keys)
        mask = head.prefill_select(r)
        if S > prm.budget and gpu_after_prefill is not None:
            gpos = gpu_after_prefill[3]
            gmask = np.ones(S, np.uint8)
            gmask[gpos] = 0
            if not np.array_equal(gmask, mask):
                # A boundary tie: every row the two disagree on must sit within
                # TIE_REL of the oracle's cut between evicted and kept rows.
                t = orc.tau(prm.tau_init, prm.tau_end, prm.anneal_steps, S - 1)
                rs = np.sort(r[prm.n_sink:S - prm.recent])
                k = S - prm.budget
                scale = np.abs(r) + np.abs(colsum) + np.abs(t * g.astype(np.float64))
                gpu_only = np.nonzero((gmask == 1) & (mask == 0))[0]
                orc_only = np.nonzero((gmask == 0) & (mask == 1))[0]
                valid = (gmask.sum() == mask.sum() and np.all(gpu_only >= prm.n_sink)
                         and np.all(gpu_only < S - prm.recent)
                         and np.all(r[gpu_only] - rs[k - 1] <= TIE_REL * scale[gpu_only])
                         and np.all(rs[k] - r[orc_only] <= TIE_REL * scale[orc_only]))
                plain_ok = valid and (np.all(r[gpu_only] - rs[k - 1] <= TIE_REL * np.abs(r[gpu_only]))
                                      and np.all(rs[k] - r[orc_only] <= TIE_REL * np.abs(r[orc_only])))
                if not plain_ok:
                    rep.prefill_tie_wide_only = valid
                    diff = np.nonzero(gmask != mask)[0]
                    rep.failures.append(f"prefill selection differs at rows {diff[:8].tolist()}"
                                        + (" (a tie only under the wider rule)" if valid else ""))
                    return rep
                rep.prefill_tie = True
                mask = gmask
        head.prefill_apply(prefill_keys, colsum, g, mask, pre_v)
        if gpu_after_prefill is not None:
            compare_state(rep, "after prefill", _state(head), gpu_after_prefill)
            if rep.failures:
                return rep
    _replay_steps(orc, prm, head, decode_keys, gpu_ev, rep, "step", checkpoints, values=dec_v)
    if rep.failures:
        return rep
    if gpu_final is not None:
        compare_state(rep, "final", _state(head), gpu_final)
    return rep


def summarise(reports) -> dict:
    """Totals over many rows' reports (for the tests' printed summaries)."""
    reps = list(reports)
    tot = lambda f: sum(getattr(r, f) for r in reps)
    return {"rows": len(reps), "evictions": tot("evictions"), "ties": tot("ties"),
            "ties_plain": tot("ties_plain"), "tie_divergences": tot("tie_divergences"),
            "tie_divergences_wide_only": tot("tie_divergences_wide_only"),
            "prefill_ties": tot("prefill_tie"), "prefill_ties_wide_only": tot("prefill_tie_wide_only"),
            "gumbel_ulp_outliers": tot("gumbel_ulp_outliers"),
            "max_key_ulp": max((r.max_key_ulp for r in reps), default=0),
            "max_score_rel": max((r.max_score_rel for r in reps), default=0.0)}
