"""Pins for the oracle's per-layer budget taper (page "PyramidKV -- Layer-Adaptive
Budget Attention-Mass Eviction", sections "The budget schedule", "Parameters",
"Evidence")."""
import os

import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pyramid_schedule_12L.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, rest = line.split(":")
        L, avg, ns, beta = head.split()
        vals, mean = rest.split(";")
        rows.append((int(L), int(avg), int(ns), float(beta), [int(v) for v in vals.split()],
                     float(mean)))
    return rows


def test_worked_example_matches_page(orc):
    for L, avg, ns, beta, want, mean in _golden():
        got = orc.budgets(L, avg, ns, beta)
        assert got == want
        assert sum(got) / L == mean


def test_beta_one_is_flat(orc):
    for L in (1, 2, 12, 32):
        assert orc.budgets(L, 512, 4, 1.0) == [512] * L


@pytest.mark.parametrize("L,avg,ns,beta", [(12, 512, 4, 2.0), (32, 512, 4, 2.0), (32, 2048, 4, 1.5),
                                           (28, 512, 4, 1.3), (7, 100, 0, 3.0), (5, 6, 4, 9.0)])
def test_invariants(orc, L, avg, ns, beta):
    b = orc.budgets(L, avg, ns, beta)
    assert len(b) == L
    assert all(x >= y for x, y in zip(b, b[1:])), "monotone non-increasing"
    assert abs(sum(b) / L - avg) <= 0.05 * avg, "mean within 5% of avg"
    assert sum(b) == L * avg, "symmetric rounding keeps the mean exact"
    assert min(b) >= ns + 1, "floored at n_sink + 1"


def test_closed_form_endpoints(orc):
    # top = avg + h, bottom = avg - h, h = min((beta-1)*avg, avg-(n_sink+1))
    b = orc.budgets(32, 2048, 4, 1.5)
    assert (b[0], b[-1]) == (3072, 1024)
    b = orc.budgets(12, 512, 4, 2.0)
    assert (b[0], b[-1]) == (512 + 507, 512 - 507)


def test_larger_beta_widens_spread(orc):
    spreads = []
    for beta in (1.0, 1.25, 1.5, 1.75, 2.0):
        b = orc.budgets(12, 512, 4, beta)
        spreads.append(b[0] - b[-1])
    assert spreads == sorted(spreads) and spreads[0] == 0 and spreads[-1] > spreads[1]


def test_edge_cases(orc):
    assert orc.budgets(1, 512, 4, 2.0) == [512]
    assert orc.budgets(0, 512, 4, 2.0) == []
    with pytest.raises(ValueError):
        orc.budgets(12, 512, 4, 0.99)
    with pytest.raises(ValueError):
        orc.budgets(12, 4, 4, 1.0)  # avg below n_sink + 1
