"""Pins for the oracle's frozen Gumbel values.

The pages fix that the value is frozen per inserted position, drawn once, and is
-log(-log(u)) (page "veloxquant_mlx.quantizers.keyformer module", THE HONESTY
CRUX item 2, KeyformerState.gumbel). They print no values, so the hash itself
is pinned only to the published SplitMix64 reference outputs and the drawn
values to the Gumbel distribution's known moments and CDF.
"""
import math
import os

import numpy as np
from scipy import stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_reference.txt")


def test_splitmix64_reference_outputs(orc):
    golden = 0x9E3779B97F4A7C15
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        base, state, *outs = line.split()
        state = int(state)
        outs = [int(x, 16 if base == "hex" else 10) for x in outs]
        # k-th output of a generator started at `state` = splitmix64(state + k*golden)
        for k, want in enumerate(outs):
            assert orc.splitmix64((state + k * golden) % 2**64) == want


def test_gumbel_moments_and_cdf(orc):
    vals = np.concatenate([orc.gumbel(seed, layer, head, 0, 20000)
                           for seed, layer, head in [(0, 0, 0), (1234, 3, 5), (7, 31, 7)]])
    vals = vals.astype(np.float64)
    n = vals.size
    euler_gamma = 0.5772156649015329
    var = math.pi ** 2 / 6
    assert abs(vals.mean() - euler_gamma) < 5 * math.sqrt(var / n)
    assert abs(vals.var() - var) < 0.05 * var
    ks = stats.kstest(vals, lambda x: np.exp(-np.exp(-x)))
    assert ks.pvalue > 1e-4


def test_gumbel_frozen_and_keyed(orc):
    a = orc.gumbel(1234, 3, 5, 100, 50)
    b = orc.gumbel(1234, 3, 5, 100, 50)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, orc.gumbel(1234, 3, 6, 100, 50))
    assert not np.array_equal(a, orc.gumbel(1234, 4, 5, 100, 50))
    assert not np.array_equal(a, orc.gumbel(1235, 3, 5, 100, 50))
    # position p of a longer draw is the same value as a draw at p alone
    assert orc.gumbel(1234, 3, 5, 130, 1)[0] == a[30]


def test_gumbel_value_from_hash(orc):
    # g = -log(-log(u)), u = (2k+1)/2^53 with k the top 52 bits of the hash
    for pos in (0, 1, 17, 4095, 123456):
        h = orc.gumbel_hash(99, 2, 3, pos)
        k = h >> 12
        u = (2 * k + 1) / 2.0 ** 53
        want = np.float32(-math.log(-math.log(u)))
        assert orc.gumbel(99, 2, 3, pos, 1)[0] == want


def test_tau_schedule_closed_form(orc):
    # keyformer page GAP #1: tau = tau_init + min(pos, T) * (tau_end - tau_init) / T
    assert orc.tau(1.0, 2.0, 2048, 0) == 1.0
    assert orc.tau(1.0, 2.0, 2048, 1024) == 1.5
    assert orc.tau(1.0, 2.0, 2048, 2048) == 2.0
    assert orc.tau(1.0, 2.0, 2048, 99999) == 2.0
    assert orc.tau(1.0, 2.0, 0, 500) == 1.0          # anneal_steps = 0: constant tau_init
    assert orc.tau(0.5, 0.5, 100, 50) == 0.5          # tau_init == tau_end: constant
    assert orc.tau(0.0, 0.0, 4096, 77) == 0.0
