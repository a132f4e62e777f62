"""Pins for the oracle's fp16 conversion and its fp32 RoPE re-rotation.

The pages fix that the re-rotation of a shifted key runs in fp32 and the key is
stored as fp16 (page "veloxquant_mlx.quantizers.keyformer module", FUSED METAL
KERNEL: keys within 1 fp16 ULP of the pure-MLX branch, the kernel rotates in
fp32) and that shifted survivors are re-rotated so the position baked into the
key stays consistent (GAP #2). The checks below tie the oracle to numpy's own
IEEE float32/float16 arithmetic and to the rotation group law R(a)R(b) = R(a+b).
"""
import numpy as np


def test_f16_decode_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = orc.f16_bits_to_f64(bits)
    finite = np.isfinite(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(np.isinf(got), np.isinf(want))


def test_f32_to_f16_matches_numpy(orc):
    rng = np.random.default_rng(0)
    xs = [rng.standard_normal(200000).astype(np.float32) * 3,
          (rng.standard_normal(50000) * 1e-5).astype(np.float32),          # subnormal range
          (rng.standard_normal(50000) * 3e4).astype(np.float32),           # near overflow
          np.array([0.0, -0.0, 65504, 65519.996, 65520, 70000, -65520, 2.0**-24, 2.0**-25,
                    3 * 2.0**-26, 2.0**-14, 1 + 2.0**-11, 1 + 3 * 2.0**-11], np.float32)]
    # exact fp16 midpoints: ties must go to even
    h = np.arange(0, 0x7BFF, 7, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    xs.append(((lo + hi) / 2).astype(np.float32))
    x = np.concatenate(xs)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16_bits(x)
    assert np.array_equal(got, want)


def _numpy_fp32_rotate(row_bits, c, s):
    D = row_bits.size
    v = row_bits.view(np.float16).astype(np.float32)
    a, b = v[: D // 2], v[D // 2:]
    x = np.float32(a * c) - np.float32(b * s)      # each op rounds to float32
    y = np.float32(a * s) + np.float32(b * c)
    return np.concatenate([x, y]).astype(np.float16).view(np.uint16)


def test_rope_consts(orc):
    for D in (64, 128):
        c, s = orc.rope_consts(500000.0, D, 0)
        assert np.all(c == 1.0) and np.all(s == 0.0)
        c, s = orc.rope_consts(10000.0, D, -1)
        w = 10000.0 ** (-(2.0 * np.arange(D // 2)) / D)
        assert np.array_equal(c, np.cos(-w).astype(np.float32))
        assert np.array_equal(s, np.sin(-w).astype(np.float32))
        assert s[0] < 0  # delta = -1 turns the fastest pair backwards


def test_rotation_is_fp32_arithmetic(orc):
    rng = np.random.default_rng(1)
    for D, theta, delta in [(64, 1e4, -1), (128, 5e5, -1), (128, 5e5, -37), (128, 1e4, -3000)]:
        c, s = orc.rope_consts(theta, D, delta)
        for _ in range(200):
            row = (rng.standard_normal(D) * 2).astype(np.float16).view(np.uint16)
            assert np.array_equal(orc.rotate_row(row, c, s), _numpy_fp32_rotate(row, c, s))


def _rot64(v, pos, theta):
    D = v.size
    w = theta ** (-(2.0 * np.arange(D // 2)) / D)
    ang = pos * w
    a, b = v[: D // 2], v[D // 2:]
    return np.concatenate([a * np.cos(ang) - b * np.sin(ang), a * np.sin(ang) + b * np.cos(ang)])


def test_rotation_group_law(orc):
    # A key rotated at position P, re-rotated by -1, is the key rotated at P-1
    # (up to fp16 storage): R(-1) R(P) = R(P-1). Pins the pairing, the
    # frequencies and the sign of the shift.
    rng = np.random.default_rng(2)
    for D, theta in [(64, 1e4), (128, 5e5)]:
        c, s = orc.rope_consts(theta, D, -1)
        for P in (1, 5, 100, 2047):
            v = rng.standard_normal(D)
            k_at_p = _rot64(v, P, theta).astype(np.float16).view(np.uint16)
            got = orc.f16_bits_to_f64(orc.rotate_row(k_at_p, c, s))
            want = _rot64(v, P - 1, theta)
            ulp = np.abs(want) * 2.0 ** -10 + 2.0 ** -24
            assert np.all(np.abs(got - want) <= 2 * ulp)
            # and repeated single shifts track R(P-k) with error growing only slowly
            row = k_at_p.copy()
            for _ in range(20):
                row = orc.rotate_row(row, c, s)
            want = _rot64(v, P - 20, theta)
            err = np.abs(orc.f16_bits_to_f64(row) - want)
            assert np.all(err <= 20 * (np.abs(want) * 2.0 ** -10 + 2.0 ** -24) + 1e-2)
