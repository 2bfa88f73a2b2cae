"""Pins for the oracle's layer output stage: binary64 -> bfloat16 / binary32
rounding, exact decoding, and y = round(y_ref + bias).

Expected values come from brute force over every finite bfloat16 value, from
numpy's IEEE conversions, from hand-worked ties, and from closed forms (a
zero row sum returns the bias pattern itself).
"""
import numpy as np

import oracle

BF16, FP16, F32 = oracle.BF16, oracle.FP16, oracle.F32


def _bf16_values():
    """Every finite non-negative bfloat16 value (exact, as float64), by pattern."""
    pats = np.arange(0x7F80, dtype=np.uint32)  # 0x0000 .. 0x7F7F
    return pats, (pats << 16).view(np.float32).astype(np.float64)


def _nearest_bf16_brute(d: float, pats, vals) -> int:
    a = abs(d)
    bf_max = vals[-1]
    half_ulp_max = 2.0 ** (127 - 8)
    sign = 0x8000 if np.signbit(d) else 0
    if a >= bf_max + half_ulp_max:
        return sign | 0x7F80
    i = int(np.searchsorted(vals, a))
    cands = [j for j in (i - 1, i) if 0 <= j < len(vals)]
    best = min(cands, key=lambda j: (abs(vals[j] - a), pats[j] & 1))
    return sign | int(pats[best])


def test_f64_to_bf16_is_the_nearest_bf16_brute_force():
    pats, vals = _bf16_values()
    rng = np.random.default_rng(11)
    d = rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 39, 3000)
    d = np.concatenate([d, rng.standard_normal(300) * 2.0 ** -130,  # bfloat16 subnormals
                        [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 3.3895313892515355e38,
                         3.4e38, -3.39e38, 2.0 ** -134, 2.0 ** -133, 2.0 ** -133 * 1.5]])
    for v in d:
        assert oracle.f64_to_bf16(v) == _nearest_bf16_brute(float(v), pats, vals), v


def test_f64_to_f32_bits_matches_numpy():
    rng = np.random.default_rng(12)
    d = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-44, 38, 5000),
                        [1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, 2.0 ** -150, 2.0 ** -149 * 1.5,
                         -0.0, 3.4028235677973366e38]])
    with np.errstate(over="ignore"):
        ref = d.astype(np.float32).view(np.uint32)
    got = np.array([oracle.f64_to_f32_bits(v) for v in d], np.uint32)
    np.testing.assert_array_equal(got, ref)


def test_decode_is_exact():
    h = np.arange(0, 65536, 97, dtype=np.uint32)
    finite16 = (h & 0x7C00) != 0x7C00
    for b in h[finite16]:
        assert oracle.decode(int(b), FP16) == float(np.uint16(b).view(np.float16))
    finite_bf = (h & 0x7F80) != 0x7F80
    for b in h[finite_bf]:
        assert oracle.decode(int(b), BF16) == float(np.uint32(b << 16).view(np.float32))
    for f in (np.float32(1.5), np.float32(-3.0e-42), np.float32(2.0 ** 100)):
        assert oracle.decode(int(f.view(np.uint32)), F32) == float(f)


def test_worked_roundings_ties_to_even():
    # v = 1 + 2^-8 lies halfway between bfloat16 1.0 (0x3F80) and 1 + 2^-7 (0x3F81)
    v, yb = oracle.gemv_output(np.array([[2.0 ** -8]]), BF16, np.array([0x3F80], np.uint16))
    assert v[0, 0] == 1.0 + 2.0 ** -8 and yb[0, 0] == 0x3F80
    # 1 + 3 * 2^-8: halfway between 0x3F81 and 0x3F82 -> the even 0x3F82
    _, yb = oracle.gemv_output(np.array([[3 * 2.0 ** -8]]), BF16, np.array([0x3F80], np.uint16))
    assert yb[0, 0] == 0x3F82
    # binary16: 1 + 2^-11 -> 0x3C00, 1 + 3 * 2^-11 -> 0x3C02
    _, yb = oracle.gemv_output(np.array([[2.0 ** -11, 3 * 2.0 ** -11]]), FP16,
                               np.array([0x3C00, 0x3C00], np.uint16))
    assert list(yb[0]) == [0x3C00, 0x3C02]
    # 1.0 + bfloat16 1.0 = 2.0 exactly
    _, yb = oracle.gemv_output(np.array([[1.0]]), BF16, np.array([0x3F80], np.uint16))
    assert yb[0, 0] == 0x4000


def test_zero_row_sum_returns_the_bias_pattern():
    """round(0 + b) == b for every finite pattern b (but -0: +0 + -0 = +0)."""
    for dtype, n in ((BF16, 1 << 16), (FP16, 1 << 16)):
        b = np.arange(n, dtype=np.uint32).astype(np.uint16)
        expo = 0x7F80 if dtype == BF16 else 0x7C00
        b = b[((b & expo) != expo) & (b != 0x8000)]
        _, yb = oracle.gemv_output(np.zeros((1, b.size)), dtype, b)
        np.testing.assert_array_equal(yb[0], b.astype(np.uint32))
    rng = np.random.default_rng(13)
    b32 = rng.standard_normal(1000).astype(np.float32).view(np.uint32)
    _, yb = oracle.gemv_output(np.zeros((1, b32.size)), F32, b32)
    np.testing.assert_array_equal(yb[0], b32)
    _, yb = oracle.gemv_output(np.zeros((1, 1)), BF16, np.array([0x8000], np.uint16))
    assert yb[0, 0] == 0x0000


def test_without_bias_is_numpy_rounding():
    rng = np.random.default_rng(14)
    y = rng.standard_normal((3, 500)) * 10.0 ** rng.integers(-6, 4, (3, 500))
    v, yb = oracle.gemv_output(y, FP16)
    assert np.array_equal(v, y)
    with np.errstate(over="ignore"):
        np.testing.assert_array_equal(yb, y.astype(np.float16).view(np.uint16).astype(np.uint32))
    _, yb = oracle.gemv_output(y, F32)
    np.testing.assert_array_equal(yb, y.astype(np.float32).view(np.uint32))


def test_bias_follows_the_listed_rows():
    """With a row list, output i uses bias[rows[i]] (a reversed list reverses the result)."""
    rng = np.random.default_rng(15)
    N = 64
    bias = rng.standard_normal(N).astype(np.float16).view(np.uint16)
    y = rng.integers(-(1 << 20), 1 << 20, (2, N)) * 2.0 ** -20  # sums with the bias are exact
    v_all, yb_all = oracle.gemv_output(y, FP16, bias)
    rows = np.arange(N)[::-1].copy()
    v_rev, yb_rev = oracle.gemv_output(y[:, ::-1].copy(), FP16, bias, rows)
    np.testing.assert_array_equal(v_rev, v_all[:, ::-1])
    np.testing.assert_array_equal(yb_rev, yb_all[:, ::-1])
    # the bias moves every output by exactly its value
    np.testing.assert_array_equal(v_all - y, np.broadcast_to(bias.view(np.float16).astype(np.float64), y.shape))
