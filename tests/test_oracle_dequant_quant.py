"""Pins for the oracle's dequantization, quantization and GEMV.

Expected values come from hand-worked examples of the pages' formula
(tests/golden/dequant_worked_examples.txt), exact power-of-two scaling,
brute force on tiny inputs, closed-form bounds and numpy's float64 matmul.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from conftest import read_golden_rows

F16_ONE = 0x3C00


def _f16(v):
    return int(np.float16(v).view(np.uint16))


def _tensor(packed, absmax_q, absmax2, offset, n, bs=64, s2=256, code2=None):
    return oracle.NF4Tensor(np.asarray(packed, np.uint8), np.asarray(absmax_q, np.uint8),
                            np.asarray(absmax2, np.uint16),
                            oracle.code2_linear() if code2 is None else np.asarray(code2, np.uint16),
                            float(np.float32(offset)), n, bs, s2)


def _expected_16bit(values_f64, dtype):
    """Round exact binary64 values to bf16 / fp16 with library routines."""
    import torch
    v = np.asarray(values_f64, np.float64)
    if dtype == oracle.FP16:
        return v.astype(np.float16).view(np.uint16)
    # bf16: binary64 -> binary32 is exact for all values used here
    assert np.all(v.astype(np.float32).astype(np.float64) == v)
    return torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _one_block_all_codes(q, a2, offset):
    """32 bytes = 64 elements: element 2j holds code j%16 (high nibble), odd = 15-j%16."""
    packed = np.array([((j % 16) << 4) | (15 - j % 16) for j in range(32)], np.uint8)
    return _tensor(packed, [q], [a2], offset, 64)


# ---------------------------------------------------------------------------
# dequantization

@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_worked_examples_from_formula(dtype):
    for name, q, a2, off, s in read_golden_rows("dequant_worked_examples.txt"):
        s = float(s)
        t = _one_block_all_codes(int(q), _f16(float(a2)), float(off))
        got = oracle.dequant(t, dtype)
        idx = np.array([(j // 2) % 16 if j % 2 == 0 else 15 - (j // 2) % 16 for j in range(64)])
        # one binary32 multiply (numpy, IEEE RNE) of the code by the
        # hand-evaluated scale, then the 16-bit rounding by library routines
        v32 = oracle.nf4_code()[idx] * np.float32(s)
        np.testing.assert_array_equal(got, _expected_16bit(v32.astype(np.float64), dtype), err_msg=name)



def test_worked_example_non_dyadic_scale():
    """absmax_q 200, absmax2 binary16(0.01), offset binary32(0.03): the scale
    is not a power-of-two combination, so every binary32 rounding of the
    formula's steps matters (tests/golden/dequant_nondyadic_example.txt)."""
    t = _one_block_all_codes(200, _f16(0.01), float(np.float32(0.03)))
    assert t.absmax2[0] == 0x211F and oracle.code2_linear()[200] == 0x388D
    bf = oracle.dequant(t, oracle.BF16)
    hf = oracle.dequant(t, oracle.FP16)
    # element 2j holds code j % 16 (high nibble of byte j)
    for idx, e_bf, e_hf in read_golden_rows("dequant_nondyadic_example.txt"):
        el = 2 * int(idx)
        assert bf[el] == int(e_bf, 16), (idx, hex(bf[el]))
        assert hf[el] == int(e_hf, 16), (idx, hex(hf[el]))
    # the decoded block scale itself, bit for bit
    assert np.float32(oracle.block_scale(t, 0)).view(np.uint32) == 0x3D122F5A

def test_nibble_order_bytes():
    s = 0.75
    for byte, (e0, e1) in {0x0F: (-s, s), 0xF0: (s, -s), 0x7F: (0.0, s), 0xF7: (s, 0.0)}.items():
        t = _tensor([byte], [255], [_f16(0.25)], 0.5, 2)
        got = oracle.dequant_f32(t)
        assert got[0] == e0 and got[1] == e1, hex(byte)


def test_block_and_group_indexing():
    """Blocks of 64 flattened elements, groups of 256 blocks; block 256 is the
    first of group 1 and must use absmax2[1]."""
    nb = 258
    n = nb * 64 - 10                     # ragged: last block partial
    packed = np.full((n + 1) // 2, 0xFF, np.uint8)       # every element code 15 (= +1)
    q = np.where(np.arange(nb) % 2 == 0, 255, 0).astype(np.uint8)   # code2 = +1 / -1
    a2 = np.array([_f16(0.25), _f16(2.0)], np.uint16)
    off = 4.0
    t = _tensor(packed, q, a2, off, n)
    v = oracle.dequant_f32(t)
    b = np.arange(n) // 64
    g = b // 256
    sign = np.where(b % 2 == 0, 1.0, -1.0)
    exp = sign * np.where(g == 0, 0.25, 2.0) + off
    np.testing.assert_array_equal(v.astype(np.float64), exp)
    # and with other power-of-two block sizes
    t2 = _tensor(packed, np.tile(q, 3)[: (n + 31) // 32], a2, off, n, bs=32, s2=4)
    v2 = oracle.dequant_f32(t2)
    b2 = np.arange(n) // 32
    exp2 = np.where(b2 % 2 == 0, 1.0, -1.0) * np.where(b2 // 4 == 0, 0.25, 2.0) + off
    mask = b2 // 4 <= 1
    np.testing.assert_array_equal(v2[mask].astype(np.float64), exp2[mask])


def test_negative_zero_and_extremes():
    t = _one_block_all_codes(0, F16_ONE, 0.5)                # s = -1 + 0.5 = -0.5
    bf = oracle.dequant(t, oracle.BF16)
    hf = oracle.dequant(t, oracle.FP16)
    # element 14 has code 7 (zero), times a negative scale: -0.0
    assert bf[14] == 0x8000 and hf[14] == 0x8000
    # code 0 -> -s = +0.5, code 15 -> +s = -0.5, exactly
    assert bf[0] == 0x3F00 and hf[0] == 0x3800        # element 0: code 0
    assert bf[1] == 0xBF00 and hf[1] == 0xB800        # element 1: code 15


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_power_of_two_scales_are_exact(dtype):
    """s = 2^k (code2=+1, absmax2=2^k, offset 0): out = RNE(NF4 * 2^k), the
    product being exact.  Covers fp16 subnormals for small k."""
    code = oracle.nf4_code().astype(np.float64)
    for k in range(-24, 16):
        if dtype == oracle.FP16 and k > 14:
            continue
        a2 = np.float16(2.0 ** k) if k >= -24 else None
        if a2 == 0:
            continue
        t = _one_block_all_codes(255, int(a2.view(np.uint16)), 0.0)
        got = oracle.dequant(t, dtype)
        idx = np.array([(j // 2) % 16 if j % 2 == 0 else 15 - (j // 2) % 16 for j in range(64)])
        np.testing.assert_array_equal(got, _expected_16bit(code[idx] * 2.0 ** k, dtype), err_msg=str(k))


def test_exhaustive_bytes_by_code2_invariants():
    """All 256 byte values x all 256 absmax_q values: codes 7 -> +-0, 0 -> -s,
    15 -> +s (bit-exact), monotone in the code, and within the rounding
    bound of the exact binary64 formula."""
    code = oracle.nf4_code().astype(np.float64)
    c2 = oracle.code2_linear().view(np.float16).astype(np.float64)
    a2 = _f16(0.0123)
    off = np.float32(0.0371)
    a2v = float(np.uint16(a2).view(np.float16))
    packed = np.tile(np.arange(256, dtype=np.uint8), 256)             # 32 bytes per block
    q = np.repeat(np.arange(256, dtype=np.uint8), 8)                  # 8 blocks per q value
    n = packed.size * 2
    t = _tensor(packed, q, [a2] * 8, off, n)
    v = oracle.dequant_f32(t).astype(np.float64)
    bf = oracle.dequant(t, oracle.BF16).view(np.uint16)
    k = np.arange(n)
    byte = packed[k // 2].astype(np.int64)
    idx = np.where(k % 2 == 0, byte >> 4, byte & 15)
    s_exact = c2[q[k // 64]] * a2v + float(off)
    # binary32 pipeline vs the exact value: three roundings of 2^-24 each
    assert np.all(np.abs(v - code[idx] * s_exact) <= 4 * 2.0 ** -24 * np.abs(s_exact) + 1e-30)
    # within each block every code-15 element is the same value s_b (x 1.0 is
    # exact) and every code-0 element is exactly -s_b
    blk = k // 64
    hi = np.full(blk[-1] + 1, np.nan)
    hi[blk[idx == 15]] = v[idx == 15]
    np.testing.assert_array_equal(v[idx == 15], hi[blk[idx == 15]])
    np.testing.assert_array_equal(v[idx == 0], -hi[blk[idx == 0]])
    zero = v[idx == 7]
    assert np.all(zero == 0.0)
    assert np.array_equal(np.signbit(zero), np.signbit(s_exact[idx == 7]) & (s_exact[idx == 7] != 0))
    # monotone in the code within each block
    for b in range(0, 2048, 97):
        sel = blk == b
        order = np.argsort(idx[sel], kind="stable")
        vals = v[sel][order]
        if s_exact[sel][0] >= 0:
            assert np.all(np.diff(vals) >= 0)
        else:
            assert np.all(np.diff(vals) <= 0)
    # bf16 output is the RNE of the binary32 value
    import torch
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bf, ref)


# ---------------------------------------------------------------------------
# quantization

def test_nearest_code_ties_and_midpoints():
    t = oracle.nf4_code()
    for j in range(16):
        assert oracle.nf4_nearest(t[j]) == j
    # exact midpoints representable in binary32: ties go to the lower index
    assert oracle.nf4_nearest(np.float32(t[8] / 2)) == 7
    assert oracle.nf4_nearest(np.float32(t[6] / 2)) == 6
    assert oracle.nf4_nearest(np.nextafter(np.float32(t[8] / 2), np.float32(1))) == 8
    assert oracle.nf4_nearest(np.nextafter(np.float32(t[6] / 2), np.float32(-1))) == 6
    assert oracle.nf4_nearest(2.0) == 15 and oracle.nf4_nearest(-3.0) == 0


def test_quantize_recovers_exact_codes():
    """Weights that are exact codes times a block scale (each block holding a
    +-1 code so its absmax is the scale) quantize back to the same codes."""
    rng = np.random.default_rng(7)
    code = oracle.nf4_code()
    n = 64 * 40 + 18
    idx = rng.integers(0, 16, n)
    idx[::64] = 15
    scales = (2.0 ** rng.integers(-12, 2, (n + 63) // 64)).astype(np.float32)
    w = (code[idx] * scales[np.arange(n) // 64]).astype(np.float32)
    absmax = oracle.block_absmax(w, 64)
    np.testing.assert_array_equal(absmax, scales)
    packed = oracle.nf4_encode(w, absmax, 64)
    k = np.arange(n)
    got = np.where(k % 2 == 0, packed[k // 2] >> 4, packed[k // 2] & 15)
    np.testing.assert_array_equal(got, idx)
    if n % 2:
        assert packed[-1] & 15 == 0


def _config0_like(n=64 * 256 * 3 + 64 * 5 + 17, seed=11, code2=None):
    w = synth.weights(seed, n, 0.001, seed + 1)
    if code2 is None:
        return w, oracle.quantize(w, 64, 256)
    return w, oracle.quantize(w, 64, 256, code2)


@pytest.mark.parametrize("table", ["linear", "dynamic"])
def test_quantizer_properties(table):
    w, t = _config0_like(code2=None if table == "linear" else oracle.code2_dynamic())
    assert table == "linear" or np.array_equal(t.code2, oracle.code2_dynamic())
    n = w.size
    bs, s2 = 64, 256
    nb = (n + bs - 1) // bs
    absmax = np.array([np.max(np.abs(w[b * bs:(b + 1) * bs])) for b in range(nb)], np.float32)
    # offset: binary32 of the mean (exact mean via fsum)
    exact_mean = math.fsum(absmax.astype(np.float64)) / nb
    assert t.offset == float(np.float32(exact_mean))
    # absmax2: fp16 of the largest |absmax - offset| in each group
    ng = (nb + s2 - 1) // s2
    assert t.absmax2.size == ng
    for g in range(ng):
        m = np.max(np.abs(absmax[g * s2:(g + 1) * s2] - np.float32(t.offset)))
        assert t.absmax2[g] == np.float32(m).astype(np.float16).view(np.uint16)
    # absmax_q: brute-force nearest code2 entry (ties to the lower index)
    c2 = t.code2.view(np.float16).astype(np.float64)
    a2 = t.absmax2.view(np.float16).astype(np.float32)
    r = (absmax - np.float32(t.offset)) / a2[np.arange(nb) // s2]
    d = np.abs(r.astype(np.float64)[:, None] - c2[None, :])
    np.testing.assert_array_equal(t.absmax_q, np.argmin(d, axis=1))
    # every full block has its absmax element on code 0 or 15
    k = np.arange(n)
    idx = np.where(k % 2 == 0, t.packed[k // 2] >> 4, t.packed[k // 2] & 15)
    for b in range(nb - 1):
        j = b * bs + int(np.argmax(np.abs(w[b * bs:(b + 1) * bs])))
        assert idx[j] == (15 if w[j] > 0 else 0)


def test_round_trip_bound():
    """|w - w_hat| <= (max half gap) * absmax + |absmax - s|, where the scale
    error is at most half a code2 step (1/255 of absmax2) plus fp16 and fp32
    rounding."""
    w, t = _config0_like(seed=12)
    n = w.size
    w_hat = oracle.dequant_f32(t).astype(np.float64)
    b = np.arange(n) // 64
    absmax = np.array([np.max(np.abs(w[i * 64:(i + 1) * 64])) for i in range(b[-1] + 1)])
    s = np.array([oracle.block_scale(t, i) for i in range(b[-1] + 1)])
    a2 = t.absmax2.view(np.float16).astype(np.float64)[np.arange(b[-1] + 1) // 256]
    scale_err = np.abs(absmax - s)
    assert np.all(scale_err <= a2 * (1 / 255 + 2.0 ** -11) + 4 * 2.0 ** -24 * np.abs(s))
    bound = 0.1519036 * absmax[b] + scale_err[b] + 2 * 2.0 ** -24 * np.abs(s[b])
    assert np.all(np.abs(w.astype(np.float64) - w_hat) <= bound * (1 + 1e-6))


def test_round_trip_bound_dynamic_table():
    """With the non-linear table the second-level error of block b is at most
    half the gap between the two table entries around r = (absmax - offset) /
    absmax2, times absmax2 (plus binary32 rounding); the element bound is the
    same as for the linear table."""
    w, t = _config0_like(seed=13, code2=oracle.code2_dynamic())
    n = w.size
    nb = (n + 63) // 64
    c2 = oracle.code2_dynamic().view(np.float16).astype(np.float64)
    absmax = np.array([np.max(np.abs(w[i * 64:(i + 1) * 64])) for i in range(nb)])
    s = np.array([oracle.block_scale(t, i) for i in range(nb)])
    a2 = t.absmax2.view(np.float16).astype(np.float64)[np.arange(nb) // 256]
    r = (absmax - t.offset) / a2
    j = np.clip(np.searchsorted(c2, r), 1, 255)
    gap = c2[j] - c2[j - 1]
    scale_err = np.abs(absmax - s)
    assert np.all(scale_err <= a2 * (gap / 2 + 2.0 ** -11) + 4 * 2.0 ** -24 * np.abs(s))
    w_hat = oracle.dequant_f32(t).astype(np.float64)
    b = np.arange(n) // 64
    bound = 0.1519036 * absmax[b] + scale_err[b] + 2 * 2.0 ** -24 * np.abs(s[b])
    assert np.all(np.abs(w.astype(np.float64) - w_hat) <= bound * (1 + 1e-6))


def test_zero_blocks():
    w = np.zeros(64 * 300, np.float32)
    w[64 * 299 + 3] = 0.5
    t = oracle.quantize(w)
    v = oracle.dequant_f32(t)
    k = np.arange(w.size)
    idx = np.where(k % 2 == 0, t.packed[k // 2] >> 4, t.packed[k // 2] & 15)
    assert np.all(idx[: 64 * 299] == 7)
    assert np.all(v[: 64 * 299] == 0.0)


# ---------------------------------------------------------------------------
# GEMV

def _gemv_case(N, K, batch, seed):
    w = synth.weights(seed, N * K)
    t = oracle.quantize(w)
    x = synth.activations(seed + 1000, batch, K)
    return t, x


@pytest.mark.parametrize("N,K,batch", [(7, 128, 1), (5, 192, 3), (3, 70, 2), (1, 2, 1)])
def test_gemv_matches_numpy_float64_matmul(N, K, batch):
    t, x = _gemv_case(N, K, batch, 5 + N)
    y, s = oracle.gemv(t, N, K, x)
    W = oracle.dequant_f32(t).astype(np.float64).reshape(N, K)
    X = x.astype(np.uint32) << 16
    X = X.view(np.float32).astype(np.float64)
    y_np = X @ W.T
    s_np = np.abs(X)[:, None, :] * np.abs(W)[None, :, :]
    np.testing.assert_allclose(y, y_np, rtol=0, atol=1e-13 * (1 + s_np.sum(-1).max()))
    np.testing.assert_allclose(s, s_np.sum(-1), rtol=1e-13)
    assert np.all(s >= np.abs(y) * (1 - 1e-15))


@pytest.mark.parametrize("N,K,batch", [(7, 128, 1), (5, 192, 3), (3, 70, 2)])
def test_gemv_abs_matches_numpy_float64_matmul(N, K, batch):
    t, _ = _gemv_case(N, K, batch, 40 + N)
    e = np.random.default_rng(N).random((batch, K)) * 10.0 ** np.random.default_rng(K).integers(-6, 2, K)
    a = oracle.gemv_abs(t, N, K, e)
    W = np.abs(oracle.dequant_f32(t).astype(np.float64).reshape(N, K))
    np.testing.assert_allclose(a, e @ W.T, rtol=1e-13, atol=0)
    # one-hot e picks |column j| exactly
    for j in (0, K - 1):
        oh = np.zeros((1, K))
        oh[0, j] = 1.0
        np.testing.assert_array_equal(oracle.gemv_abs(t, N, K, oh)[0], W[:, j])


def test_gemv_special_cases():
    N, K = 6, 256
    # every block scale is 0.25 * 1 + 0.5 = 0.75: w_hat = fp32(code * 0.75)
    packed = np.random.default_rng(1).integers(0, 256, N * K // 2).astype(np.uint8)
    t = _tensor(packed, [255] * (N * K // 64), [_f16(0.25)], 0.5, N * K)
    k = np.arange(N * K)
    idx = np.where(k % 2 == 0, packed[k // 2] >> 4, packed[k // 2] & 15)
    W = (oracle.nf4_code()[idx] * np.float32(0.75)).astype(np.float64).reshape(N, K)
    for col in (0, 1, 131, 255):
        x = np.zeros((1, K), np.uint16)
        x[0, col] = 0x3F80                            # bf16 1.0
        y, _ = oracle.gemv(t, N, K, x)
        np.testing.assert_array_equal(y[0], W[:, col])
    y0, s0 = oracle.gemv(t, N, K, np.zeros((1, K), np.uint16))
    assert np.all(y0 == 0) and np.all(s0 == 0)
    # batch rows are independent; doubling x doubles y exactly
    xb = synth.activations(9, 3, K)
    yb, _ = oracle.gemv(t, N, K, xb)
    for b in range(3):
        y1, _ = oracle.gemv(t, N, K, xb[b:b + 1])
        np.testing.assert_array_equal(yb[b], y1[0])
    x2 = (xb.astype(np.uint32) + (1 << 7)).astype(np.uint16)     # exponent + 1 => x * 2
    y2, _ = oracle.gemv(t, N, K, x2)
    np.testing.assert_array_equal(y2, 2 * yb)
    # sampled rows equal the full result
    rows = np.array([5, 0, 3])
    yr, sr = oracle.gemv(t, N, K, xb, rows=rows)
    np.testing.assert_array_equal(yr, yb[:, rows])


def test_dequant_at_matches_full():
    w, t = _config0_like(n=64 * 300 + 7, seed=13)
    full = oracle.dequant(t, oracle.FP16)
    idx = np.array([0, 1, 63, 64, 64 * 256, 64 * 300 + 6, 9999])
    np.testing.assert_array_equal(oracle.dequant_at(t, idx, oracle.FP16), full[idx])
