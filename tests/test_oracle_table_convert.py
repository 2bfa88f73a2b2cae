"""Pins for the oracle's NF4 code book, code2 table and IEEE conversions.

Nothing here compares the oracle with itself: every expected value comes from
the pages (tests/golden), a closed form, or an independent library routine
(numpy / torch CPU conversions, scipy's normal quantile function).
"""
import math

import numpy as np
import pytest

import oracle
from conftest import read_golden_rows


def _golden_table():
    rows = read_golden_rows("nf4_code_table.txt")
    idx = [int(r[0]) for r in rows]
    assert idx == list(range(16))
    return np.array([float(r[1]) for r in rows]), np.array([float(r[2]) for r in rows])


def test_code_book_equals_printed_literals():
    opt, _ = _golden_table()
    got = oracle.nf4_code()
    assert got.dtype == np.float32
    np.testing.assert_array_equal(got, opt.astype(np.float32))


def test_code_book_matches_second_page_to_its_printed_digits():
    _, rpt = _golden_table()
    assert np.max(np.abs(oracle.nf4_code().astype(np.float64) - rpt)) <= 0.5e-4 + 1e-9


def test_code_book_invariants():
    t = oracle.nf4_code()
    assert t[0] == -1.0 and t[7] == 0.0 and t[15] == 1.0
    assert np.all(np.diff(t) > 0)
    assert np.sum(t > 0) == 8 and np.sum(t < 0) == 7
    gaps = np.diff(t.astype(np.float64))
    assert int(np.argmax(gaps)) == 0
    assert abs(gaps.max() - 0.3038072) < 1e-7


def test_code_book_is_normal_quantiles():
    """The pages build NF4 from equal-probability quantiles of N(0,1), one
    side with 8 codes and the other with 7, an exact zero, scaled to [-1, 1]
    ("NF4反量化算子优化", section "NF4 table").  With the outermost probability
    fitted from a single code, all sixteen printed values follow."""
    from scipy.optimize import brentq
    from scipy.stats import norm

    t = oracle.nf4_code().astype(np.float64)

    def table(d):
        pos = norm.ppf(np.linspace(d, 0.5, 9)[:-1])
        neg = -norm.ppf(np.linspace(d, 0.5, 8)[:-1])
        v = np.sort(np.concatenate([pos, [0.0], neg]))
        return v / np.max(np.abs(v))

    d = brentq(lambda d: table(d)[14] - t[14], 0.9, 0.999)
    assert np.max(np.abs(table(d) - t)) < 5e-7


# ---------------------------------------------------------------------------
# IEEE conversions against numpy / torch CPU

def _sweep_f32(seed=0, count=20000):
    rng = np.random.default_rng(seed)
    u = rng.integers(0, 2 ** 32, count, dtype=np.uint64).astype(np.uint32)
    u = u[(u & 0x7F800000) != 0x7F800000]                       # finite only
    special = np.array([0x00000000, 0x80000000, 0x00000001, 0x807FFFFF, 0x00800000,
                        0x7F7FFFFF, 0xFF7FFFFF, 0x3F808000, 0x3F818000, 0x3F80C000,
                        0x477FEFFF, 0x477FF000, 0x477FE000, 0x33800000, 0x33000000,
                        0x33000001, 0x387FC000, 0x38800000, 0x3F7FFFFF], np.uint32)
    # exact ties for bf16 (low 16 bits 0x8000) and for fp16 (low 13 bits 0x1000)
    ties_bf16 = (rng.integers(0, 2 ** 16, 2000).astype(np.uint32) << 16) | 0x8000
    ties_f16 = ((rng.integers(0x33000000 >> 13, 0x47800000 >> 13, 2000).astype(np.uint32)) << 13) | 0x1000
    allu = np.concatenate([u, special, ties_bf16, ties_f16])
    allu = allu[(allu & 0x7F800000) != 0x7F800000]
    return allu.view(np.float32)


def test_f32_to_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    f = _sweep_f32(1)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(v) for v in f], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_f32_to_f16_matches_numpy():
    f = _sweep_f32(2)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16(v) for v in f], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_f64_to_f16_single_rounding_matches_numpy():
    rng = np.random.default_rng(3)
    d = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-9, 5, 5000),
                        (np.arange(256) - 127.5) / 127.5,
                        # values that double-round differently via binary32
                        np.array([1.0 + 2.0 ** -11 + 2.0 ** -40, 1.0 + 2.0 ** -11 - 2.0 ** -40,
                                  2.0 ** -25 + 2.0 ** -60, 2.0 ** -25, 65519.99, 65520.0])])
    with np.errstate(over="ignore"):
        ref = d.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f64_to_f16(v) for v in d], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_f16_to_f32_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(v)) for v in h], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_to_f32_is_top_half():
    for h in (0x0000, 0x8000, 0x3F80, 0xBF40, 0x0001, 0x7F7F):
        assert np.float32(oracle.bf16_to_f32(h)).view(np.uint32) == np.uint32(h << 16)


# ---------------------------------------------------------------------------
# second-level table

def test_code2_linear_table():
    c = oracle.code2_linear()
    assert c[0] == 0xBC00 and c[255] == 0x3C00          # -1, +1
    assert c[127] == 0x9C04 and c[128] == 0x1C04        # -/+ 1/255 in fp16
    vals = c.view(np.float16).astype(np.float64)
    assert np.all(np.diff(vals) > 0)
    np.testing.assert_array_equal(c[::-1], c ^ 0x8000)  # antisymmetric
    exact = (np.arange(256) - 127.5) / 127.5
    # each entry is within half an fp16 ulp of the exact value
    half_ulp = np.array([2.0 ** (math.floor(math.log2(abs(v))) - 11) for v in exact])
    assert np.all(np.abs(vals - exact) <= half_ulp)


def test_generator_code2_table_matches_oracle():
    import synth
    np.testing.assert_array_equal(synth.code2_linear(), oracle.code2_linear())


def test_code2_dynamic_table():
    """The non-linear second-level table: increasing, antisymmetric, ends at
    -1/+1, powers of two exactly every sixteenth entry, sixteen entries per
    octave, consecutive magnitudes in the ratio 2^(1/16) up to binary16
    rounding."""
    c = oracle.code2_dynamic()
    assert c[0] == 0xBC00 and c[255] == 0x3C00
    np.testing.assert_array_equal(c[::-1], c ^ 0x8000)
    vals = c.view(np.float16).astype(np.float64)
    assert np.all(np.diff(vals) > 0)
    for m in range(8):                      # entry 255 - 16 m is 2^-m, exactly
        assert c[255 - 16 * m] == (15 - m) << 10, m
    pos = vals[128:]
    for m in range(7):                      # 16 entries in each octave [2^-(m+1), 2^-m)
        assert np.count_nonzero((pos >= 2.0 ** -(m + 1)) & (pos < 2.0 ** -m)) == 16
    ratio = pos[1:] / pos[:-1]
    # binary16 carries 11 significant bits: each entry is within 2^-11 relative
    assert np.all(np.abs(ratio / 2.0 ** (1 / 16) - 1) <= 2 * 2.0 ** -11)
    assert 2.0 ** -8 < pos[0] < 2.0 ** -7   # smallest magnitude 2^(-127/16)


def test_generator_code2_dynamic_matches_oracle():
    import synth
    np.testing.assert_array_equal(synth.code2_dynamic(), oracle.code2_dynamic())
