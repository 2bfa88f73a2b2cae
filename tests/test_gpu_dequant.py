"""GPU parity for nf4_dequant: bit-exact against the CPU oracle."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import gpu_dequant

pytestmark = pytest.mark.gpu


def _f16(v):
    return int(np.float16(v).view(np.uint16))


def _quant_case(case: synth.DequantCase):
    w = synth.weights(case.seed, case.n, case.outlier_frac, case.outlier_seed)
    return oracle.quantize(w, 64, 256, synth.code2_linear())


def _compare_full(t, dtype):
    got = gpu_dequant(t, dtype)
    exp = oracle.dequant(t, dtype)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}: got {got[bad[:5]]} exp {exp[bad[:5]]}"


def _compare_sampled(t, dtype, seed=0, count=1 << 20):
    got = gpu_dequant(t, dtype)
    rng = np.random.default_rng(seed)
    idx = np.unique(np.concatenate([np.arange(min(t.n, 65536)), np.arange(max(0, t.n - 65536), t.n),
                                    rng.integers(0, t.n, count)]))
    exp = oracle.dequant_at(t, idx, dtype)
    bad = np.nonzero(got[idx] != exp)[0]
    assert bad.size == 0, f"{bad.size} sampled mismatches, first at {idx[bad[:5]]}"


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("a2,off", [(0.0123, 0.0371), (1.0, -0.5), (6e-5, 0.0), (60000.0, 0.0),
                                    (0.25, 0.5)])
def test_exhaustive_bytes_by_absmax_q(dtype, a2, off):
    """All 256 packed bytes x all 256 absmax_q values, several scale settings
    (fp16 subnormal outputs, overflow to infinity, negative scales, -0.0)."""
    packed = np.tile(np.arange(256, dtype=np.uint8), 256)
    q = np.repeat(np.arange(256, dtype=np.uint8), 8)
    n = packed.size * 2
    code2 = synth.code2_linear() if a2 != 60000.0 else \
        np.where(np.arange(256) < 128, _f16(-2.0), _f16(2.0)).astype(np.uint16)
    t = oracle.NF4Tensor(packed, q, np.array([_f16(a2)] * 8, np.uint16), code2,
                         float(np.float32(off)), n)
    _compare_full(t, dtype)


def test_config0_1024x1024_bf16():
    _compare_full(_quant_case(synth.CONFIG0), oracle.BF16)


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_config1_4096x4096_outliers(dtype):
    _compare_full(_quant_case(synth.CONFIG1), dtype)


@pytest.mark.parametrize("layer", synth.QWEN_1P5B_LAYERS, ids=lambda l: l.name)
def test_config2_qwen_layer_dequant(layer):
    w = synth.weights(layer.seed, layer.N * layer.K)
    _compare_full(oracle.quantize(w, 64, 256, synth.code2_linear()), oracle.BF16)


@pytest.mark.parametrize("case", [c for c in synth.CONFIG4 if c.n <= (1 << 26)], ids=lambda c: c.name)
def test_config4_sweep_full(case):
    _compare_full(_quant_case(case), oracle.BF16)


@pytest.mark.slow
@pytest.mark.parametrize("case", [c for c in synth.CONFIG4 if c.n > (1 << 26)], ids=lambda c: c.name)
def test_config4_sweep_large_sampled(case):
    _compare_sampled(_quant_case(case), oracle.BF16)


@pytest.mark.parametrize("n", [1, 2, 3, 5, 63, 64, 65, 127, 1023, 1024, 1025, 1536, 2047, 2055,
                               64 * 256 + 1, 64 * 256 * 2 + 33, 4 * 1024 * 3 + 999])
@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_ragged_sizes(n, dtype):
    w = synth.weights(1000 + n, n, 0.01, 2000 + n)
    _compare_full(oracle.quantize(w, 64, 256, synth.code2_linear()), dtype)


@pytest.mark.parametrize("bs,s2", [(2, 1), (4, 2), (8, 256), (16, 3 + 1), (32, 256), (128, 256),
                                   (256, 1), (4096, 2), (64, 1), (64, 1024)])
def test_other_block_sizes(bs, s2):
    n = 3 * 4096 + 70
    w = synth.weights(77 + bs, n, 0.01, 78)
    t = oracle.quantize(w, bs, s2, synth.code2_linear())
    for dtype in (oracle.BF16, oracle.FP16):
        _compare_full(t, dtype)


@pytest.mark.parametrize("out_offset,packed_offset", [(1, 0), (0, 1), (0, 2), (3, 3), (8, 4)])
def test_misaligned_buffers(out_offset, packed_offset):
    n = 5000
    w = synth.weights(31, n)
    t = oracle.quantize(w, 64, 256, synth.code2_linear())
    got = gpu_dequant(t, oracle.BF16, out_offset=out_offset, packed_offset=packed_offset)
    np.testing.assert_array_equal(got, oracle.dequant(t, oracle.BF16))


def test_stream_and_graph_capture():
    """Runs on the caller's stream and replays inside a CUDA graph."""
    import torch
    import w4a16_gemv_gb300 as nf4
    from gpu_helpers import to_device
    t = _quant_case(synth.CONFIG0)
    d = to_device(t)
    out = torch.empty(t.n, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        nf4.nf4_dequant(d["packed"], d["absmax_q"], d["absmax2"], d["code2"], t.offset, t.n, out=out)
    s.synchronize()
    exp = oracle.dequant(t, oracle.BF16)
    np.testing.assert_array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), exp)
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nf4.nf4_dequant(d["packed"], d["absmax_q"], d["absmax2"], d["code2"], t.offset, t.n, out=out)
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), exp)
