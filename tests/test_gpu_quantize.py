"""GPU parity for nf4_quantize: packed codes, absmax_q, absmax2 and offset
bit-identical to the CPU oracle's quantizer."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _gpu_quantize(w, bs, s2):
    import w4a16_gemv_gb300 as nf4
    code2 = torch.from_numpy(synth.code2_linear().view(np.float16)).cuda()
    q = nf4.nf4_quantize(torch.from_numpy(w).cuda(), code2, bs, s2)
    torch.cuda.synchronize()
    return q


def _check(w, bs=64, s2=256):
    ref = oracle.quantize(w, bs, s2, synth.code2_linear())
    q = _gpu_quantize(w, bs, s2)
    np.testing.assert_array_equal(q.packed.cpu().numpy(), ref.packed)
    np.testing.assert_array_equal(q.absmax_q.cpu().numpy(), ref.absmax_q)
    np.testing.assert_array_equal(q.absmax2.cpu().numpy().view(np.uint16), ref.absmax2)
    assert np.float32(q.offset).view(np.uint32) == np.float32(ref.offset).view(np.uint32)


def test_config0():
    c = synth.CONFIG0
    _check(synth.weights(c.seed, c.n))


def test_config1_outliers():
    c = synth.CONFIG1
    _check(synth.weights(c.seed, c.n, c.outlier_frac, c.outlier_seed))


def test_ragged_case():
    c = synth.CONFIG4[-1]
    _check(synth.weights(c.seed, c.n))


@pytest.mark.parametrize("n", [1, 2, 3, 64, 65, 999, 64 * 256 + 3])
def test_small_and_odd(n):
    _check(synth.weights(40 + n, n, 0.05, 41))


@pytest.mark.parametrize("bs,s2", [(2, 1), (32, 256), (128, 4), (4096, 2), (64, 1)])
def test_block_sizes(bs, s2):
    _check(synth.weights(50 + bs, 5 * 4096 + 10, 0.01, 51), bs, s2)


def test_zero_blocks_and_exact_codes():
    w = np.zeros(64 * 600, np.float32)
    w[64 * 300:64 * 301] = np.linspace(-1, 1, 64, dtype=np.float32)
    w[-1] = 3.0
    _check(w)


def test_round_trip_through_gpu_dequant():
    """quantize (GPU) -> dequant (GPU) equals the oracle's dequant of its own quantization."""
    import w4a16_gemv_gb300 as nf4
    w = synth.weights(3, 1 << 18)
    q = _gpu_quantize(w, 64, 256)
    out = nf4.dequant(q, torch.float16)
    ref = oracle.quantize(w, 64, 256, synth.code2_linear())
    np.testing.assert_array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16),
                                  oracle.dequant(ref, oracle.FP16))
