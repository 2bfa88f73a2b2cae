"""Second-level table generality: the whole path with a non-linear code2
table (logarithmically spaced magnitudes, oracle.code2_dynamic), which
"NF4反量化算子优化", section "第二层量化", motivates by storing the scales in
an 8-bit floating-point format. The quantizer and the dequantization must be
bit-identical to the oracle, the GEMV within its tolerance, on the 1024x1024
workload and the Llama-7B-shaped layers."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_gemv_close, gpu_dequant, gpu_gemv, to_device

pytestmark = pytest.mark.gpu


def _gpu_quantize(w, code2_bits, bs=64, s2=256):
    import w4a16_gemv_gb300 as nf4
    code2 = torch.from_numpy(code2_bits.view(np.float16)).cuda()
    q = nf4.nf4_quantize(torch.from_numpy(w).cuda(), code2, bs, s2)
    torch.cuda.synchronize()
    return q


def _quantize_both(w):
    table = synth.code2_dynamic()
    ref = oracle.quantize(w, 64, 256, table)
    q = _gpu_quantize(w, table)
    np.testing.assert_array_equal(q.packed.cpu().numpy(), ref.packed)
    np.testing.assert_array_equal(q.absmax_q.cpu().numpy(), ref.absmax_q)
    np.testing.assert_array_equal(q.absmax2.cpu().numpy().view(np.uint16), ref.absmax2)
    assert np.float32(q.offset).view(np.uint32) == np.float32(ref.offset).view(np.uint32)
    # the table is used: block scales land on many different entries
    assert len(np.unique(ref.absmax_q)) > 64
    return ref


def test_table_is_the_oracles():
    np.testing.assert_array_equal(synth.code2_dynamic(), oracle.code2_dynamic())


def test_config0_quantize_and_dequant():
    c = synth.CONFIG0
    ref = _quantize_both(synth.weights(c.seed, c.n))
    for dtype in (oracle.BF16, oracle.FP16):
        np.testing.assert_array_equal(gpu_dequant(ref, dtype), oracle.dequant(ref, dtype))


def test_config0_gemv():
    c = synth.CONFIG0
    ref = oracle.quantize(synth.weights(c.seed, c.n), 64, 256, synth.code2_dynamic())
    N, K = c.shape
    for batch in (1, 4, 8, 16):
        x = synth.activations(900 + batch, batch, K)
        y = gpu_gemv(ref, N, K, x)
        y_ref, s_abs = oracle.gemv(ref, N, K, x)
        assert_gemv_close(y, y_ref, s_abs, f"1024x1024 batch {batch}")


@pytest.mark.parametrize("layer", synth.LLAMA_7B_LAYERS, ids=lambda l: l.name)
def test_config3_layers(layer):
    ref = _quantize_both(synth.weights(layer.seed, layer.N * layer.K))
    idx = np.unique(np.concatenate([np.arange(4096), ref.n - 1 - np.arange(4096),
                                    synth.draws(77, 0, 65536) % ref.n]).astype(np.int64))
    got = gpu_dequant(ref, oracle.BF16)
    np.testing.assert_array_equal(got[idx], oracle.dequant_at(ref, idx, oracle.BF16))
    d = to_device(ref)
    for batch in synth.LLAMA_BATCHES:
        x = synth.activations(synth.llama_x_seed(batch), batch, layer.K)
        y = gpu_gemv(ref, layer.N, layer.K, x, d=d)
        y_ref, s_abs = oracle.gemv(ref, layer.N, layer.K, x)
        assert_gemv_close(y, y_ref, s_abs, f"{layer.name} batch {batch}")
