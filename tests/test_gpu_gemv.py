"""GPU parity for nf4_gemv: |y - y_ref| <= 1e-3 * sum|w_hat x| + 1e-6 against
the oracle's binary64 GEMV."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import assert_gemv_close, gpu_gemv, to_device

pytestmark = pytest.mark.gpu


def _layer(layer):
    w = synth.weights(layer.seed, layer.N * layer.K)
    return oracle.quantize(w, 64, 256, synth.code2_linear())


@pytest.mark.parametrize("layer", synth.QWEN_1P5B_LAYERS, ids=lambda l: l.name)
def test_config2_qwen_layers_batch1(layer):
    t = _layer(layer)
    x = synth.activations(synth.QWEN_X_SEED, 1, layer.K)
    y = gpu_gemv(t, layer.N, layer.K, x)
    y_ref, s_abs = oracle.gemv(t, layer.N, layer.K, x)
    assert_gemv_close(y, y_ref, s_abs, layer.name)


@pytest.mark.parametrize("layer", synth.LLAMA_7B_LAYERS, ids=lambda l: l.name)
def test_config3_llama7b_layers(layer):
    t = _layer(layer)
    d = to_device(t)
    for batch in synth.LLAMA_BATCHES:
        x = synth.activations(synth.llama_x_seed(batch), batch, layer.K)
        y = gpu_gemv(t, layer.N, layer.K, x, d=d)
        y_ref, s_abs = oracle.gemv(t, layer.N, layer.K, x)
        assert_gemv_close(y, y_ref, s_abs, f"{layer.name} batch {batch}")


@pytest.mark.parametrize("K", [1536, 4096, 1032, 1040, 4104, 70, 2, 8960])
@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 6, 7, 8])
def test_all_batches_and_chunk_widths(K, batch):
    """Every batch size with K values that select each chunk width (16, 8, 4
    packed bytes per lane) and the generic kernel (K % 8 != 0)."""
    N = 37
    w = synth.weights(500 + K, N * K, 0.001, 501)
    t = oracle.quantize(w, 64, 256, synth.code2_linear())
    x = synth.activations(600 + batch, batch, K)
    y = gpu_gemv(t, N, K, x)
    y_ref, s_abs = oracle.gemv(t, N, K, x)
    assert_gemv_close(y, y_ref, s_abs, f"N={N} K={K} batch={batch}")


@pytest.mark.parametrize("N,K", [(1536, 512), (4096, 4096), (37, 1536), (300, 8960), (1000, 40)])
def test_batch1_binary32_x_fallback(N, K):
    """x whose first 32-element chunk spans 2^60 .. 2^-60: no power-of-two
    scaling of the chunk fits binary16, so every CTA of the batch-1 kernel
    takes its binary32-x path (and K = 40 the generic kernel)."""
    w = synth.weights(720 + K, N * K)
    t = oracle.quantize(w, 64, 256, synth.code2_linear())
    x = synth.activations(820 + K, 1, K).copy()
    x[0, 0] = 0x5D80                                # bf16 2^60
    x[0, 1] = 0x2180                                # bf16 2^-60
    y = gpu_gemv(t, N, K, x)
    y_ref, s_abs = oracle.gemv(t, N, K, x)
    assert_gemv_close(y, y_ref, s_abs, f"N={N} K={K}")


@pytest.mark.parametrize("N", [1, 2, 7, 31, 32, 33, 255, 256, 257, 1000])
def test_row_counts(N):
    K = 1536
    w = synth.weights(700 + N, N * K)
    t = oracle.quantize(w, 64, 256, synth.code2_linear())
    for batch in (1, 4):
        x = synth.activations(800 + N, batch, K)
        y = gpu_gemv(t, N, K, x)
        y_ref, s_abs = oracle.gemv(t, N, K, x)
        assert_gemv_close(y, y_ref, s_abs, f"N={N} batch={batch}")


@pytest.mark.parametrize("bs,s2", [(32, 256), (128, 4), (16, 256), (8, 1), (2, 1), (4096, 1)])
def test_block_sizes(bs, s2):
    N, K = 40, 4096
    w = synth.weights(900 + bs, N * K, 0.001, 901)
    t = oracle.quantize(w, bs, s2, synth.code2_linear())
    for batch in (1, 3):
        x = synth.activations(902, batch, K)
        y = gpu_gemv(t, N, K, x)
        y_ref, s_abs = oracle.gemv(t, N, K, x)
        assert_gemv_close(y, y_ref, s_abs, f"bs={bs} s2={s2} batch={batch}")


@pytest.mark.parametrize("K, bs, batch, x_offset", [(1040, 16, 12, 0), (70, 2, 9, 0),
                                                    (1536, 32, 20, 0), (1536, 64, 17, 1)])
def test_wide_batches_in_slabs(K, bs, batch, x_offset):
    """Batches above 8 that the tensor-core kernel does not take (K not a
    multiple of 64, block sizes below 64, x not 16-byte aligned) run as slabs
    of at most eight vectors through the CUDA-core kernels."""
    N = 45
    t = oracle.quantize(synth.weights(1000 + K, N * K, 0.001, 1001), bs, 256, synth.code2_linear())
    x = synth.activations(1002 + batch, batch, K)
    y = gpu_gemv(t, N, K, x, x_offset=x_offset)
    y_ref, s_abs = oracle.gemv(t, N, K, x)
    assert_gemv_close(y, y_ref, s_abs, f"K={K} bs={bs} batch={batch} x_offset={x_offset}")


def test_ragged_k_blocks_straddle_rows():
    """K = 1000 is not a multiple of 64: blocks straddle rows (generic kernel)."""
    N, K = 33, 1000
    w = synth.weights(950, N * K)
    t = oracle.quantize(w, 64, 256, synth.code2_linear())
    x = synth.activations(951, 2, K)
    y = gpu_gemv(t, N, K, x)
    y_ref, s_abs = oracle.gemv(t, N, K, x)
    assert_gemv_close(y, y_ref, s_abs)


def test_misaligned_x_and_zero_k():
    N, K = 64, 1536
    w = synth.weights(960, N * K)
    t = oracle.quantize(w, 64, 256, synth.code2_linear())
    x = synth.activations(961, 1, K)
    y = gpu_gemv(t, N, K, x, x_offset=1)
    y_ref, s_abs = oracle.gemv(t, N, K, x)
    assert_gemv_close(y, y_ref, s_abs, "misaligned x")
    y0 = gpu_gemv(t, N, 0, np.zeros((2, 0), np.uint16))
    assert np.all(y0 == 0.0)


def test_special_inputs():
    """x = 0 gives y = 0; a one-hot x gives the dequantized column."""
    N, K = 128, 4096
    w = synth.weights(970, N * K)
    t = oracle.quantize(w, 64, 256, synth.code2_linear())
    y = gpu_gemv(t, N, K, np.zeros((1, K), np.uint16))
    assert np.all(y == 0.0)
    W = oracle.dequant_f32(t).reshape(N, K).astype(np.float64)
    x = np.zeros((3, K), np.uint16)
    cols = [0, 1, 4095]
    for b, c in enumerate(cols):
        x[b, c] = 0x3F80                           # bf16 1.0
    y = gpu_gemv(t, N, K, x)
    for b, c in enumerate(cols):
        np.testing.assert_allclose(y[b], W[:, c], rtol=1e-3, atol=1e-6)


def test_no_device_error_flags_after_gemv():
    """No bounded wait of the streaming GEMV ran out during the tests above."""
    import w4a16_gemv_gb300 as nf4
    N, K = 4096, 4096
    w = synth.weights(990, N * K)
    t = oracle.quantize(w, 64, 256, synth.code2_linear())
    x = synth.activations(991, 1, K)
    y = gpu_gemv(t, N, K, x)
    assert nf4.nf4_device_error_flags() == 0
    y_ref, s_abs = oracle.gemv(t, N, K, x)
    assert_gemv_close(y, y_ref, s_abs)
