"""GPU parity for nf4_gemv_ex, the GEMV with the layer's output stage fused
(bias, and y in bfloat16, binary16 or binary32), against the oracle's binary64
GEMV and output stage."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import (assert_gemv_close, assert_layer_close, gpu_gemv, gpu_gemv_ex,
                         to_device)

pytestmark = pytest.mark.gpu

DTYPES = {"bf16": oracle.BF16, "fp16": oracle.FP16, "f32": oracle.F32}


def _quantized(seed, N, K, outliers=0.0):
    w = synth.weights(seed, N * K, outliers, seed + 1)
    return oracle.quantize(w, 64, 256, synth.code2_linear())


@pytest.mark.parametrize("layer", synth.QWEN_1P5B_LAYERS, ids=lambda l: l.name)
def test_qwen_layers_with_bias_every_output_type(layer):
    t = _quantized(layer.seed, layer.N, layer.K)
    d = to_device(t)
    x = synth.activations(synth.QWEN_X_SEED, 1, layer.K)
    y_ref, s_abs = oracle.gemv(t, layer.N, layer.K, x)
    for name, dt in DTYPES.items():
        b = synth.bias(70 + layer.seed, layer.N, name)
        y = gpu_gemv_ex(t, layer.N, layer.K, x, dt, b, d=d)
        assert_layer_close(y, y_ref, s_abs, dt, b, f"{layer.name} {name} + bias")
        y = gpu_gemv_ex(t, layer.N, layer.K, x, dt, None, d=d)
        assert_layer_close(y, y_ref, s_abs, dt, None, f"{layer.name} {name}")


@pytest.mark.parametrize("layer", synth.LLAMA_7B_LAYERS, ids=lambda l: l.name)
def test_llama_layers_bf16_and_fp16_with_bias(layer):
    t = _quantized(layer.seed, layer.N, layer.K)
    d = to_device(t)
    for batch in synth.LLAMA_BATCHES:
        x = synth.activations(synth.llama_x_seed(batch), batch, layer.K)
        y_ref, s_abs = oracle.gemv(t, layer.N, layer.K, x)
        for name in ("bf16", "fp16"):
            dt = DTYPES[name]
            b = synth.bias(80 + batch, layer.N, name)
            y = gpu_gemv_ex(t, layer.N, layer.K, x, dt, b, d=d)
            assert_layer_close(y, y_ref, s_abs, dt, b, f"{layer.name} batch {batch} {name}")


@pytest.mark.parametrize("K", [1536, 1040, 4104, 70, 8960])
@pytest.mark.parametrize("batch", [1, 2, 3, 5, 8])
def test_every_kernel_path(K, batch):
    """K values that select the batch-1 / batched streaming kernels, the
    row-streaming kernel (each chunk width) and the generic kernel."""
    N = 37
    t = _quantized(510 + K, N, K, 0.001)
    d = to_device(t)
    x = synth.activations(610 + batch, batch, K)
    y_ref, s_abs = oracle.gemv(t, N, K, x)
    for name, dt in DTYPES.items():
        b = synth.bias(620 + K, N, name)
        y = gpu_gemv_ex(t, N, K, x, dt, b, d=d)
        assert_layer_close(y, y_ref, s_abs, dt, b, f"K={K} batch={batch} {name}")


@pytest.mark.parametrize("N", [1, 31, 257, 1000, 100000])
def test_row_counts_and_tall_ctas(N):
    """Many rows per CTA (N = 100000, K = 64: over 512 rows per CTA) exercise
    the bias staging beyond one row per thread."""
    K = 1536 if N < 100000 else 64
    t = _quantized(720 + N, N, K)
    d = to_device(t)
    for batch in (1, 4):
        x = synth.activations(820 + N, batch, K)
        y_ref, s_abs = oracle.gemv(t, N, K, x)
        b = synth.bias(830 + N, N, "bf16")
        y = gpu_gemv_ex(t, N, K, x, oracle.BF16, b, d=d)
        assert_layer_close(y, y_ref, s_abs, oracle.BF16, b, f"N={N} batch={batch}")


def test_zero_k_and_zero_x_give_the_bias():
    """K = 0 (an empty sum) and x = 0 both give y = round(0 + bias) = bias."""
    N, K = 300, 4096
    t = _quantized(840, N, K)
    for name, dt in DTYPES.items():
        b = synth.bias(841, N, name)
        want = np.broadcast_to(b.astype(np.uint32), (2, N))
        y = gpu_gemv_ex(t, N, 0, np.zeros((2, 0), np.uint16), dt, b)
        np.testing.assert_array_equal(y, want)
        y = gpu_gemv_ex(t, N, K, np.zeros((2, K), np.uint16), dt, b)
        np.testing.assert_array_equal(y, want)
        y = gpu_gemv_ex(t, N, 0, np.zeros((1, 0), np.uint16), dt, None)
        assert np.all(y == 0)


def test_f32_without_bias_is_nf4_gemv():
    """nf4_gemv_ex(NULL bias, binary32) writes exactly what nf4_gemv writes."""
    for N, K, batch in ((4096, 4096, 1), (256, 1536, 4), (37, 70, 3)):
        t = _quantized(850 + K, N, K)
        d = to_device(t)
        x = synth.activations(851, batch, K)
        y0 = gpu_gemv(t, N, K, x, d=d)
        y1 = gpu_gemv_ex(t, N, K, x, oracle.F32, None, d=d)
        np.testing.assert_array_equal(y1, y0.view(np.uint32))
        y_ref, s_abs = oracle.gemv(t, N, K, x)
        assert_gemv_close(y0, y_ref, s_abs)



@pytest.mark.parametrize("batch", [9, 16, 33, 64])
def test_wide_batches(batch):
    """Batches above 8 (the tensor-core kernel; one ragged 128-row tile, K
    split over a cluster): every output type, with and without bias."""
    N, K = 37, 1536
    t = _quantized(870 + batch, N, K, 0.001)
    d = to_device(t)
    x = synth.activations(880 + batch, batch, K)
    y_ref, s_abs = oracle.gemv(t, N, K, x)
    for name, dt in DTYPES.items():
        b = synth.bias(890, N, name)
        y = gpu_gemv_ex(t, N, K, x, dt, b, d=d)
        assert_layer_close(y, y_ref, s_abs, dt, b, f"batch={batch} {name} + bias")
    y = gpu_gemv(t, N, K, x, d=d)
    assert_gemv_close(y, y_ref, s_abs, f"batch={batch} fp32")


@pytest.mark.parametrize("N, K, batch, bs", [(300, 4096, 32, 64), (5100, 1024, 24, 64),
                                             (300, 4096, 16, 256), (130, 2048, 48, 128),
                                             (10200, 1024, 16, 64), (10200, 1024, 40, 128)])
def test_tensor_core_tiles_and_cluster_splits(N, K, batch, bs):
    """Batches above 8 on the tensor-core kernel: several 128-row tiles with a
    ragged last tile; K split over clusters of 8 ranks (300 x 4096 on 152 SMs),
    2 ranks (5100 x 1024) and 4 ranks (130 x 2048); clusters of 3 ranks over
    pairs of tiles (10200 x 1024: 80 tiles, the middle rank's stages run from
    one tile into the next); x tiles of 32 and 48 rows; block sizes of 128 and
    256, where one block scale spans several 64-element stages."""
    seed = 900 + N + batch
    t = oracle.quantize(synth.weights(seed, N * K, 0.001, seed + 1), bs, 256, synth.code2_linear())
    d = to_device(t)
    x = synth.activations(seed + 2, batch, K)
    y_ref, s_abs = oracle.gemv(t, N, K, x)
    y = gpu_gemv(t, N, K, x, d=d)
    assert_gemv_close(y, y_ref, s_abs, f"{N}x{K} batch {batch} blocksize {bs}")
    b = synth.bias(seed + 3, N, "bf16")
    y = gpu_gemv_ex(t, N, K, x, oracle.BF16, b, d=d)
    assert_layer_close(y, y_ref, s_abs, oracle.BF16, b, f"{N}x{K} batch {batch} bf16 + bias")


@pytest.mark.parametrize("layer", synth.LLAMA_7B_LAYERS, ids=lambda l: l.name)
def test_llama_layers_batch_64_sampled_rows(layer):
    """Full-size 7B layers at batch 64, checked on 192 sampled rows."""
    t = _quantized(layer.seed, layer.N, layer.K)
    x = synth.activations(synth.llama_x_seed(64), 64, layer.K)
    y = gpu_gemv(t, layer.N, layer.K, x)
    rows = np.sort(np.random.default_rng(layer.seed).choice(layer.N, 192, replace=False))
    rows[0], rows[-1] = 0, layer.N - 1
    y_ref, s_abs = oracle.gemv(t, layer.N, layer.K, x, rows=rows)
    assert_gemv_close(y[:, rows], y_ref, s_abs, f"{layer.name} batch 64")
