"""GPU tests of the decode step (nf4_step_create / nf4_step_launch): a
recorded sequence of fused GEMVs, each node's input the step's x or an
earlier node's bf16 output, one kernel per node group.

* Parity: chains and decoder-shaped graphs of layers against the oracle,
  with an error bound carried along every edge (each layer's tolerance plus
  how far its input may be from the oracle's input); every output is checked.
* Mechanism: replays write exactly what the same nodes launched one by one
  write, for new inputs written between replays.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import decode_bits, dev, to_device, u16_to_torch

pytestmark = pytest.mark.gpu

BF16, FP16, F32 = oracle.BF16, oracle.FP16, oracle.F32
_TDT = {BF16: torch.bfloat16, FP16: torch.float16, F32: torch.float32}


def _weight(t: oracle.NF4Tensor, N: int, K: int):
    import w4a16_gemv_gb300 as nf4
    d = to_device(t)
    return nf4.NF4Weight(d["packed"], d["absmax_q"], d["absmax2"], d["code2"], t.offset, t.n,
                         (N, K), t.blocksize, t.s2_blocksize)


def _bits(y: torch.Tensor) -> np.ndarray:
    if y.dtype == torch.float32:
        return y.cpu().numpy().view(np.uint32)
    return y.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32)


def _round_all(v: np.ndarray, dtype: int) -> np.ndarray:
    return np.vectorize(lambda a: oracle.round_f64(a, dtype), otypes=[np.uint32])(v)


def _check_dag(spec, batch, seed, kernels=None, x_edit=None):
    """spec: list of (N, K, y dtype, has_bias, input) nodes. Builds the step
    from oracle-quantized weights, runs it once and checks every node's
    output against the oracle with the carried error bound:
    for a node with oracle input x_or and input bound e (|x_gpu - x_or| <= e),
    v = W x_or + bias, P = sum |w_hat| e, D = 1e-3 (sum |w_hat x_or| + P +
    |bias|) + 1e-6 + P; the GPU output lies in [round(v - D), round(v + D)];
    the node's own output bound is the distance from round(v) to those ends."""
    import w4a16_gemv_gb300 as nf4
    ts, nodes, biases = [], [], []
    for i, (N, K, dt, has_bias, inp) in enumerate(spec):
        t = oracle.quantize(synth.weights(seed + i, N * K), 64, 256, synth.code2_linear())
        ts.append(t)
        name = {BF16: "bf16", FP16: "fp16", F32: "f32"}[dt]
        b = synth.bias(seed + 50 + i, N, name) if has_bias else None
        biases.append(b)
        bt = None
        if b is not None:
            bt = torch.from_numpy(b.view(np.int32 if dt == F32 else np.int16)).to(dev()).view(_TDT[dt])
        y = torch.full((batch, N), float("nan"), dtype=_TDT[dt], device=dev())
        nodes.append(dict(weight=_weight(t, N, K), y=y, bias=bt, input=inp))
    x_bits = synth.activations(seed + 99, batch, spec[0][1])
    if x_edit is not None:
        x_bits = x_edit(x_bits.copy())
    x = u16_to_torch(x_bits, torch.bfloat16).view(batch, -1)
    step = nf4.DecodeStep(nodes, x)
    if kernels is not None:
        assert step.kernel_count() == kernels
    step.launch()
    torch.cuda.synchronize()
    assert nf4.nf4_device_error_flags() == 0

    outs = {}                                  # node -> (oracle output bits, bound)
    for i, (N, K, dt, _, inp) in enumerate(spec):
        if inp == -1:
            x_or, e = x_bits, np.zeros((batch, K))
        else:
            x_or, e = outs[inp]
        y_ref, s_abs = oracle.gemv(ts[i], N, K, x_or)
        p = oracle.gemv_abs(ts[i], N, K, e)
        v, y_or = oracle.gemv_output(y_ref, dt, biases[i])
        babs = 0.0 if biases[i] is None else np.abs(decode_bits(biases[i], dt))[None, :]
        D = 1e-3 * (s_abs + p + babs) + 1e-6 + p
        lo, hi = _round_all(v - D, dt), _round_all(v + D, dt)
        y = decode_bits(_bits(nodes[i]["y"]), dt)
        bad = ~((decode_bits(lo, dt) <= y) & (y <= decode_bits(hi, dt)))
        assert not bad.any(), f"node {i}: {bad.sum()} outputs outside the carried bound"
        c = decode_bits(y_or, dt)
        outs[i] = (y_or.astype(np.uint16), np.maximum(decode_bits(hi, dt) - c, c - decode_bits(lo, dt)))
    step.close()


# q_proj -> o_proj -> gate_proj -> down_proj shapes of a Qwen2.5-1.5B-sized
# decoder layer, each feeding the next (the last in binary32).
CHAIN = [(1536, 1536, BF16, True, -1), (1536, 1536, BF16, False, 0), (8960, 1536, BF16, True, 1),
         (1536, 8960, F32, True, 2)]


@pytest.mark.parametrize("batch", [1, 4, 16])
def test_chain_parity_with_carried_error_bound(batch):
    _check_dag(CHAIN, batch, 200)


def _small_decoder(layers, h=512, kv=128, inter=1536):
    """Decoder-shaped node graph at reduced width: q, k, v from the layer
    input; o from q; gate, up from o; down from gate; next layer from down."""
    spec = []
    for layer in range(layers):
        base = 7 * layer
        inp = -1 if layer == 0 else base - 1
        spec += [(h, h, BF16, True, inp), (kv, h, BF16, True, inp), (kv, h, FP16, True, inp),
                 (h, h, BF16, False, base), (inter, h, BF16, False, base + 3),
                 (inter, h, F32, False, base + 3), (h, inter, BF16, False, base + 4)]
    return spec


@pytest.mark.parametrize("batch", [1, 2, 16])
def test_decoder_graph_parity(batch):
    """Two decoder layers: eight launches (q/k/v and gate/up grouped) up to
    batch 8; one tensor-core launch per node at batch 16."""
    _check_dag(_small_decoder(2), batch, 260, kernels=8 if batch <= 8 else 14)


@pytest.mark.parametrize("batch", [1, 4])
def test_large_group_with_small_arrays_above_the_table(batch):
    """gate/up-sized pair sharing one launch: at batch 4 the per-CTA scales,
    absmax_q and partial sums (145 rows x 64 blocks) no longer fit below the
    pair table and are placed above it; parity against the oracle."""
    spec = [(11008, 4096, BF16, False, -1), (11008, 4096, BF16, False, -1)]
    _check_dag(spec, batch, 330, kernels=1)


@pytest.mark.parametrize("model", ["qwen", "llama"])
def test_full_size_layers_group_qkv_and_gate_up(model):
    """At the Qwen2.5-1.5B and Llama-7B layer shapes (random codes and
    scales; grouping only, no parity), k and v share q's launch and up shares
    gate's: four launches per decoder layer at batch 1 and batch 4."""
    import w4a16_gemv_gb300 as nf4
    h, kv, inter = (1536, 256, 8960) if model == "qwen" else (4096, 4096, 11008)
    g = torch.Generator(device=dev())
    g.manual_seed(31)
    code2 = u16_to_torch(synth.code2_linear(), torch.float16)
    for batch in (1, 4):
        nodes = []
        for layer in range(2):
            base = 7 * layer
            inp = -1 if layer == 0 else base - 1
            for j, (N, K, src) in enumerate([(h, h, inp), (kv, h, inp), (kv, h, inp), (h, h, base),
                                             (inter, h, base + 3), (inter, h, base + 3), (h, inter, base + 4)]):
                n = N * K
                w = nf4.NF4Weight(torch.randint(0, 256, (n // 2,), dtype=torch.uint8, device=dev(), generator=g),
                                  torch.randint(0, 256, (n // 64,), dtype=torch.uint8, device=dev(), generator=g),
                                  (torch.rand((n // 64 + 255) // 256, device=dev(), generator=g) * 0.04 + 0.01).half(),
                                  code2, 0.01, n, (N, K), 64, 256)
                nodes.append(dict(weight=w, y=torch.empty((batch, N), dtype=torch.bfloat16, device=dev()),
                                  bias=None, input=src))
        x = torch.randn((batch, h), device=dev(), generator=g).to(torch.bfloat16)
        step = nf4.DecodeStep(nodes, x)
        assert step.kernel_count() == 8, (model, batch)
        step.launch()
        torch.cuda.synchronize()
        assert nf4.nf4_device_error_flags() == 0
        step.close()


def test_step_with_binary32_x_input():
    """The step's input spans 2^10 .. 2^-30 in its first 32-element chunk (a
    range binary16 cannot hold after any power-of-two scaling), so the first
    launch (q/k/v) runs the batch-1 kernel's binary32-x path inside the
    recorded graph; the values stay inside the binary16 output range of v."""
    def extreme(x):
        x[:, 0] = 0x4480                            # bf16 2^10
        x[:, 1] = 0x3080                            # bf16 2^-30
        return x
    _check_dag(_small_decoder(1), 1, 265, kernels=4, x_edit=extreme)


def test_small_and_fallback_node_groups():
    """Groups with fewer rows than SMs, and a node (K = 40, not a multiple
    of 32) that the streaming kernels do not take (its own launch)."""
    spec = [(64, 256, BF16, True, -1), (7, 256, BF16, False, -1), (256, 64, BF16, True, 0),
            (2, 256, F32, False, 2), (40, 256, BF16, True, 2), (256, 40, FP16, False, 4)]
    _check_dag(spec, 1, 290)
    _check_dag(spec, 3, 291)


def _decoder_nodes(layers, batch, seed):
    """Two decoder layers' linear layers with GPU-quantized weights: q, k, v
    from the layer input; o from q; gate and up from o; down from gate; the
    next layer's input is down's output."""
    import w4a16_gemv_gb300 as nf4
    code2 = u16_to_torch(synth.code2_linear(), torch.float16)
    shapes = [(l.N, l.K) for l in synth.QWEN_1P5B_LAYERS]  # q k v o gate up down
    inputs = [-1, -1, -1, 0, 3, 3, 4]                       # index within the layer
    nodes = []
    for layer in range(layers):
        base = 7 * layer
        for j, (N, K) in enumerate(shapes):
            g = torch.Generator(device="cpu").manual_seed(seed + base + j)
            w = (torch.randn(N * K, generator=g) * 0.02).to(dev())
            wt = nf4.nf4_quantize(w, code2)
            wt.shape = (N, K)
            inp = inputs[j]
            if inp == -1:
                inp = -1 if layer == 0 else base - 1       # previous layer's down_proj
            else:
                inp = base + inp
            bias = None
            if j < 3:                                      # q, k, v carry a bias
                bias = (torch.randn(N, generator=g) * 0.5).bfloat16().to(dev())
            y = torch.empty((batch, N), dtype=torch.bfloat16, device=dev())
            nodes.append(dict(weight=wt, y=y, bias=bias, input=inp))
    return nodes


@pytest.mark.parametrize("batch", [1, 3, 24])
def test_replays_equal_node_by_node_launches(batch):
    import w4a16_gemv_gb300 as nf4
    nodes = _decoder_nodes(2, batch, 300)
    x = torch.empty((batch, 1536), dtype=torch.bfloat16, device=dev())
    step = nf4.DecodeStep(nodes, x)
    ref = [torch.empty_like(nd["y"]) for nd in nodes]
    stream = torch.cuda.Stream()
    for rep in range(3):
        g = torch.Generator(device="cpu").manual_seed(400 + rep)
        x.copy_(torch.randn((batch, 1536), generator=g).bfloat16())
        for nd in nodes:
            nd["y"].fill_(float("nan"))
        with torch.cuda.stream(stream):
            step.launch(stream)
        stream.synchronize()
        for i, nd in enumerate(nodes):
            src = x if nd["input"] == -1 else ref[nd["input"]]
            wt = nd["weight"]
            N, K = wt.shape
            nf4.nf4_gemv_ex(wt.packed, wt.absmax_q, wt.absmax2, wt.code2, wt.offset, N, K, src,
                            bias=nd["bias"], y=ref[i], out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        for i, nd in enumerate(nodes):
            assert torch.equal(nd["y"].view(torch.int16), ref[i].view(torch.int16)), (rep, i)
    step.close()


def test_many_replays_back_to_back_and_empty_nodes():
    """Replays queued without synchronisation run in order (each replay's
    input is written by a copy queued before it), and empty nodes are skipped."""
    import w4a16_gemv_gb300 as nf4
    N, K = 512, 1536
    t = oracle.quantize(synth.weights(500, N * K), 64, 256, synth.code2_linear())
    wt = _weight(t, N, K)
    x = torch.empty((1, K), dtype=torch.bfloat16, device=dev())
    y = torch.empty((1, N), dtype=torch.float32, device=dev())
    empty = nf4.NF4Weight(wt.packed, wt.absmax_q, wt.absmax2, wt.code2, wt.offset, 0, (0, K))
    y0 = torch.empty((1, 0), dtype=torch.bfloat16, device=dev())
    step = nf4.DecodeStep([dict(weight=empty, y=y0), dict(weight=wt, y=y)], x)
    xs = [synth.activations(510 + r, 1, K) for r in range(8)]
    outs = []
    s = torch.cuda.current_stream()
    for r in range(8):
        x.copy_(u16_to_torch(xs[r], torch.bfloat16).view(1, K), non_blocking=True)
        step.launch(s)
        outs.append(y.clone())
    torch.cuda.synchronize()
    for r in range(8):
        y_ref, s_abs = oracle.gemv(t, N, K, xs[r])
        err = np.abs(outs[r].cpu().numpy().astype(np.float64) - y_ref)
        assert np.all(err <= 1e-3 * s_abs + 1e-6), r
    step.close()


@pytest.mark.parametrize("batch", [1, 2, 4, 8])
@pytest.mark.parametrize("Ns", [(1536, 256, 256), (37, 1, 300, 1000, 5), (5, 7), (8960, 8960)])
def test_grouped_nodes_against_the_oracle(Ns, batch):
    """Consecutive nodes reading the same x run as one grouped launch (up to
    four weights; CTAs spread over them by rows); each output is checked
    against the oracle, with mixed output types and biases."""
    import w4a16_gemv_gb300 as nf4
    K = 1536
    x_bits = synth.activations(600 + batch, batch, K)
    x = u16_to_torch(x_bits, torch.bfloat16).view(batch, K)
    kinds = [(BF16, True), (FP16, False), (F32, True), (BF16, False), (FP16, True)]
    ts, nodes, biases = [], [], []
    for j, N in enumerate(Ns):
        dt, has_bias = kinds[j % len(kinds)]
        t = oracle.quantize(synth.weights(610 + j + N, N * K), 64, 256, synth.code2_linear())
        ts.append(t)
        name = {BF16: "bf16", FP16: "fp16", F32: "f32"}[dt]
        b = synth.bias(620 + j, N, name) if has_bias else None
        biases.append(b)
        bt = None
        if b is not None:
            bt = torch.from_numpy(b.view(np.int32 if dt == F32 else np.int16)).to(dev()).view(_TDT[dt])
        y = torch.full((batch, N), float("nan"), dtype=_TDT[dt], device=dev())
        nodes.append(dict(weight=_weight(t, N, K), y=y, bias=bt, input=-1))
    step = nf4.DecodeStep(nodes, x)
    step.launch()
    torch.cuda.synchronize()
    for j, N in enumerate(Ns):
        dt = kinds[j % len(kinds)][0]
        y_ref, s_abs = oracle.gemv(ts[j], N, K, x_bits)
        v, _ = oracle.gemv_output(y_ref, dt, biases[j])
        babs = 0.0 if biases[j] is None else np.abs(decode_bits(biases[j], dt))[None, :]
        tol = 1e-3 * (s_abs + babs) + 1e-6
        lo, hi = _round_all(v - tol, dt), _round_all(v + tol, dt)
        y = decode_bits(_bits(nodes[j]["y"]), dt)
        bad = ~((decode_bits(lo, dt) <= y) & (y <= decode_bits(hi, dt)))
        assert not bad.any(), f"node {j} (N={N}): {bad.sum()} outputs outside tolerance"
    step.close()
