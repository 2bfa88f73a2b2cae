"""Helpers for the GPU parity tests: move oracle-quantized tensors to the GPU,
call the library through its binding, compare with the oracle."""
import numpy as np
import torch

import oracle

GUARD = 2048          # sentinel elements after every output buffer
SENTINEL16 = 0x7E5A   # a NaN pattern no kernel writes
SENTINEL32 = np.uint32(0x7FC0DEAD)


def dev():
    return torch.device("cuda:0")


def u16_to_torch(a: np.ndarray, dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).to(dev()).view(dtype)


def to_device(t: oracle.NF4Tensor):
    return dict(packed=torch.from_numpy(t.packed).to(dev()),
                absmax_q=torch.from_numpy(t.absmax_q).to(dev()),
                absmax2=u16_to_torch(t.absmax2, torch.float16),
                code2=u16_to_torch(t.code2, torch.float16))


def gpu_dequant(t: oracle.NF4Tensor, dtype: int, d=None, out_offset: int = 0, packed_offset: int = 0):
    """Run nf4_dequant into a guarded buffer; return the n outputs as uint16 bits."""
    import w4a16_gemv_gb300 as nf4
    d = d or to_device(t)
    tdt = torch.bfloat16 if dtype == oracle.BF16 else torch.float16
    buf = torch.full((out_offset + t.n + GUARD,), SENTINEL16, dtype=torch.int16, device=dev())
    out = buf[out_offset:out_offset + t.n].view(tdt)
    packed = d["packed"]
    if packed_offset:
        pbuf = torch.zeros(packed.numel() + packed_offset, dtype=torch.uint8, device=dev())
        pbuf[packed_offset:] = packed
        packed = pbuf[packed_offset:]
    nf4.nf4_dequant(packed, d["absmax_q"], d["absmax2"], d["code2"], t.offset, t.n, t.blocksize,
                    t.s2_blocksize, out=out, out_dtype=tdt)
    torch.cuda.synchronize()
    host = buf.cpu().numpy().view(np.uint16)
    assert np.all(host[:out_offset] == SENTINEL16), "write before the output"
    assert np.all(host[out_offset + t.n:] == SENTINEL16), "write past the output"
    return host[out_offset:out_offset + t.n]


def gpu_gemv(t: oracle.NF4Tensor, N: int, K: int, x_bits: np.ndarray, d=None, x_offset: int = 0):
    import w4a16_gemv_gb300 as nf4
    d = d or to_device(t)
    batch = x_bits.shape[0]
    xbuf = torch.zeros(x_offset + batch * K, dtype=torch.int16, device=dev())
    if batch * K:
        xbuf[x_offset:] = torch.from_numpy(np.ascontiguousarray(x_bits).reshape(-1).view(np.int16)).to(dev())
    x = xbuf[x_offset:].view(torch.bfloat16).view(batch, K)
    ybuf = torch.from_numpy(np.full(batch * N + GUARD, SENTINEL32, np.uint32).view(np.int32)).to(dev())
    y = ybuf[: batch * N].view(torch.float32).view(batch, N)
    nf4.nf4_gemv(d["packed"], d["absmax_q"], d["absmax2"], d["code2"], t.offset, N, K, x, y=y,
                 blocksize=t.blocksize, s2_blocksize=t.s2_blocksize)
    torch.cuda.synchronize()
    host = ybuf.cpu().numpy().view(np.uint32)
    assert np.all(host[batch * N:] == SENTINEL32), "write past y"
    return host[: batch * N].view(np.float32).reshape(batch, N)


def assert_gemv_close(y, y_ref, s_abs, what=""):
    """|y - y_ref| <= 1e-3 * sum|w_hat x| + 1e-6 on the fp32 result."""
    err = np.abs(y.astype(np.float64) - y_ref)
    bound = 1e-3 * s_abs + 1e-6
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} outputs outside tolerance; worst err/bound "
                           f"{(err / bound).max():.3f}")
    return float((err / bound).max())


_TORCH_Y = {oracle.BF16: "bfloat16", oracle.FP16: "float16", oracle.F32: "float32"}


def gpu_gemv_ex(t: oracle.NF4Tensor, N: int, K: int, x_bits: np.ndarray, dtype: int,
                bias_bits: np.ndarray | None = None, d=None):
    """Run nf4_gemv_ex into a guarded buffer; return y as bit patterns (uint32 [batch, N])."""
    import w4a16_gemv_gb300 as nf4
    d = d or to_device(t)
    tdt = getattr(torch, _TORCH_Y[dtype])
    batch = x_bits.shape[0]
    x = torch.zeros(batch * K, dtype=torch.int16, device=dev())
    if batch * K:
        x[:] = torch.from_numpy(np.ascontiguousarray(x_bits).reshape(-1).view(np.int16)).to(dev())
    x = x.view(torch.bfloat16).view(batch, K)
    wide = dtype == oracle.F32
    store = np.uint32 if wide else np.uint16
    sent = SENTINEL32 if wide else np.uint16(SENTINEL16)
    host = np.full(batch * N + GUARD, sent, store)
    ybuf = torch.from_numpy(host.view(np.int32 if wide else np.int16)).to(dev())
    y = ybuf[: batch * N].view(tdt).view(batch, N)
    b = None
    if bias_bits is not None:
        b = torch.from_numpy(np.ascontiguousarray(bias_bits, store).view(np.int32 if wide else np.int16))
        b = b.to(dev()).view(tdt)
    nf4.nf4_gemv_ex(d["packed"], d["absmax_q"], d["absmax2"], d["code2"], t.offset, N, K, x,
                    bias=b, y=y, out_dtype=tdt, blocksize=t.blocksize, s2_blocksize=t.s2_blocksize)
    torch.cuda.synchronize()
    out = ybuf.cpu().numpy().view(store)
    assert np.all(out[batch * N:] == sent), "write past y"
    return out[: batch * N].astype(np.uint32).reshape(batch, N)


def decode_bits(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact float64 values of bf16 / fp16 / f32 patterns (numpy views)."""
    bits = np.asarray(bits, np.uint32)
    if dtype == oracle.BF16:
        return (bits << 16).view(np.float32).astype(np.float64)
    if dtype == oracle.FP16:
        return bits.astype(np.uint16).view(np.float16).astype(np.float64)
    return bits.view(np.float32).astype(np.float64)


def assert_layer_close(y_bits, y_ref, s_abs, dtype, bias_bits=None, what=""):
    """The fused output stage: y must be the rounding (to dtype) of some value
    within 1e-3 * (sum|w_hat x| + |bias|) + 1e-6 of v = y_ref + bias, i.e.
    round(v - tol) <= y <= round(v + tol) (rounding is monotone)."""
    v, _ = oracle.gemv_output(y_ref, dtype, bias_bits)
    babs = 0.0 if bias_bits is None else np.abs(decode_bits(bias_bits, dtype))[None, :]
    tol = 1e-3 * (s_abs + babs) + 1e-6
    lo = np.vectorize(lambda a: oracle.round_f64(a, dtype), otypes=[np.uint32])(v - tol)
    hi = np.vectorize(lambda a: oracle.round_f64(a, dtype), otypes=[np.uint32])(v + tol)
    y = decode_bits(y_bits, dtype)
    bad = ~((decode_bits(lo, dtype) <= y) & (y <= decode_bits(hi, dtype)))
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outputs outside the rounded "
                           f"tolerance interval; first at {np.argwhere(bad)[0]}")
