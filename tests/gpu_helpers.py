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
