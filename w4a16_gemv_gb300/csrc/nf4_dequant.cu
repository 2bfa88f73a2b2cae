// nf4_dequant.cu -- NF4 double-quant dequantization kernels for sm_103a.
//
// Computes, for every element k (the formula of "NF4 双重量化反量化 CUDA
// Kernel 实现报告", section 1.3, nibble order of section 2.2):
//   s      = fp32(fp32(code2[absmax_q[k >> lbs]] * absmax2[k >> (lbs+ls2)]) + offset)
//   out[k] = RNE16(fp32(NF4[idx(k)] * s))
// bit-exactly, with every multiply and add a separately rounded binary32 op.
//
// Design (GB300, HBM-bound: 0.5 B read + 2 B written per element):
//   * A warp owns a tile of 1024 elements: four 128-byte coalesced loads of
//     packed codes (lane l takes bytes 4l..4l+3 of each 128-byte row) and four
//     512-byte coalesced 16-byte stores, so every store instruction writes
//     whole 32-byte sectors.
//   * The block scale is decoded once per 8 elements (one per store), which
//     covers any power-of-two block size >= 8 with the same code.
//   * The NF4 code book and code2 (widened to binary32) live in shared
//     memory; the 16-entry code book occupies 16 distinct banks, so the
//     per-element lookups never conflict.
//   * Grid-stride loop over tiles, several tiles in flight per warp; the
//     ragged tail (< 1024 elements) is done by one warp with scalar stores.
#include "nf4_internal.cuh"

namespace nf4 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTileElems = 1024;

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kBF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

template <bool kBF16>
__device__ __forceinline__ uint16_t round16(float v) {
  if constexpr (kBF16) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  } else {
    return __half_as_ushort(__float2half_rn(v));
  }
}

// Expand one 32-bit word of packed codes (8 elements) with scale s into four
// 32-bit words of 16-bit outputs (element order preserved: byte i gives the
// elements 2i (high nibble) and 2i+1 (low nibble)).
template <bool kBF16>
__device__ __forceinline__ uint4 expand8(uint32_t w, float s, const float* sT) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t byte = (w >> (8 * i)) & 0xffu;
    const float v_even = __fmul_rn(sT[byte >> 4], s);
    const float v_odd = __fmul_rn(sT[byte & 0xfu], s);
    o[i] = pack2<kBF16>(v_even, v_odd);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ void load_tables(const QuantTensor& t, float* sT, float* sC2) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sC2[i] = half_bits_to_float(t.code2[i]);
  if (threadIdx.x < 16) sT[threadIdx.x] = kCode[threadIdx.x];
  __syncthreads();
}

// Scalar path for elements [first, n): one byte (two elements) per lane step.
template <bool kBF16>
__device__ __forceinline__ void dequant_scalar_range(const QuantTensor& t, const float* sT,
                                                     const float* sC2, int64_t first, int64_t n,
                                                     int64_t start, int64_t step,
                                                     uint16_t* __restrict__ out) {
  const int64_t nbytes = (n + 1) >> 1;
  for (int64_t i = (first >> 1) + start; i < nbytes; i += step) {
    const uint32_t byte = t.packed[i];
    const int64_t e = 2 * i;
    const float s = block_scale(t, sC2, e >> t.lbs);
    out[e] = round16<kBF16>(__fmul_rn(sT[byte >> 4], s));
    if (e + 1 < n) out[e + 1] = round16<kBF16>(__fmul_rn(sT[byte & 0xfu], s));
  }
}

template <bool kBF16, int U>
__global__ void __launch_bounds__(kThreads) dequant_tiles_kernel(QuantTensor t, int64_t n,
                                                                 int64_t ntiles,
                                                                 uint16_t* __restrict__ out) {
  __shared__ float sT[16];
  __shared__ float sC2[256];
  load_tables(t, sT, sC2);

  const int lane = threadIdx.x & 31;
  const int64_t gwarp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = int64_t(gridDim.x) * kWarps;

  for (int64_t tile0 = gwarp * U; tile0 < ntiles; tile0 += nwarps * U) {
    uint32_t w[U][4];
    float s[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t tile = tile0 + u < ntiles ? tile0 + u : ntiles - 1;
      const uint8_t* p = t.packed + tile * (kTileElems / 2) + 4 * lane;
#pragma unroll
      for (int j = 0; j < 4; ++j) w[u][j] = ldg_stream_u32(p + 128 * j);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t tile = tile0 + u < ntiles ? tile0 + u : ntiles - 1;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t e = tile * kTileElems + 256 * j + 8 * lane;
        s[u][j] = block_scale(t, sC2, e >> t.lbs);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t tile = tile0 + u;
      if (tile < ntiles) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t e = tile * kTileElems + 256 * j + 8 * lane;
          const uint4 o = expand8<kBF16>(w[u][j], s[u][j], sT);
          __stcs(reinterpret_cast<uint4*>(out + e), o);
        }
      }
    }
  }
  const int64_t tail = ntiles * kTileElems;
  if (tail < n && gwarp == nwarps - 1)
    dequant_scalar_range<kBF16>(t, sT, sC2, tail, n, lane, 32, out);
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads) dequant_generic_kernel(QuantTensor t, int64_t n,
                                                                   uint16_t* __restrict__ out) {
  __shared__ float sT[16];
  __shared__ float sC2[256];
  load_tables(t, sT, sC2);
  dequant_scalar_range<kBF16>(t, sT, sC2, 0, n, int64_t(blockIdx.x) * blockDim.x + threadIdx.x,
                              int64_t(gridDim.x) * blockDim.x, out);
}

constexpr int kUnroll = 2;

template <bool kBF16>
cudaError_t launch_typed(const QuantTensor& t, int64_t n, uint16_t* out, cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const bool vec_ok = t.lbs >= 3 && (reinterpret_cast<uintptr_t>(t.packed) & 3u) == 0 &&
                      (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  const int64_t max_blocks = int64_t(sms) * (2048 / kThreads);
  if (vec_ok) {
    const int64_t ntiles = n / kTileElems;
    int64_t blocks = (ntiles + int64_t(kWarps) * kUnroll - 1) / (int64_t(kWarps) * kUnroll);
    if (blocks < 1) blocks = 1;
    if (blocks > max_blocks) blocks = max_blocks;
    dequant_tiles_kernel<kBF16, kUnroll>
        <<<dim3(unsigned(blocks)), kThreads, 0, stream>>>(t, n, ntiles, out);
  } else {
    const int64_t nbytes = (n + 1) / 2;
    int64_t blocks = (nbytes + kThreads - 1) / kThreads;
    if (blocks > max_blocks) blocks = max_blocks;
    dequant_generic_kernel<kBF16><<<dim3(unsigned(blocks)), kThreads, 0, stream>>>(t, n, out);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dequant(const QuantTensor& t, int64_t n, void* out, nf4_dtype dtype,
                           cudaStream_t stream) {
  uint16_t* o = static_cast<uint16_t*>(out);
  return dtype == NF4_BF16 ? launch_typed<true>(t, n, o, stream)
                           : launch_typed<false>(t, n, o, stream);
}

}  // namespace nf4
