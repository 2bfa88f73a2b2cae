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
//   * Persistent CTAs; each warp walks its tiles with the next tile's loads
//     (packed words and the scale inputs) issued before the current tile is
//     expanded and stored, so reads and writes overlap.
//   * With block size >= 64 one scale is decoded per 64-element segment by
//     one lane and handed to the storing lanes by a shuffle; smaller power-
//     of-two block sizes (>= 8) decode one scale per 8-element run.
//   * The NF4 code book and code2 (widened to binary32) live in shared
//     memory; the 16-entry code book occupies 16 distinct banks (a lane reads
//     one of 16 words, equal words broadcast). Measured on GB300 all the
//     same: 1.18 wavefronts per code lookup on average; the data-dependent
//     code2[absmax_q] reads (one per 64 elements) add 1.44 per decode.
//     Nibbles become byte offsets with two masks and one byte permute each;
//     the two codes of a byte are scaled with one packed binary32 multiply.
//   * The ragged tail (< 1024 elements) is done by one warp with scalar
//     stores.
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

// Kernel prologue: let the next kernel in the stream be scheduled, fill the
// code book (immediates, no memory access), wait for the previous grid, then
// read code2 (the first global memory access).
__device__ __forceinline__ void load_tables(const QuantTensor& t, float* sT, float* sC2) {
  pdl_allow_dependents();
  if (threadIdx.x < 16) sT[threadIdx.x] = nf4_code_select(int(threadIdx.x));
  pdl_wait_prior_grid();
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sC2[i] = half_bits_to_float(t.code2[i]);
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

__device__ __forceinline__ float2 fmul2_rn(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// Expand one 32-bit word of packed codes (8 elements) with scale s into four
// words of 16-bit outputs. The nibbles are turned into byte offsets of the
// binary32 code book in shared memory with two masks, one byte permute per
// code, and the two codes of a byte are scaled by one packed multiply
// (two independent IEEE binary32 products, round to nearest).
template <bool kBF16>
__device__ __forceinline__ uint4 expand8_fast(uint32_t w, float s, const unsigned char* sTb) {
  const uint32_t hi4 = (w >> 2) & 0x3c3c3c3cu;  // 4 * high nibble of every byte (even elements)
  const uint32_t lo4 = (w << 2) & 0x3c3c3c3cu;  // 4 * low nibble (odd elements)
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t ae = __byte_perm(hi4, 0u, 0x4440u | uint32_t(i));
    const uint32_t ao = __byte_perm(lo4, 0u, 0x4440u | uint32_t(i));
    const float2 tv = make_float2(*reinterpret_cast<const float*>(sTb + ae),
                                  *reinterpret_cast<const float*>(sTb + ao));
    const float2 v = fmul2_rn(tv, make_float2(s, s));
    o[i] = pack2<kBF16>(v.x, v.y);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Raw inputs of one group of U tiles, loaded one group ahead of its use.
template <int U, bool kSegScale>
struct DqGroup {
  static constexpr int kSegRegs = kSegScale ? (U * 16 + 31) / 32 : 4 * U;
  uint32_t w[U][4];
  uint32_t q[kSegRegs];   // absmax_q of the block of each scale slot
  uint32_t a2[kSegRegs];  // absmax2 bits of that block's group
};

// Scale slots: with block size >= 64 (kSegScale) every 64-element segment of
// the group has one scale and lane l decodes segments l, l+32, ...; the
// lanes that store a segment fetch its scale with a shuffle. Otherwise each
// lane decodes the scale of each of its own 8-element runs.
template <int U, bool kSegScale>
__device__ __forceinline__ void dq_load(const QuantTensor& t, int64_t tile0, int64_t ntiles, int lane,
                                        DqGroup<U, kSegScale>& g) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t tile = tile0 + u < ntiles ? tile0 + u : ntiles - 1;
    const uint8_t* p = t.packed + tile * (kTileElems / 2) + 4 * lane;
#pragma unroll
    for (int j = 0; j < 4; ++j) g.w[u][j] = ldg_stream_u32(p + 128 * j);
  }
#pragma unroll
  for (int k = 0; k < DqGroup<U, kSegScale>::kSegRegs; ++k) {
    int64_t e;
    if constexpr (kSegScale) {
      const int m = (lane + 32 * k) % (16 * U);
      const int64_t tile = tile0 + m / 16 < ntiles ? tile0 + m / 16 : ntiles - 1;
      e = tile * kTileElems + (m % 16) * 64;
    } else {
      const int u = k / 4, j = k % 4;
      const int64_t tile = tile0 + u < ntiles ? tile0 + u : ntiles - 1;
      e = tile * kTileElems + 256 * j + 8 * lane;
    }
    const int64_t b = e >> t.lbs;
    g.q[k] = __ldg(t.absmax_q + b);
    g.a2[k] = __ldg(t.absmax2 + (b >> t.ls2));
  }
}

template <bool kBF16, int U, bool kSegScale>
__device__ __forceinline__ void dq_store(const QuantTensor& t, int64_t tile0, int64_t ntiles, int lane,
                                         const DqGroup<U, kSegScale>& g, const float* sC2,
                                         const unsigned char* sTb, uint16_t* __restrict__ out) {
  constexpr int R = DqGroup<U, kSegScale>::kSegRegs;
  float sv[R];
#pragma unroll
  for (int k = 0; k < R; ++k)
    sv[k] = __fadd_rn(__fmul_rn(sC2[g.q[k]], half_bits_to_float(uint16_t(g.a2[k]))), t.offset);
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t tile = tile0 + u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float s;
      if constexpr (kSegScale) {
        const int m = u * 16 + 4 * j + (lane >> 3);  // segment of this lane's 8 elements
        s = __shfl_sync(0xffffffffu, sv[(u * 16 + 4 * j) / 32], m % 32);
      } else {
        s = sv[u * 4 + j];
      }
      if (tile < ntiles) {
        const uint4 o = expand8_fast<kBF16>(g.w[u][j], s, sTb);
        __stcs(reinterpret_cast<uint4*>(out + tile * kTileElems + 256 * j + 8 * lane), o);
      }
    }
  }
}

template <bool kBF16, int U, bool kSegScale>
__global__ void __launch_bounds__(kThreads) dequant_tiles_kernel(QuantTensor t, int64_t n,
                                                                 int64_t ntiles,
                                                                 uint16_t* __restrict__ out) {
  __shared__ float sT[16];
  __shared__ float sC2[256];
  load_tables(t, sT, sC2);
  const unsigned char* sTb = reinterpret_cast<const unsigned char*>(sT);

  const int lane = threadIdx.x & 31;
  const int64_t gwarp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = int64_t(gridDim.x) * kWarps;
  const int64_t stride = nwarps * U;

  int64_t tile0 = gwarp * U;
  DqGroup<U, kSegScale> cur;
  if (tile0 < ntiles) dq_load<U, kSegScale>(t, tile0, ntiles, lane, cur);
  while (tile0 < ntiles) {
    const int64_t next = tile0 + stride;
    DqGroup<U, kSegScale> nxt;
    if (next < ntiles) dq_load<U, kSegScale>(t, next, ntiles, lane, nxt);
    dq_store<kBF16, U, kSegScale>(t, tile0, ntiles, lane, cur, sC2, sTb, out);
    cur = nxt;
    tile0 = next;
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

#ifndef NF4_DQ_BLOCKS_PER_SM
#define NF4_DQ_BLOCKS_PER_SM 4
#endif
#ifndef NF4_DQ_PDL
#define NF4_DQ_PDL 0
#endif
constexpr int kBlocksPerSm = NF4_DQ_BLOCKS_PER_SM;  // persistent CTAs per SM

template <bool kBF16, int U>
cudaError_t launch_tiles(const QuantTensor& t, int64_t n, int64_t ntiles, uint16_t* out, int sms,
                         cudaStream_t stream) {
  int64_t blocks = (ntiles + int64_t(kWarps) * U - 1) / (int64_t(kWarps) * U);
  if (blocks < 1) blocks = 1;
  if (blocks > int64_t(sms) * kBlocksPerSm) blocks = int64_t(sms) * kBlocksPerSm;
  if (t.lbs >= 6)
    return launch_k_pdl(NF4_DQ_PDL, dequant_tiles_kernel<kBF16, U, true>, dim3(unsigned(blocks)),
                        dim3(kThreads), 0, stream, t, n, ntiles, out);
  return launch_k_pdl(NF4_DQ_PDL, dequant_tiles_kernel<kBF16, U, false>, dim3(unsigned(blocks)),
                      dim3(kThreads), 0, stream, t, n, ntiles, out);
}

template <bool kBF16>
cudaError_t launch_typed(const QuantTensor& t, int64_t n, uint16_t* out, cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const bool vec_ok = t.lbs >= 3 && (reinterpret_cast<uintptr_t>(t.packed) & 3u) == 0 &&
                      (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  if (vec_ok) {
    // Tiles per warp step by size (measured on GB300): one when the tensor
    // gives the warps under two tiles each (1024^2: 3.0 -> 2.7 us), four from
    // 32 tiles per warp (28672x8192: 101 -> 94 us), two in between.
    const int64_t ntiles = n / kTileElems;
    const int64_t warps = int64_t(sms) * kBlocksPerSm * kWarps;
    if (ntiles < 2 * warps) return launch_tiles<kBF16, 1>(t, n, ntiles, out, sms, stream);
    if (ntiles >= 32 * warps) return launch_tiles<kBF16, 4>(t, n, ntiles, out, sms, stream);
    return launch_tiles<kBF16, 2>(t, n, ntiles, out, sms, stream);
  } else {
    const int64_t nbytes = (n + 1) / 2;
    int64_t blocks = (nbytes + kThreads - 1) / kThreads;
    const int64_t max_blocks = int64_t(sms) * (2048 / kThreads);
    if (blocks > max_blocks) blocks = max_blocks;
    return launch_k(dequant_generic_kernel<kBF16>, dim3(unsigned(blocks)), dim3(kThreads), 0,
                    stream, t, n, out);
  }
}

}  // namespace

cudaError_t launch_dequant(const QuantTensor& t, int64_t n, void* out, nf4_dtype dtype,
                           cudaStream_t stream) {
  uint16_t* o = static_cast<uint16_t*>(out);
  return dtype == NF4_BF16 ? launch_typed<true>(t, n, o, stream)
                           : launch_typed<false>(t, n, o, stream);
}

}  // namespace nf4
