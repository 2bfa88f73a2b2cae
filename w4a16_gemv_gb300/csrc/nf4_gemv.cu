// nf4_gemv.cu -- decode GEMV y = W_hat x with NF4 double-quant dequantization
// fused, for sm_103a.
//
// The fused form follows "RTX 4060 上的 LLM 量化实测：4-bit decode 比 FP16 慢在
// 哪里", section "Fused kernel：把反量化搬到片上": packed codes are read once,
// decoded, scaled and accumulated on chip in binary32; only y is written. The
// work split follows "CUDA 进阶手册 / 量化与 GEMV", section "GEMV kernel 的写法":
// warps own rows, lanes walk K with 16-byte loads, a shuffle reduction ends
// each row, and a warp handles several rows at once so every lane has many
// loads in flight.
//
// GB300 design (HBM-bound at batch 1: ~0.52 B per weight):
//   * Code lookup without the constant cache and without bank conflicts: a
//     256-entry table maps a packed BYTE to both of its codes as a binary16
//     pair, replicated once per lane so that lane l always reads bank l
//     (256 x 32 x 4 B = 32 KB of shared memory per CTA). One shared load
//     yields two weights; two conversions and one packed fma.rn.f32x2
//     accumulate them against two activations.
//   * The NF4 codes are held as binary16 in that table (relative rounding
//     error <= 2^-11, inside the GEMV tolerance); the per-block scale is
//     applied once per chunk in binary32 (acc += s * sum_chunk(code * x)).
//   * x is read through the read-only path and widened to binary32 in
//     registers; each x chunk is reused for R rows.
//   * For thin layers several warps split K (ks > 1) and combine through
//     shared memory, so that small N still spreads over all SMs.
#include "nf4_internal.cuh"

namespace nf4 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// 32-bit shared-window loads.
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds_u128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds_u64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Two bfloat16 (low half = lower-index element) widened to binary32 (exact).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t h) {
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

template <int CB>
struct Chunk;
template <>
struct Chunk<16> {
  uint32_t w[4];
  __device__ __forceinline__ void load(const uint8_t* p) {
    const uint4 v = ldg_stream_u128(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  }
};
template <>
struct Chunk<8> {
  uint32_t w[2];
  __device__ __forceinline__ void load(const uint8_t* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    w[0] = v.x; w[1] = v.y;
  }
};
template <>
struct Chunk<4> {
  uint32_t w[1];
  __device__ __forceinline__ void load(const uint8_t* p) { w[0] = ldg_stream_u32(p); }
};

// Byte -> (binary16 code of the high nibble, binary16 code of the low nibble),
// one copy per lane: word [e * 32 + lane]. The codes are selected per lane
// from immediates and exchanged by shuffles (no memory access).
__device__ __forceinline__ void build_pair_table(uint32_t* sTab) {
  const uint32_t my_code16 =
      __half_as_ushort(__float2half_rn(nf4_code_select(int(threadIdx.x & 15))));
  for (int i = threadIdx.x; i < 256 * 8; i += blockDim.x) {
    const int e = i >> 3, q = i & 7;
    const uint32_t hi = __shfl_sync(0xffffffffu, my_code16, e >> 4);
    const uint32_t lo = __shfl_sync(0xffffffffu, my_code16, e & 15);
    const uint32_t v = hi | (lo << 16);
    *reinterpret_cast<uint4*>(sTab + e * 32 + q * 4) = make_uint4(v, v, v, v);
  }
}

// B activation vectors, CB packed bytes per lane per row per step (2*CB
// elements, inside one quantization block), R rows per warp, ks warps per
// row tile splitting K.
template <int B, int CB, int R>
__global__ void __launch_bounds__(kThreads) gemv_fast_kernel(QuantTensor t, int64_t N, int64_t K,
                                                             int ks, const uint16_t* __restrict__ x,
                                                             float* __restrict__ y) {
  extern __shared__ __align__(16) uint32_t sTab[];
  __shared__ float sC2[256];
  __shared__ float sRed[kWarps][R * B];
  pdl_allow_dependents();
  build_pair_table(sTab);
  pdl_wait_prior_grid();
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sC2[i] = half_bits_to_float(t.code2[i]);
  __syncthreads();

  constexpr int CE = 2 * CB;  // elements per chunk
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int rt = warp / ks;
  const int kslice = warp - rt * ks;
  const int64_t row0 = (int64_t(blockIdx.x) * (kWarps / ks) + rt) * R;
  const int64_t cpr = K / CE;
  const int64_t row_bytes = K >> 1;

  int64_t rows[R];
#pragma unroll
  for (int r = 0; r < R; ++r) rows[r] = (row0 + r < N) ? row0 + r : N - 1;

  float acc[R][B];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int b = 0; b < B; ++b) acc[r][b] = 0.0f;

  const uint32_t* tab = sTab + lane;
  for (int64_t c = int64_t(kslice) * 32 + lane; c < cpr; c += 32 * ks) {
    Chunk<CB> wc[R];
    float s[R];
#pragma unroll
    for (int r = 0; r < R; ++r) wc[r].load(t.packed + rows[r] * row_bytes + c * CB);
#pragma unroll
    for (int r = 0; r < R; ++r) s[r] = block_scale(t, sC2, (rows[r] * K + c * CE) >> t.lbs);

    float2 xf[B][CB];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const uint4* xp = reinterpret_cast<const uint4*>(x + int64_t(b) * K + c * CE);
#pragma unroll
      for (int q = 0; q < CB / 4; ++q) {
        const uint4 v = __ldg(xp + q);
        xf[b][4 * q + 0] = bf16x2_to_float2(v.x);
        xf[b][4 * q + 1] = bf16x2_to_float2(v.y);
        xf[b][4 * q + 2] = bf16x2_to_float2(v.z);
        xf[b][4 * q + 3] = bf16x2_to_float2(v.w);
      }
    }

#pragma unroll
    for (int r = 0; r < R; ++r) {
      float2 pa[B];
#pragma unroll
      for (int b = 0; b < B; ++b) pa[b] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int wi = 0; wi < CB / 4; ++wi) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t byte = (wc[r].w[wi] >> (8 * i)) & 0xffu;
          const float2 tw = half2_bits_to_float2(tab[byte * 32]);
#pragma unroll
          for (int b = 0; b < B; ++b) pa[b] = ffma2(tw, xf[b][4 * wi + i], pa[b]);
        }
      }
#pragma unroll
      for (int b = 0; b < B; ++b) acc[r][b] = fmaf(s[r], pa[b].x + pa[b].y, acc[r][b]);
    }
  }

#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int b = 0; b < B; ++b) acc[r][b] = warp_sum(acc[r][b]);

  if (ks == 1) {
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (row0 + r < N)
#pragma unroll
          for (int b = 0; b < B; ++b) y[int64_t(b) * N + row0 + r] = acc[r][b];
    }
  } else {
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b) sRed[warp][r * B + b] = acc[r][b];
    }
    __syncthreads();
    if (kslice == 0 && lane < R * B) {
      float v = 0.0f;
      for (int j = 0; j < ks; ++j) v += sRed[warp + j][lane];
      const int r = lane / B, b = lane - (lane / B) * B;
      if (row0 + r < N) y[int64_t(b) * N + row0 + r] = v;
    }
  }
}

// Any even K, any power-of-two block size, any element alignment: one warp
// per row, one packed byte per lane step.
template <int B>
__global__ void __launch_bounds__(kThreads) gemv_generic_kernel(QuantTensor t, int64_t N,
                                                                int64_t K,
                                                                const uint16_t* __restrict__ x,
                                                                float* __restrict__ y) {
  __shared__ float sT[16];
  __shared__ float sC2[256];
  pdl_allow_dependents();
  if (threadIdx.x < 16) sT[threadIdx.x] = nf4_code_select(int(threadIdx.x));
  pdl_wait_prior_grid();
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sC2[i] = half_bits_to_float(t.code2[i]);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = int64_t(gridDim.x) * kWarps;
  const int64_t half_k = K >> 1;
  for (int64_t row = gwarp; row < N; row += nwarps) {
    float acc[B];
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b] = 0.0f;
    for (int64_t j = lane; j < half_k; j += 32) {
      const int64_t flat = row * K + 2 * j;
      const uint32_t byte = t.packed[flat >> 1];
      const float s = block_scale(t, sC2, flat >> t.lbs);
      const float w0 = __fmul_rn(sT[byte >> 4], s);
      const float w1 = __fmul_rn(sT[byte & 0xfu], s);
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const float x0 = __uint_as_float(uint32_t(x[int64_t(b) * K + 2 * j]) << 16);
        const float x1 = __uint_as_float(uint32_t(x[int64_t(b) * K + 2 * j + 1]) << 16);
        acc[b] = fmaf(w0, x0, fmaf(w1, x1, acc[b]));
      }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const float v = warp_sum(acc[b]);
      if (lane == 0) y[int64_t(b) * N + row] = v;
    }
  }
}

// Sum V values over the 32 lanes of a warp. On return lane l holds the total
// of value index transposed_index<V>(l); lanes l < V cover every index once.
template <int V>
__device__ __forceinline__ float transposed_warp_reduce(float (&v)[V], int lane) {
#pragma unroll
  for (int step = 0; (1 << step) < V; ++step) {
    const int cnt = V >> step;
    const int m = 1 << step;
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const float send = upper ? v[i] : v[i + cnt / 2];
      const float keep = upper ? v[i + cnt / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  float r = v[0];
#pragma unroll
  for (int m = V; m < 32; m <<= 1) r += __shfl_xor_sync(0xffffffffu, r, m);
  return r;
}

template <int V>
__device__ __forceinline__ int transposed_index(int lane) {
  int r = 0;
#pragma unroll
  for (int step = 0; (1 << step) < V; ++step)
    if (lane & (1 << step)) r += V >> (step + 1);
  return r;
}

__device__ unsigned int g_device_flags = 0;

constexpr uint32_t kPairTableBytes = 256u * 64u * 4u;

// ---------------------------------------------------------------------------
// Batch-1 streaming GEMV. Every thread owns one column chunk of CB packed
// bytes (CE = 2*CB elements) of every row and keeps the matching slice of x
// in registers for the whole kernel. A CTA owns a contiguous range of rows;
// one thread streams them through a ring of shared-memory stages with bulk
// asynchronous copies (cp.async.bulk completing on mbarriers), every stage
// that fits issued up front, together with the absmax_q bytes of the range.
// `groups` copies of the thread layout process different rows of a stage;
// a stage ends with one CTA barrier and a two-level reduction (transposed
// warp butterfly, then across the warps of a row group).
//
// Inner loop (per packed byte, i.e. two weights): one byte permute forms the
// shared address of the byte's entry in a lane-private table of binary16
// code pairs (the table sits at a 64 KB-aligned shared address, so the
// permute supplies every address bit); one 32-bit shared load; two
// mixed-precision fma.rn.f32.f16 (binary16 x binary16 -> binary32
// accumulate, product exact). x is held as binary16 after an exact
// power-of-two scaling chosen per thread; a CTA whose x slice does not
// convert exactly (extreme dynamic range, NaN/Inf) or whose table is not
// 64 KB-aligned runs the same loop on binary32 x with conversions and packed
// fma.rn.f32x2 instead. The NF4 codes carry a binary16 rounding error of at
// most 3.3e-4 relative, inside the GEMV tolerance.
constexpr int kMaxSlots = 16;
#ifndef NF4_STREAM_DEPTH
#define NF4_STREAM_DEPTH 2
#endif

struct StreamPlan {
  int64_t rows_per_cta;
  int tk;           // threads per row group; thread c owns column chunk c (c < cpr)
  int groups;       // row groups per CTA
  int stage_rows;   // groups * RPG
  int nslots;       // ring slots
  int depth;        // stages in flight ahead of the first unlanded one
  uint32_t stage_bytes;
  int spr;          // quantization blocks per row (K / blocksize)
  int ng_cap;       // absmax2 entries held per CTA
  uint32_t q_cap;   // absmax_q bytes held per CTA
  uint32_t off_red, off_c2, off_a2, off_bar, off_q, off_scale, off_part, off_tab;
  uint32_t off_slot[kMaxSlots];
  uint32_t smem_bytes;
};

__device__ __forceinline__ void mbar_arrive_plain(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// acc_a += T(lo half) * x0, acc_b += T(hi half) * x1, binary16 inputs, binary32 accumulate.
__device__ __forceinline__ void fma2_f16_f32(uint32_t tpair, unsigned short x0, unsigned short x1,
                                             float& acc_a, float& acc_b) {
  asm("{\n\t.reg .f16 t0, t1;\n\t"
      "mov.b32 {t0, t1}, %2;\n\t"
      "fma.rn.f32.f16 %0, t0, %3, %0;\n\t"
      "fma.rn.f32.f16 %1, t1, %4, %1;\n\t}"
      : "+f"(acc_a), "+f"(acc_b)
      : "r"(tpair), "h"(x0), "h"(x1));
}

// Consumer warps: wait for a stage, compute the dot products of this warp's
// rows, release the slot (one arrival per warp on the slot's "empty"
// barrier), reduce across the warp and store the warp's partial sums in its
// own slot of sPart[row][warp] (deterministic order, no atomics).
template <int CB, int RPG, bool kFast>
__device__ __forceinline__ bool stream_consume(
    const QuantTensor& t, int64_t K, const StreamPlan& p, unsigned char* smem, int64_t row_begin,
    int64_t row_end, int nstages, const uint4 (&xv)[CB / 4], float xscale,
    const unsigned short (&x16)[2 * CB]) {
  constexpr int CE = 2 * CB;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int g = tid / p.tk;
  const int c = tid - g * p.tk;
  const int wig = c >> 5;
  const int wpg = p.tk >> 5;
  const int64_t cpr = K / CE;
  const int cc = (c < cpr) ? c : int(cpr - 1);
  const int64_t row_bytes = K >> 1;
  const float* sScale = reinterpret_cast<const float*>(smem + p.off_scale);
  float* sPart = reinterpret_cast<float*>(smem + p.off_part);
  uint64_t* sFull = reinterpret_cast<uint64_t*>(smem + p.off_bar) + 1;
  uint64_t* sEmpty = sFull + kMaxSlots;
  const uint32_t smem_s = smem_u32(smem);
  const uint32_t tab_s = smem_s + p.off_tab;
  const uint32_t lanebase = (tab_s & 0xffff0000u) | (uint32_t(lane) << 2);
  const uint32_t lane4 = uint32_t(lane) << 2;
  const int scol = int((int64_t(cc) * CE) >> t.lbs);

  float2 xf[CB];
  if constexpr (!kFast) {
#pragma unroll
    for (int q = 0; q < CB / 4; ++q) {
      xf[4 * q + 0] = bf16x2_to_float2(xv[q].x);
      xf[4 * q + 1] = bf16x2_to_float2(xv[q].y);
      xf[4 * q + 2] = bf16x2_to_float2(xv[q].z);
      xf[4 * q + 3] = bf16x2_to_float2(xv[q].w);
    }
  }

  bool ok_all = true;
  for (int s = 0; s < nstages; ++s) {
    const int slot = s % p.nslots;
    const bool ok = mbar_wait_bounded(&sFull[slot], uint32_t((s / p.nslots) & 1), kWaitLimitCycles);
    ok_all = ok_all && ok;
    const uint32_t st_s = smem_s + p.off_slot[slot];
    const int rbase = s * p.stage_rows + g * RPG;  // first row of this group, relative to row_begin
    float part[RPG];
#pragma unroll
    for (int r = 0; r < RPG; ++r) {
      const int rl = g * RPG + r;
      const bool rv = row_begin + rbase + r < row_end;
      const int rlc = rv ? rl : 0;  // stage row 0 always holds data
      const uint32_t wp = st_s + uint32_t(rlc) * uint32_t(row_bytes) + uint32_t(cc) * CB;
      uint32_t w[CB / 4];
      if constexpr (CB == 16) {
        const uint4 v = lds_u128(wp);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
      } else {
        const uint2 v = lds_u64(wp);
        w[0] = v.x; w[1] = v.y;
      }
      const float sc = sScale[uint32_t(s * p.stage_rows + rlc) * uint32_t(p.spr) + uint32_t(scol)];
      float sum;
      if constexpr (kFast) {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int wi = 0; wi < CB / 4; ++wi) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t addr = __byte_perm(w[wi], lanebase, 0x7604u | (uint32_t(i) << 4));
            const uint32_t h = lds_u32(addr);
            const int k = 4 * wi + i;
            if (i & 1) fma2_f16_f32(h, x16[2 * k], x16[2 * k + 1], a2, a3);
            else fma2_f16_f32(h, x16[2 * k], x16[2 * k + 1], a0, a1);
          }
        }
        sum = (a0 + a1) + (a2 + a3);
      } else {
        float2 pa = make_float2(0.f, 0.f), pb = make_float2(0.f, 0.f);
#pragma unroll
        for (int wi = 0; wi < CB / 4; ++wi) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t addr = tab_s + __byte_perm(w[wi], lane4, 0x5504u | (uint32_t(i) << 4));
            const float2 tw = half2_bits_to_float2(lds_u32(addr));
            if (i & 1) pb = ffma2(tw, xf[4 * wi + i], pb);
            else pa = ffma2(tw, xf[4 * wi + i], pa);
          }
        }
        sum = (pa.x + pa.y) + (pb.x + pb.y);
      }
      part[r] = __fmul_rn(sc, xscale) * sum;
    }
    // this warp is done reading the slot
    __syncwarp();
    if (lane == 0) mbar_arrive_plain(&sEmpty[slot]);
    const float red = transposed_warp_reduce<RPG>(part, lane);
    if (lane < RPG) {
      const int rr = rbase + transposed_index<RPG>(lane);
      if (row_begin + rr < row_end) sPart[rr * wpg + wig] = red;
    }
  }
  return ok_all;
}

// Producer (one lane of the extra warp). Stage s is issued once stage
// s - depth has landed (so only `depth` stages per CTA are in flight and the
// earliest stage is not delayed behind the whole slab) and once every
// consumer warp has released the slot's previous stage.
__device__ __forceinline__ bool stream_produce(const QuantTensor& t, int64_t K,
                                               const StreamPlan& p, unsigned char* smem,
                                               int64_t row_begin, int64_t row_end, int nstages,
                                               int issued) {
  const int64_t row_bytes = K >> 1;
  uint64_t* sFull = reinterpret_cast<uint64_t*>(smem + p.off_bar) + 1;
  uint64_t* sEmpty = sFull + kMaxSlots;
  bool ok = true;
  for (int s = issued; s < nstages; ++s) {
    const int slot = s % p.nslots;
    const int sl = s - p.depth;
    if (sl >= 0)
      ok = ok && mbar_wait_bounded(&sFull[sl % p.nslots], uint32_t((sl / p.nslots) & 1), kWaitLimitCycles);
    if (s >= p.nslots)
      ok = ok && mbar_wait_bounded(&sEmpty[slot], uint32_t(((s / p.nslots) - 1) & 1), kWaitLimitCycles);
    if (!ok) break;
    fence_proxy_async_smem();
    const int64_t r0 = row_begin + int64_t(s) * p.stage_rows;
    const int64_t rows = (r0 + p.stage_rows < row_end) ? p.stage_rows : row_end - r0;
    const uint32_t bytes = uint32_t(rows * row_bytes);
    mbar_arrive_expect_tx(&sFull[slot], bytes);
    bulk_copy_g2s(smem + p.off_slot[slot], t.packed + r0 * row_bytes, bytes, &sFull[slot]);
  }
  return ok;
}

template <int CB, int RPG>
__global__ void __launch_bounds__(544, 1) gemv_b1_stream_kernel(QuantTensor t, int64_t N, int64_t K,
                                                                 const uint16_t* __restrict__ x,
                                                                 float* __restrict__ y, StreamPlan p) {
  constexpr int CE = 2 * CB;
  extern __shared__ __align__(128) unsigned char smem[];
  float* sC2 = reinterpret_cast<float*>(smem + p.off_c2);
  float* sA2 = reinterpret_cast<float*>(smem + p.off_a2);
  uint64_t* sBar = reinterpret_cast<uint64_t*>(smem + p.off_bar);  // [0] absmax_q, then full[], empty[]
  uint64_t* sFull = sBar + 1;
  uint64_t* sEmpty = sFull + kMaxSlots;
  unsigned char* sQ = smem + p.off_q;
  float* sScale = reinterpret_cast<float*>(smem + p.off_scale);
  const float* sPart = reinterpret_cast<const float*>(smem + p.off_part);
  uint32_t* sTab = reinterpret_cast<uint32_t*>(smem + p.off_tab);

  const int tid = threadIdx.x;
  const int nconsumer = p.tk * p.groups;  // the last warp is the producer
  const bool consumer = tid < nconsumer;
  const int64_t row_bytes = K >> 1;
  const int64_t row_begin = int64_t(blockIdx.x) * p.rows_per_cta;
  const int64_t row_end = (row_begin + p.rows_per_cta < N) ? row_begin + p.rows_per_cta : N;
  const int nstages = int((row_end - row_begin + p.stage_rows - 1) / p.stage_rows);
  const int issued0 = nstages < p.depth ? nstages : p.depth;
  const int64_t b0 = (row_begin * K) >> t.lbs;
  const int64_t nq = (row_end - row_begin) * p.spr;
  const int64_t g0 = b0 >> t.ls2;
  const int ng = int(((b0 + nq - 1) >> t.ls2) - g0 + 1);
  const bool q_bulk = (reinterpret_cast<uintptr_t>(t.absmax_q) & 15u) == 0;
  const int64_t q_main = q_bulk ? (nq & ~int64_t(15)) : 0;  // bytes brought by the bulk copy
  const int g = tid / p.tk;
  const int c = tid - g * p.tk;
  const int64_t cpr = K / CE;
  const int cc = (c < cpr) ? c : int(cpr - 1);

  // Prologue. Nothing before the grid-dependency wait touches global memory:
  // barriers and the pair table (codes selected from immediates, exchanged
  // by shuffles) are built first.
  pdl_allow_dependents();
  if (tid == 0) {
    mbar_init(&sBar[0], 1);
    for (int s = 0; s < p.nslots; ++s) {
      mbar_init(&sFull[s], 1);
      mbar_init(&sEmpty[s], uint32_t(nconsumer / 32));
    }
    fence_mbar_init();
  }
  {
    const uint32_t my_code16 =
        __half_as_ushort(__float2half_rn(nf4_code_select(int(threadIdx.x & 15))));
    for (int i = tid; i < 256 * 8; i += blockDim.x) {
      const int e = i >> 3, q = i & 7;
      const uint32_t hi = __shfl_sync(0xffffffffu, my_code16, e >> 4);
      const uint32_t lo = __shfl_sync(0xffffffffu, my_code16, e & 15);
      const uint32_t v = hi | (lo << 16);
      *reinterpret_cast<uint4*>(sTab + e * 64 + q * 4) = make_uint4(v, v, v, v);
    }
  }
  pdl_wait_prior_grid();

  // The small loads go out before the bulk weight stream.
  uint4 xv[CB / 4];
#pragma unroll
  for (int q = 0; q < CB / 4; ++q)
    xv[q] = (consumer && c < cpr)
                ? __ldg(reinterpret_cast<const uint4*>(x + int64_t(cc) * CE) + q)
                : make_uint4(0u, 0u, 0u, 0u);
  const uint16_t c2v = (tid < 256) ? __ldg(t.code2 + tid) : uint16_t(0);
  const uint16_t a2v = (tid < ng) ? __ldg(t.absmax2 + g0 + tid) : uint16_t(0);
  for (int64_t i = q_main + tid; i < nq; i += blockDim.x) sQ[i] = __ldg(t.absmax_q + b0 + i);
  __syncthreads();
  if (tid == 0) {
    // absmax_q first, then the first `depth` stages.
    if (q_main > 0) {
      mbar_arrive_expect_tx(&sBar[0], uint32_t(q_main));
      bulk_copy_g2s(sQ, t.absmax_q + b0, uint32_t(q_main), &sBar[0]);
    } else {
      mbar_arrive_plain(&sBar[0]);
    }
    for (int s = 0; s < issued0; ++s) {
      const int64_t r0 = row_begin + int64_t(s) * p.stage_rows;
      const int64_t rows = (r0 + p.stage_rows < row_end) ? p.stage_rows : row_end - r0;
      const uint32_t bytes = uint32_t(rows * row_bytes);
      mbar_arrive_expect_tx(&sFull[s], bytes);
      bulk_copy_g2s(smem + p.off_slot[s], t.packed + r0 * row_bytes, bytes, &sFull[s]);
    }
  }
  if (tid < 256) sC2[tid] = half_bits_to_float(c2v);
  if (tid < ng) sA2[tid] = half_bits_to_float(a2v);

  // x slice: exact binary16 after a power-of-two scaling, else the binary32
  // path. The scale 2^-e brings the largest |x| into [2^14, 2^15); scaling
  // by a power of two is exact in binary32, and a value that binary16 cannot
  // hold exactly fails the round-trip comparison.
  float m = 0.0f;
#pragma unroll
  for (int q = 0; q < CB / 4; ++q) {
    const uint32_t wv[4] = {xv[q].x, xv[q].y, xv[q].z, xv[q].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = bf16x2_to_float2(wv[j]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  const int em = int((__float_as_uint(m) >> 23) & 0xffu) - 127;
  const int e = (m > 0.0f && m <= 3.0e38f && em > -100) ? em - 14 : 0;
  const float down = __uint_as_float(uint32_t(127 - e) << 23);  // 2^-e, e in [-113, 113]
  bool x_exact = !(m != m);  // a NaN takes the binary32 path
  unsigned short x16[2 * CB];
#pragma unroll
  for (int q = 0; q < CB / 4; ++q) {
    const uint32_t wv[4] = {xv[q].x, xv[q].y, xv[q].z, xv[q].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = bf16x2_to_float2(wv[j]);
      const float s0 = __fmul_rn(f.x, down), s1 = __fmul_rn(f.y, down);
      const __half h0 = __float2half_rn(s0), h1 = __float2half_rn(s1);
      x_exact = x_exact && (__half2float(h0) == s0) && (__half2float(h1) == s1);
      x16[2 * (4 * q + j)] = __half_as_ushort(h0);
      x16[2 * (4 * q + j) + 1] = __half_as_ushort(h1);
    }
  }
  const bool aligned = (smem_u32(sTab) & 0xffffu) == 0u;
  const bool fast = !__syncthreads_or(!(x_exact && aligned));
  const bool q_ok = mbar_wait_bounded(&sBar[0], 0u, kWaitLimitCycles);
  // One decoded scale per block of this CTA's rows (32-bit indices: b0 is
  // only needed modulo the group size).
  if (q_ok) {
    const uint32_t b0_in_group = uint32_t(b0 & ((int64_t(1) << t.ls2) - 1));
    for (int i = tid; i < int(nq); i += blockDim.x)
      sScale[i] = __fadd_rn(__fmul_rn(sC2[sQ[i]], sA2[(b0_in_group + uint32_t(i)) >> t.ls2]), t.offset);
  }
  bool ok = !__syncthreads_or(!q_ok);
  if (ok) {
    if (consumer) {
      ok = fast ? stream_consume<CB, RPG, true>(t, K, p, smem, row_begin, row_end, nstages, xv,
                                                __uint_as_float(uint32_t(127 + e) << 23), x16)
                : stream_consume<CB, RPG, false>(t, K, p, smem, row_begin, row_end, nstages, xv,
                                                 1.0f, x16);
    } else if (tid == nconsumer) {
      ok = stream_produce(t, K, p, smem, row_begin, row_end, nstages, issued0);
    }
  }
  if (!__syncthreads_or(!ok)) {
    // every row's partial sums are in place: one sum per row, warps in order
    const int wpg = p.tk >> 5;
    for (int64_t r = tid; r < row_end - row_begin; r += blockDim.x) {
      float sum = 0.0f;
      for (int w = 0; w < wpg; ++w) sum += sPart[r * wpg + w];
      y[row_begin + r] = sum;
    }
  } else {
    // A copy did not complete within the limit: report it, mark this CTA's
    // outputs as invalid, wait (bounded) for the copies that may be in flight.
    if (tid == 0) atomicOr(&g_device_flags, 1u);
    for (int64_t i = row_begin + tid; i < row_end; i += blockDim.x) y[i] = __int_as_float(0x7fc00000);
    if (tid == 0) {
      (void)mbar_wait_bounded(&sBar[0], 0u, kWaitLimitCycles / 8);
      for (int s2 = nstages - p.nslots; s2 < nstages; ++s2)
        if (s2 >= 0)
          (void)mbar_wait_bounded(&sFull[s2 % p.nslots], uint32_t((s2 / p.nslots) & 1),
                                  kWaitLimitCycles / 8);
    }
  }
}

// ---- row-streaming kernel (batch > 1) and generic kernel launchers -----------

constexpr size_t kTableBytes = 256 * 32 * sizeof(uint32_t);

struct FastConfig {
  int cb, r, ks;
};

template <int B, int CB, int R>
cudaError_t launch_fast_typed(const QuantTensor& t, int64_t N, int64_t K, int ks,
                              const uint16_t* x, float* y, cudaStream_t stream) {
  static_assert(kTableBytes <= 48 * 1024, "table fits the default dynamic shared memory");
  const int64_t rows_per_cta = int64_t(kWarps / ks) * R;
  const int64_t blocks = (N + rows_per_cta - 1) / rows_per_cta;
  return launch_k(gemv_fast_kernel<B, CB, R>, dim3(unsigned(blocks)), dim3(kThreads), kTableBytes,
                  stream, t, N, K, ks, x, y);
}

// K == 0: every output is an empty sum.
__global__ void zero_fill_kernel(float* __restrict__ y, int64_t count) {
  pdl_allow_dependents();
  pdl_wait_prior_grid();
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += int64_t(gridDim.x) * blockDim.x)
    y[i] = 0.0f;
}

template <int B>
cudaError_t launch_generic_typed(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x,
                                 float* y, cudaStream_t stream) {
  const int sms = device_sm_count();
  int64_t blocks = (N + kWarps - 1) / kWarps;
  const int64_t max_blocks = int64_t(sms > 0 ? sms : 1) * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  return launch_k(gemv_generic_kernel<B>, dim3(unsigned(blocks)), dim3(kThreads), 0, stream, t, N,
                  K, x, y);
}

// Chooses chunk width, rows per warp and the K split for the row-streaming
// kernel. Returns cb = 0 if it does not apply.
FastConfig choose_config(const QuantTensor& t, int64_t N, int64_t K, int batch,
                         const uint16_t* x, int sms) {
  FastConfig f{0, 1, 1};
  const uintptr_t pa = reinterpret_cast<uintptr_t>(t.packed);
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x);
  if ((xa & 15u) != 0 || (K % 8) != 0) return f;
  int cands[3] = {16, 8, 4};
  int best = 0;
  double best_eff = -1.0;
  for (int cb : cands) {
    if (batch >= 2 && cb > 8) continue;
    if (batch >= 3 && cb > 4) continue;
    const int ce = 2 * cb;
    if (K % ce != 0) continue;
    if ((int64_t(1) << t.lbs) < ce) continue;
    if ((pa & uintptr_t(cb - 1)) != 0) continue;
    const int64_t cpr = K / ce;
    const int64_t iters = (cpr + 31) / 32;
    const double eff = double(cpr) / double(iters * 32);
    if (eff > best_eff + 0.05) {  // prefer wider chunks unless clearly less efficient
      best_eff = eff;
      best = cb;
    }
  }
  if (best == 0) return f;
  f.cb = best;
  f.r = (batch == 1) ? 4 : 2;
  // Spread small N over the SMs by splitting K across warps of a CTA.
  const int64_t target_ctas = 2 * int64_t(sms);
  f.ks = 1;
  while (f.ks < kWarps) {
    const int64_t rows_per_cta = int64_t(kWarps / f.ks) * f.r;
    const int64_t ctas = (N + rows_per_cta - 1) / rows_per_cta;
    const int64_t cpr = K / (2 * f.cb);
    if (ctas >= target_ctas || cpr < int64_t(64) * f.ks) break;
    f.ks *= 2;
  }
  if (f.r > 1) {
    const int64_t rows_per_cta = int64_t(kWarps / f.ks) * f.r;
    if ((N + rows_per_cta - 1) / rows_per_cta < sms) f.r = 1;
  }
  return f;
}

// ---- batch-1 streaming plan --------------------------------------------------

constexpr int kMaxSmemPerCta = 227 * 1024;

uint32_t align_up_u32(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

int reserved_smem_per_block() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < 64 && cache[dev] > 0) return cache[dev] - 1;  // stored as value + 1
  int r = 0;
  if (cudaDeviceGetAttribute(&r, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) return -1;
  if (dev < 64) cache[dev] = r + 1;  // +1: distinguishes a cached 0 from "not queried"
  return r;
}

// Shared memory: [reduction | code2 | absmax2 | mbarriers | absmax_q | ring
// slots ...] [pair table at the next 64 KB-aligned shared address] [more
// ring slots]. The dynamic window starts after the per-block reserved
// shared memory (the kernel has no static shared variables).
bool plan_stream(const QuantTensor& t, int64_t N, int64_t K, int cb, int rpg, int sms, StreamPlan* p) {
  const int64_t bs = int64_t(1) << t.lbs;
  const int ce = 2 * cb;
  if (K % 32 != 0 || K % ce != 0 || K % bs != 0 || bs < ce) return false;
  const int64_t cpr = K / ce;
  const int64_t tk = (cpr + 31) / 32 * 32;
  if (tk > 512) return false;
  int groups = int(512 / tk);
  if (groups > 8) groups = 8;
  const int64_t row_bytes = K / 2;
  p->tk = int(tk);
  p->groups = groups;
  p->stage_rows = groups * rpg;
  p->spr = int(K / bs);
  const int64_t stage_bytes = int64_t(p->stage_rows) * row_bytes;
  if (stage_bytes > (int64_t(1) << 20) - 16) return false;
  p->stage_bytes = uint32_t(stage_bytes);
  const int64_t ctas0 = N < sms ? N : sms;
  int64_t rpc = (N + ctas0 - 1) / ctas0;
  while ((rpc * p->spr) % 16 != 0) ++rpc;  // each CTA's absmax_q range starts 16-byte aligned
  p->rows_per_cta = rpc;
  const int threads = p->tk * groups + 32;  // consumers + one producer warp
  p->ng_cap = int(((rpc * p->spr) >> t.ls2) + 2);
  if (p->ng_cap > threads) return false;
  p->q_cap = align_up_u32(uint32_t(rpc * p->spr), 16);
  const int64_t nstages = (rpc + p->stage_rows - 1) / p->stage_rows;
  const int res = reserved_smem_per_block();
  if (res < 0) return false;
  uint32_t off = 0;
  p->off_red = off;
  off += align_up_u32(uint32_t(2 * groups * (p->tk / 32) * rpg * 4), 128);
  p->off_c2 = off;
  off += 1024;
  p->off_a2 = off;
  off += align_up_u32(uint32_t(p->ng_cap * 4), 128);
  p->off_bar = off;
  off += align_up_u32(uint32_t((2 * kMaxSlots + 1) * 8), 128);
  p->off_q = off;
  off += align_up_u32(p->q_cap, 128);
  p->off_scale = off;
  off += align_up_u32(uint32_t(rpc * p->spr * 4), 128);
  p->off_part = off;
  off += align_up_u32(uint32_t(rpc * (p->tk / 32) * 4), 128);
  uint32_t tab = (65536u - uint32_t(res) % 65536u) % 65536u;
  if (tab % 256u != 0u) return false;  // the table's 16-byte stores and 256-byte rows need this
  while (tab < off) tab += 65536u;
  p->off_tab = tab;
  if (tab + kPairTableBytes > uint32_t(kMaxSmemPerCta)) return false;
  int slots = 0;
  uint32_t front = off;
  const int64_t want = nstages < kMaxSlots ? nstages : kMaxSlots;
  while (slots < want && front + p->stage_bytes <= tab) {
    p->off_slot[slots++] = front;
    front = align_up_u32(front + p->stage_bytes, 128);
  }
  uint32_t back = tab + kPairTableBytes;
  while (slots < want && back + p->stage_bytes <= uint32_t(kMaxSmemPerCta)) {
    p->off_slot[slots++] = back;
    back = align_up_u32(back + p->stage_bytes, 128);
  }
  if (slots < 1 || (slots < 2 && nstages > 1)) return false;
  p->nslots = slots;
  p->depth = slots < NF4_STREAM_DEPTH ? slots : NF4_STREAM_DEPTH;
  p->smem_bytes = back > tab + kPairTableBytes ? back : tab + kPairTableBytes;
  return true;
}

template <int CB, int RPG>
cudaError_t launch_stream(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x, float* y,
                          const StreamPlan& p, cudaStream_t stream) {
  auto kern = gemv_b1_stream_kernel<CB, RPG>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemPerCta);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = 1;
  }
  const int64_t grid = (N + p.rows_per_cta - 1) / p.rows_per_cta;
  return launch_k(kern, dim3(unsigned(grid)), dim3(unsigned(p.tk * p.groups + 32)), p.smem_bytes,
                  stream, t, N, K, x, y, p);
}

#ifndef NF4_STREAM_RPG
#define NF4_STREAM_RPG 4
#endif

cudaError_t try_stream_b1(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x, float* y,
                          int sms, cudaStream_t stream, bool* done) {
  *done = false;
  if ((reinterpret_cast<uintptr_t>(t.packed) & 15u) != 0 || (reinterpret_cast<uintptr_t>(x) & 15u) != 0)
    return cudaSuccess;
  // chunk width: 16 bytes unless that leaves more than 10% of the lanes idle
  int cb = 0;
  if (K % 32 == 0) {
    const int64_t cpr = K / 32;
    cb = (double(cpr) / double((cpr + 31) / 32 * 32) >= 0.9) ? 16 : 8;
  }
  if (cb == 0) return cudaSuccess;
  StreamPlan p;
  if (cb == 16 && plan_stream(t, N, K, 16, NF4_STREAM_RPG, sms, &p)) {
    *done = true;
    return launch_stream<16, NF4_STREAM_RPG>(t, N, K, x, y, p, stream);
  }
  if (plan_stream(t, N, K, 8, NF4_STREAM_RPG, sms, &p)) {
    *done = true;
    return launch_stream<8, NF4_STREAM_RPG>(t, N, K, x, y, p, stream);
  }
  return cudaSuccess;
}

template <int B>
cudaError_t dispatch_batch(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x,
                           float* y, cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  if (K == 0) {
    const int64_t count = int64_t(B) * N;
    int64_t blocks = (count + kThreads - 1) / kThreads;
    if (blocks > int64_t(sms) * 8) blocks = int64_t(sms) * 8;
    return launch_k(zero_fill_kernel, dim3(unsigned(blocks)), dim3(kThreads), 0, stream, y, count);
  }
#ifndef NF4_GEMV_STREAM
#define NF4_GEMV_STREAM 1
#endif
  if constexpr (B == 1) {
    if (NF4_GEMV_STREAM) {
      bool done = false;
      const cudaError_t ek = try_stream_b1(t, N, K, x, y, sms, stream, &done);
      if (done || ek != cudaSuccess) return ek;
    }
  }
  const FastConfig f = choose_config(t, N, K, B, x, sms);
  if (f.cb == 0) return launch_generic_typed<B>(t, N, K, x, y, stream);
  if constexpr (B == 1) {
    if (f.cb == 16) {
      if (f.r == 4) return launch_fast_typed<1, 16, 4>(t, N, K, f.ks, x, y, stream);
      if (f.r == 2) return launch_fast_typed<1, 16, 2>(t, N, K, f.ks, x, y, stream);
      return launch_fast_typed<1, 16, 1>(t, N, K, f.ks, x, y, stream);
    }
    if (f.cb == 8) {
      if (f.r == 4) return launch_fast_typed<1, 8, 4>(t, N, K, f.ks, x, y, stream);
      if (f.r == 2) return launch_fast_typed<1, 8, 2>(t, N, K, f.ks, x, y, stream);
      return launch_fast_typed<1, 8, 1>(t, N, K, f.ks, x, y, stream);
    }
    if (f.r == 4) return launch_fast_typed<1, 4, 4>(t, N, K, f.ks, x, y, stream);
    if (f.r == 2) return launch_fast_typed<1, 4, 2>(t, N, K, f.ks, x, y, stream);
    return launch_fast_typed<1, 4, 1>(t, N, K, f.ks, x, y, stream);
  } else if constexpr (B == 2) {
    if (f.cb == 8) {
      if (f.r == 2) return launch_fast_typed<2, 8, 2>(t, N, K, f.ks, x, y, stream);
      return launch_fast_typed<2, 8, 1>(t, N, K, f.ks, x, y, stream);
    }
    if (f.r == 2) return launch_fast_typed<2, 4, 2>(t, N, K, f.ks, x, y, stream);
    return launch_fast_typed<2, 4, 1>(t, N, K, f.ks, x, y, stream);
  } else {
    if (f.r == 2) return launch_fast_typed<B, 4, 2>(t, N, K, f.ks, x, y, stream);
    return launch_fast_typed<B, 4, 1>(t, N, K, f.ks, x, y, stream);
  }
}

}  // namespace

cudaError_t read_and_clear_device_flags(unsigned int* flags) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flags, g_device_flags, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_flags, &zero, sizeof(unsigned int));
}

cudaError_t launch_gemv(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x, int batch,
                        float* y, cudaStream_t stream) {
  switch (batch) {
    case 1: return dispatch_batch<1>(t, N, K, x, y, stream);
    case 2: return dispatch_batch<2>(t, N, K, x, y, stream);
    case 3: return dispatch_batch<3>(t, N, K, x, y, stream);
    case 4: return dispatch_batch<4>(t, N, K, x, y, stream);
    case 5: return dispatch_batch<5>(t, N, K, x, y, stream);
    case 6: return dispatch_batch<6>(t, N, K, x, y, stream);
    case 7: return dispatch_batch<7>(t, N, K, x, y, stream);
    case 8: return dispatch_batch<8>(t, N, K, x, y, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nf4
