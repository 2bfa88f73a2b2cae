// nf4_gemv_stream.cu -- batch-1 decode GEMV y = W_hat x with the NF4 double-quant
// dequantization fused, for sm_103a.
//
// What is computed follows "RTX 4060 上的 LLM 量化实测：4-bit decode 比 FP16 慢在
// 哪里", section "Fused kernel：把反量化搬到片上" (packed codes read once,
// decoded and accumulated on chip, only y written) with the scale formula of
// "NF4 双重量化反量化 CUDA Kernel 实现报告", section 1.3. The work split is the
// k-stationary transpose of the warp-per-row GEMV in "CUDA 进阶手册 / 量化与
// GEMV", section "GEMV kernel 的写法": each thread owns one column chunk of
// every row, so x is read once per CTA and kept in registers.
//
// Layout of a CTA (one per SM, 16 warps):
//   * The CTA owns a contiguous, balanced range of rows, split into G
//     contiguous sub-ranges, one per row group of W warps; lane l of warp w of
//     a group owns column chunk 32 w + l (CB packed bytes, 2 CB weights) of
//     every row of its sub-range. Warps beyond G * W only help with the
//     prologue.
//   * Weights go straight from global memory into registers with 16-byte
//     streaming loads (a warp reads 512 contiguous bytes of a row), RPG rows
//     per step and three steps in flight, so no shared-memory staging is
//     needed. (On this GPU a 1-D bulk copy costs about one memory latency of
//     copy-engine time per copy, so copies under ~32 KB cannot stream a CTA's
//     rows at full bandwidth.)
//   * After the grid-dependency wait the small loads (x, code2, absmax2, absmax_q) go out together (as
//     volatile loads, so the compiler keeps them ahead of the weight stream),
//     and the first weight steps once they have arrived and x is converted
//     (loads queue per SM, so a small load issued next to a weight stream
//     would wait behind it); the block scales of the CTA are decoded once
//     into shared memory.
//   * Inner loop per packed byte: one byte permute forms the complete shared
//     address of the byte's entry in a lane-private table of binary16 code
//     pairs (table at a 64 KB-aligned shared address, 256-byte rows, lane l at
//     byte 4l of a row); one 32-bit shared load; two fma.rn.f32.f16 with
//     binary32 accumulation.
//   * x is converted once per CTA into binary16 after an exact power-of-two
//     scaling per column chunk (the upper halves of the table rows hold the
//     converted chunks); a CTA whose x does not convert exactly (dynamic range
//     beyond binary16, NaN/Inf) uses binary32 x with conversions of the codes
//     and packed fma.rn.f32x2 instead. The codes carry a binary16 rounding
//     error of at most 3.3e-4 relative, inside the GEMV tolerance.
//   * Per-warp partial sums of each row go to shared memory; the group's
//     threads add them in warp order (deterministic, no atomics).
#include "nf4_internal.cuh"

namespace nf4 {
namespace {

#ifndef NF4_B1_RPG
#define NF4_B1_RPG 4
#endif

constexpr int kMaxGroups = 15;         // named barriers 1..15

// The weight CTA `cta` serves, selected with compile-time indices only (no
// dynamic indexing of the parameter block).
template <int NSUB>
__device__ __forceinline__ SubTensor pick_sub(const SubTensor (&s)[kMaxSub], int nsub, int cta) {
  SubTensor v = s[0];
#pragma unroll
  for (int i = 1; i < NSUB; ++i)
    if (i < nsub && cta >= s[i].cta0) v = s[i];
  return v;
}
constexpr uint32_t kTabBytes = 65536;  // 256 rows of 256 B
constexpr int kMaxSmemPerCta = 227 * 1024;

// Everything a launch needs, in one argument block. A launch serves one to
// kMaxSub weights that share x (a grouped launch): CTAs [cta0, cta0 + ctas)
// serve weight j, CTA cta0 + b owning its rows [b*N/ctas, (b+1)*N/ctas).
struct B1Args {
  SubTensor sub[kMaxSub];
  int nsub;
  const uint16_t* x;
  int32_t K;
  int W;     // warps per row group (32 * W >= chunks per row)
  int G;     // row groups
  int spr;   // quantization blocks per row
  int cpr;   // column chunks per row
  uint32_t off_c2, off_a2, off_xs, off_q, off_scale, off_part, off_bias, off_tab;
};

struct B1Plan {
  B1Args a;
  int grid;
  uint32_t smem_bytes;
};

bool any_bias(const SubTensor* subs, int nsub) {
  for (int j = 0; j < nsub; ++j)
    if (subs[j].out.bias) return true;
  return false;
}

// Spreads one wave of CTAs (at most `sms`) over the weights of a launch in
// proportion to their rows, at least one CTA per weight and at most one per
// row, and fills cta0 / ctas of out[]. Returns the largest number of rows a
// CTA owns, or -1 when the weights cannot share a launch (an empty weight,
// or block sizes that differ).
int assign_ctas(const SubTensor* subs, int nsub, int sms, SubTensor* out, int* grid_out) {
  if (nsub < 1 || nsub > kMaxSub || sms < nsub) return -1;
  int64_t total = 0;
  for (int j = 0; j < nsub; ++j) {
    if (subs[j].N <= 0 || subs[j].t.lbs != subs[0].t.lbs || subs[j].t.ls2 != subs[0].t.ls2)
      return -1;
    total += subs[j].N;
  }
  const int grid = int(total < sms ? total : sms);
  int ctas[kMaxSub];
  int used = 0;
  for (int j = 0; j < nsub; ++j) {
    int64_t c = int64_t(grid) * subs[j].N / total;
    if (c < 1) c = 1;
    if (c > subs[j].N) c = subs[j].N;
    ctas[j] = int(c);
    used += ctas[j];
  }
  // rows per CTA of weight j with c CTAs, rounded up
  auto load = [&](int j, int c) { return (subs[j].N + c - 1) / c; };
  while (used < grid) {  // give the spare CTAs to the most loaded weights
    int best = -1;
    for (int j = 0; j < nsub; ++j)
      if (ctas[j] < subs[j].N && (best < 0 || load(j, ctas[j]) > load(best, ctas[best]))) best = j;
    if (best < 0) break;
    ++ctas[best];
    ++used;
  }
  while (used > grid) {  // take back from the least loaded
    int best = -1;
    for (int j = 0; j < nsub; ++j)
      if (ctas[j] > 1 && (best < 0 || load(j, ctas[j] - 1) < load(best, ctas[best] - 1))) best = j;
    if (best < 0) return -1;
    --ctas[best];
    --used;
  }
  int64_t max_rows = 0;
  int c0 = 0;
  for (int j = 0; j < kMaxSub; ++j) {
    if (j < nsub) {
      out[j] = subs[j];
      out[j].cta0 = c0;
      out[j].ctas = ctas[j];
      c0 += ctas[j];
      const int64_t r = load(j, ctas[j]);
      if (r > max_rows) max_rows = r;
    } else {
      out[j] = out[0];
      out[j].cta0 = used;  // never selected: past the last CTA
    }
  }
  *grid_out = used;
  return max_rows > (int64_t(1) << 30) ? -1 : int(max_rows);
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds_u128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Prologue loads as volatile PTX, so that they are issued in program order
// (ahead of the weight stream) instead of being moved to their first use.
__device__ __forceinline__ uint4 ldg_v4_ordered(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint16_t ldg_u16_ordered(const uint16_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_u32_ordered(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
// Bias bits of row r (16 or 32 bits as stored), issued in program order.
__device__ __forceinline__ uint32_t bias_bits_ordered(const YOut& o, int64_t r) {
  if (o.dtype == NF4_F32) return ldg_u32_ordered(reinterpret_cast<const uint32_t*>(o.bias) + r);
  return ldg_u16_ordered(reinterpret_cast<const uint16_t*>(o.bias) + r);
}
__device__ __forceinline__ uint8_t ldg_u8_ordered(const uint8_t* p) {
  unsigned int v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
  return uint8_t(v);
}

__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// acc_a += T(low half) * x(low half), acc_b += T(high half) * x(high half):
// binary16 inputs (code pair and x pair, each packed in 32 bits), binary32
// accumulation (the products are exact).
__device__ __forceinline__ void fma2_f16_f32(uint32_t tpair, uint32_t xpair, float& acc_a,
                                             float& acc_b) {
  asm("{\n\t.reg .f16 t0, t1, x0, x1;\n\t"
      "mov.b32 {t0, t1}, %2;\n\t"
      "mov.b32 {x0, x1}, %3;\n\t"
      "fma.rn.f32.f16 %0, t0, x0, %0;\n\t"
      "fma.rn.f32.f16 %1, t1, x1, %1;\n\t}"
      : "+f"(acc_a), "+f"(acc_b)
      : "r"(tpair), "r"(xpair));
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t h) {
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
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

// First row (relative to the CTA) of row group g: balanced contiguous split.
__device__ __forceinline__ int group_row0(int nrows, int G, int g) {
  const int q = nrows / G, r = nrows - q * G;
  return q * g + (g < r ? g : r);
}

// Shared offset of the binary16 x chunk c: the upper 128 bytes of table rows,
// 32 / CB chunks of 4 * CB bytes per row.
template <int CB>
__device__ __forceinline__ uint32_t x16_offset(int c) {
  constexpr int per_row = 32 / CB;
  return uint32_t(c / per_row) * 256u + 128u + uint32_t(c % per_row) * uint32_t(4 * CB);
}

// One step of RPG rows of this lane's column chunk, held in registers.
template <int CB, int RPG>
struct Step {
  uint32_t w[RPG][CB / 4];
};

template <int CB, int RPG>
__device__ __forceinline__ void load_step(Step<CB, RPG>& st, const uint8_t* p, uint32_t row_bytes,
                                          int rows) {
#pragma unroll
  for (int r = 0; r < RPG; ++r) {
    if (r < rows) {
      if constexpr (CB == 16) {
        const uint4 v = ldg_stream_u128(p + r * row_bytes);
        st.w[r][0] = v.x; st.w[r][1] = v.y; st.w[r][2] = v.z; st.w[r][3] = v.w;
      } else if constexpr (CB == 4) {
        st.w[r][0] = ldg_stream_u32(p + r * row_bytes);
      } else {
        uint2 v;
        asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0,%1}, [%2];"
                     : "=r"(v.x), "=r"(v.y)
                     : "l"(p + r * row_bytes));
        st.w[r][0] = v.x; st.w[r][1] = v.y;
      }
    }
  }
}

// Dot product of one row's chunk (CB packed bytes in w) with the lane's x
// chunk. kFast: binary16 x (pre-scaled) and mixed-precision FMAs on the
// binary16 code pairs; otherwise binary32 x and packed binary32 FMAs.
template <int CB, bool kFast>
__device__ __forceinline__ float row_dot(const uint32_t (&w)[CB / 4], uint32_t lanebase,
                                         uint32_t tab_s, uint32_t lane4, const uint32_t (&x16)[CB],
                                         const float2 (&xf)[CB]) {
  if constexpr (kFast) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int wi = 0; wi < CB / 4; ++wi) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t addr = __byte_perm(w[wi], lanebase, 0x7604u | (uint32_t(i) << 4));
        const uint32_t h = lds_u32(addr);
        const int k = 4 * wi + i;
        if (i & 1) fma2_f16_f32(h, x16[k], a2, a3);
        else fma2_f16_f32(h, x16[k], a0, a1);
      }
    }
    return (a0 + a1) + (a2 + a3);
  } else {
    float2 pa = make_float2(0.f, 0.f), pb = make_float2(0.f, 0.f);
#pragma unroll
    for (int wi = 0; wi < CB / 4; ++wi) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t addr = tab_s + __byte_perm(w[wi], lane4, 0x5504u | (uint32_t(i) << 4));
        const float2 tw = half2_bits_to_float2(lds_u32(addr));
        if (i & 1) pb = __ffma2_rn(tw, xf[4 * wi + i], pb);
        else pa = __ffma2_rn(tw, xf[4 * wi + i], pa);
      }
    }
    return (pa.x + pa.y) + (pb.x + pb.y);
  }
}

// Per-thread state of the consumer loop.
template <int CB>
struct Lane {
  uint32_t lanebase, tab_s, lane4;
  uint32_t x16[CB];  // binary16 x pairs (element 2k in the low half)
  float2 xf[CB];
  float xs;  // power of two undoing the x scaling of this chunk (fast path)
  bool act;  // this lane owns a real chunk
  int scol;  // quantization block of the chunk within a row
  const float* sScale;  // decoded scale of block i of the CTA (i = row * spr + scol)
  __device__ __forceinline__ float scale(int i) const { return sScale[i]; }
};

// Computes one step (rows r0 .. r0 + rows - 1 of the CTA) from registers,
// reduces it across the warp and stores one partial per (row, warp).
template <int CB, int RPG, bool kFast>
__device__ __forceinline__ void compute_step(const Step<CB, RPG>& st, const Lane<CB>& L,
                                             float* sPart, int spr, int W, int wg, int lane,
                                             int r0, int rows) {
  // One code path for full and partial steps (a second path for the last
  // step made the loop body too large for the instruction cache): rows past
  // the end are computed from stale registers and dropped.
  float part[RPG];
#pragma unroll
  for (int r = 0; r < RPG; ++r) {
    const float sum = row_dot<CB, kFast>(st.w[r], L.lanebase, L.tab_s, L.lane4, L.x16, L.xf);
    part[r] = (L.act && r < rows) ? __fmul_rn(L.scale((r0 + (r < rows ? r : 0)) * spr + L.scol), L.xs) * sum
                                  : 0.0f;
  }
  const float red = transposed_warp_reduce<RPG>(part, lane);
  if (lane < RPG) {
    const int rr = transposed_index<RPG>(lane);
    if (rr < rows) sPart[(r0 + rr) * W + wg] = red;
  }
}

// The consumer loop of one row group: three steps of RPG rows in flight.
template <int CB, int RPG, bool kFast>
__device__ __forceinline__ void consume(const B1Args& p, const uint8_t* lane_src, uint32_t row_bytes,
                                        Step<CB, RPG>& A, Step<CB, RPG>& B, Step<CB, RPG>& C,
                                        const Lane<CB>& L, float* sPart, int wg, int lane,
                                        int rg0, int rg1) {
  const int n = rg1 - rg0;
  const int ns = (n + RPG - 1) / RPG;
  auto rows_of = [&](int s) { return (n - s * RPG < RPG) ? n - s * RPG : RPG; };
  auto src_of = [&](int s) { return lane_src + uint32_t(rg0 + s * RPG) * row_bytes; };
  for (int s = 0; s < ns; s += 3) {
    compute_step<CB, RPG, kFast>(A, L, sPart, p.spr, p.W, wg, lane, rg0 + s * RPG, rows_of(s));
    if (s + 3 < ns) load_step<CB, RPG>(A, src_of(s + 3), row_bytes, rows_of(s + 3));
    if (s + 1 < ns) {
      compute_step<CB, RPG, kFast>(B, L, sPart, p.spr, p.W, wg, lane, rg0 + (s + 1) * RPG,
                                   rows_of(s + 1));
      if (s + 4 < ns) load_step<CB, RPG>(B, src_of(s + 4), row_bytes, rows_of(s + 4));
    }
    if (s + 2 < ns) {
      compute_step<CB, RPG, kFast>(C, L, sPart, p.spr, p.W, wg, lane, rg0 + (s + 2) * RPG,
                                   rows_of(s + 2));
      if (s + 5 < ns) load_step<CB, RPG>(C, src_of(s + 5), row_bytes, rows_of(s + 5));
    }
  }
}

template <int CB, int RPG, int kThreads, int NSUB>
__global__ void __launch_bounds__(kThreads, 1) gemv_b1_kernel(const B1Args p) {
  constexpr int CE = 2 * CB;  // elements per column chunk
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  // Pair table first (it needs no argument: it sits at shared window address
  // 64 KB, which the host plan reserves). Row e holds (binary16 code of
  // e >> 4, binary16 code of e & 15) at bytes 4l..4l+3 for every lane l;
  // codes come from immediates via shuffles.
  unsigned char* const tab = smem + (65536u - smem_u32(smem));
  {
    const uint32_t my_code16 = __half_as_ushort(__float2half_rn(nf4_code_select(lane & 15)));
#pragma unroll
    for (int j = 0; j < (256 * 8 + kThreads - 1) / kThreads; ++j) {
      const int i = tid + j * kThreads;
      if (i >= 256 * 8) break;  // warp-uniform (all sizes are multiples of 32)
      const int e = i >> 3, q = i & 7;
      const uint32_t hi = __shfl_sync(0xffffffffu, my_code16, e >> 4);
      const uint32_t lo = __shfl_sync(0xffffffffu, my_code16, e & 15);
      const uint32_t v = hi | (lo << 16);
      *reinterpret_cast<uint4*>(tab + e * 256 + q * 16) = make_uint4(v, v, v, v);
    }
  }
  pdl_allow_dependents();

  const SubTensor sb = pick_sub<NSUB>(p.sub, p.nsub, int(blockIdx.x));
  const QuantTensor& t = sb.t;
  const uint16_t* __restrict__ x = p.x;
  const int64_t N = sb.N;
  const int64_t K = p.K;
  float* sC2 = reinterpret_cast<float*>(smem + p.off_c2);
  float* sA2 = reinterpret_cast<float*>(smem + p.off_a2);
  float* sXs = reinterpret_cast<float*>(smem + p.off_xs);
  unsigned char* sQ = smem + p.off_q;
  float* sScale = reinterpret_cast<float*>(smem + p.off_scale);
  float* sPart = reinterpret_cast<float*>(smem + p.off_part);
  uint32_t* sBias = reinterpret_cast<uint32_t*>(smem + p.off_bias);

  const int64_t row_bytes = K >> 1;
  const int64_t bid = int64_t(blockIdx.x) - sb.cta0;
  const int64_t row_begin = (bid * N) / sb.ctas;
  const int64_t row_end = ((bid + 1) * N) / sb.ctas;
  const int nrows = int(row_end - row_begin);
  const int64_t b0 = (row_begin * K) >> t.lbs;  // first quantization block of the CTA
  const int nq = nrows * p.spr;
  const int64_t g0 = b0 >> t.ls2;
  const int ng = nq > 0 ? int(((b0 + nq - 1) >> t.ls2) - g0 + 1) : 0;
  const uint8_t* slab = t.packed + row_begin * row_bytes;

  // This thread's place among the consumers.
  const int g = warp / p.W;
  const int wg = warp - g * p.W;
  const bool consumer = g < p.G;
  const int c = wg * 32 + lane;
  const bool act = consumer && c < p.cpr;
  const int cc = act ? c : p.cpr - 1;
  const int rg0 = consumer ? group_row0(nrows, p.G, g) : 0;
  const int rg1 = consumer ? group_row0(nrows, p.G, g + 1) : 0;
  const uint8_t* lane_src = slab + int64_t(cc) * CB;

  pdl_wait_prior_grid();

  // First round of loads, all issued before any is consumed: x pieces (4 per
  // thread), code2, absmax2, absmax_q.
  constexpr int kPiecesPerChunk = CE / 8;
  const int npieces = int(K / 8);
  uint4 xv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int pc = tid + j * kThreads;
    xv[j] = pc < npieces ? ldg_v4_ordered(reinterpret_cast<const uint4*>(x) + pc) : make_uint4(0u, 0u, 0u, 0u);
  }
  const uint16_t c2v = tid < 256 ? ldg_u16_ordered(t.code2 + tid) : uint16_t(0);
  uint16_t av[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = tid + j * kThreads;
    av[j] = i < ng ? ldg_u16_ordered(t.absmax2 + g0 + i) : uint16_t(0);
  }
  // absmax_q of the CTA: the 16-byte-aligned middle as 16-byte loads, the
  // head and tail bytes singly. Shared index of byte i is q_lead + i, with
  // q_lead = (address of byte 0) mod 16, so the middle lands 16-byte aligned.
  const uintptr_t qa = reinterpret_cast<uintptr_t>(t.absmax_q + b0);
  const int q_lead = int(qa & 15u);
  int q_head = int((16u - (qa & 15u)) & 15u);
  int q_mid_end = int(((qa + uintptr_t(nq)) & ~uintptr_t(15)) - qa);
  if (q_mid_end <= q_head) {  // no aligned middle: every byte singly
    q_head = nq;
    q_mid_end = nq;
  }
  const int q_vecs = (q_mid_end - q_head) / 16;
  uint4 qm[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = tid + j * kThreads;
    qm[j] = i < q_vecs ? ldg_v4_ordered(reinterpret_cast<const uint4*>(t.absmax_q + b0 + q_head) + i)
                       : make_uint4(0u, 0u, 0u, 0u);
  }
  int qi = -1;
  if (tid < q_head) qi = tid;
  else if (tid >= 32 && tid - 32 < nq - q_mid_end) qi = q_mid_end + (tid - 32);
  const uint8_t qb = qi >= 0 ? ldg_u8_ordered(t.absmax_q + b0 + qi) : uint8_t(0);
  // bias of the CTA's rows, kept (as stored) in shared memory for the end
  const bool has_bias = sb.out.bias != nullptr;
  const uint32_t bias_v = (has_bias && tid < nrows) ? bias_bits_ordered(sb.out, row_begin + tid) : 0u;
  // Shared copies of the small inputs (further batches for long ranges).
  if (tid < 256) sC2[tid] = half_bits_to_float(c2v);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = tid + j * kThreads;
    if (i < ng) sA2[i] = half_bits_to_float(av[j]);
    if (i < q_vecs) *reinterpret_cast<uint4*>(sQ + q_lead + q_head + 16 * i) = qm[j];
  }
  if (qi >= 0) sQ[q_lead + qi] = qb;
  if (has_bias) {
    if (tid < nrows) sBias[tid] = bias_v;
    for (int i = tid + kThreads; i < nrows; i += kThreads) sBias[i] = y_bias_bits(sb.out, row_begin + i);
  }
  for (int base = 4 * kThreads; base < ng; base += 4 * kThreads) {  // small group sizes only
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = base + tid + j * kThreads;
      av[j] = i < ng ? __ldg(t.absmax2 + g0 + i) : uint16_t(0);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = base + tid + j * kThreads;
      if (i < ng) sA2[i] = half_bits_to_float(av[j]);
    }
  }

  // x pieces of 8 elements. The chunk's largest |x| (maximum of the bf16
  // magnitude bits, order-preserving) fixes a power of two 2^-e that brings
  // it into [2^14, 2^15); scaling by it is exact, and an element that
  // binary16 cannot hold exactly fails the round-trip test.
  bool x_exact = true;
  for (int base = 0; base < npieces; base += 4 * kThreads) {
    if (base > 0) {  // later batches (rows longer than 16384 elements)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pc = base + tid + j * kThreads;
        xv[j] = pc < npieces ? __ldg(reinterpret_cast<const uint4*>(x) + pc) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (base + j * kThreads + warp * 32 >= npieces) continue;  // warp-uniform
      const int pc = base + tid + j * kThreads;
      const uint32_t w[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
      uint32_t mb = 0u;
#pragma unroll
      for (int q = 0; q < 4; ++q) mb = __vmaxu2(mb, w[q] & 0x7fff7fffu);
      mb = max(mb & 0xffffu, mb >> 16);
#pragma unroll
      for (int m = 1; m < kPiecesPerChunk; m <<= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, m));
      // mb: bf16 magnitude bits of the chunk maximum (>= 0x7f80: Inf/NaN)
      const int em = int(mb >> 7) - 127;  // unbiased exponent (zero/subnormal: -127)
      const int e = (mb == 0u || mb >= 0x7f80u || em <= -100) ? 0 : em - 14;
      const float down = __uint_as_float(uint32_t(127 - e) << 23);  // 2^-e, |e| <= 113
      bool ex = mb < 0x7f80u;
      uint32_t h[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float f0 = __fmul_rn(__uint_as_float(w[q] << 16), down);
        const float f1 = __fmul_rn(__uint_as_float(w[q] & 0xffff0000u), down);
        const __half h0 = __float2half_rn(f0), h1 = __float2half_rn(f1);
        ex = ex && (__half2float(h0) == f0) && (__half2float(h1) == f1);
        h[q] = uint32_t(__half_as_ushort(h0)) | (uint32_t(__half_as_ushort(h1)) << 16);
      }
      if (pc < npieces) {
        const int ch = pc / kPiecesPerChunk;
        const int within = pc - ch * kPiecesPerChunk;
        *reinterpret_cast<uint4*>(tab + x16_offset<CB>(ch) + uint32_t(within) * 16u) =
            make_uint4(h[0], h[1], h[2], h[3]);
        if (within == 0) sXs[ch] = __uint_as_float(uint32_t(127 + e) << 23);
        x_exact = x_exact && ex;
      }
    }
  }
  // The first three weight steps go out once this thread's small loads have
  // arrived and its x pieces are converted: loads queue per SM, so a small
  // load issued next to a weight stream would wait behind it.
  asm volatile("" ::: "memory");  // keep the weight loads after the stores above
  Step<CB, RPG> A, B, C;
  const int n_rows = rg1 - rg0;
  const int n_steps = (n_rows + RPG - 1) / RPG;
  auto rows_of = [&](int s) { return (n_rows - s * RPG < RPG) ? n_rows - s * RPG : RPG; };
  const uint32_t rb = uint32_t(row_bytes);
  if (n_steps > 0) load_step<CB, RPG>(A, lane_src + uint32_t(rg0) * rb, rb, rows_of(0));
  if (n_steps > 1) load_step<CB, RPG>(B, lane_src + uint32_t(rg0 + RPG) * rb, rb, rows_of(1));
  if (n_steps > 2) load_step<CB, RPG>(C, lane_src + uint32_t(rg0 + 2 * RPG) * rb, rb, rows_of(2));

  // the table must be where the plan put it (64 KB-aligned) for the fast path
  const bool fast = !__syncthreads_or(!(x_exact && tab == smem + p.off_tab));

  // One decoded scale per block of this CTA's rows: fp32(fp32(code2[q] *
  // absmax2[g]) + offset) (32-bit indices: b0 is only needed modulo the group
  // size).
  {
    const uint32_t b0g = uint32_t(b0 & ((int64_t(1) << t.ls2) - 1));
    for (int i = tid; i < nq; i += kThreads)
      sScale[i] = __fadd_rn(__fmul_rn(sC2[sQ[q_lead + i]], sA2[(b0g + uint32_t(i)) >> t.ls2]), t.offset);
  }
  __syncthreads();
  if (!consumer) return;

  Lane<CB> L;
  L.tab_s = smem_u32(tab);
  L.lanebase = (L.tab_s & 0xffff0000u) | (uint32_t(lane) << 2);
  L.lane4 = uint32_t(lane) << 2;
  L.act = act;
  L.scol = int((int64_t(cc) * CE) >> t.lbs);
  L.sScale = sScale;
  if (fast) {
    L.xs = act ? sXs[cc] : 1.0f;
#pragma unroll
    for (int q = 0; q < CE / 8; ++q) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (act) v = lds_u128(L.tab_s + x16_offset<CB>(cc) + uint32_t(q) * 16u);
      L.x16[4 * q + 0] = v.x;
      L.x16[4 * q + 1] = v.y;
      L.x16[4 * q + 2] = v.z;
      L.x16[4 * q + 3] = v.w;
    }
    consume<CB, RPG, true>(p, lane_src, uint32_t(row_bytes), A, B, C, L, sPart, wg, lane, rg0, rg1);
  } else {
    L.xs = 1.0f;
#pragma unroll
    for (int q = 0; q < CE / 8; ++q) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (act) v = __ldg(reinterpret_cast<const uint4*>(x + int64_t(cc) * CE) + q);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        L.xf[4 * q + j] = make_float2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u));
    }
    consume<CB, RPG, false>(p, lane_src, uint32_t(row_bytes), A, B, C, L, sPart, wg, lane, rg0, rg1);
  }

  // End of the group: one sum per row over the group's warps, in order.
  named_barrier(1 + g, p.W * 32);
  const int gt = tid - g * p.W * 32;
  for (int r = rg0 + gt; r < rg1; r += p.W * 32) {
    float v = 0.0f;
    for (int w = 0; w < p.W; ++w) v += sPart[r * p.W + w];
    y_store(sb.out, row_begin + r, v, has_bias ? sBias[r] : 0u);
  }
}

uint32_t align_up_u32(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

int reserved_smem_per_block() {
  static PerDeviceCache cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  return cache.get(dev, [dev] {
    int r = 0;
    if (cudaDeviceGetAttribute(&r, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) return -1;
    return r;
  });
}

// Shared memory: [code2 | absmax2 | x scales | absmax_q | scales | partial
// sums] below the pair table (+ binary16 x) at shared window address 64 KB.
// The dynamic window starts after the per-block reserved shared memory (the
// kernel has no static shared variables).
bool plan_b1(const SubTensor* subs, int nsub, int64_t K, const uint16_t* x, int cb, int threads,
             int sms, B1Plan* plan) {
  const int kWarps = threads / 32;
  B1Args* p = &plan->a;
  const QuantTensor& t = subs[0].t;
  const int64_t bs = int64_t(1) << t.lbs;
  const int ce = 2 * cb;
  if (K % 32 != 0 || K % bs != 0 || bs < ce || K > 16384) return false;
  const int64_t cpr = K / ce;
  const int W = int((cpr + 31) / 32);
  if (W > kWarps) return false;
  int G = kWarps / W;
  if (G > kMaxGroups) G = kMaxGroups;
  const int max_rows = assign_ctas(subs, nsub, sms, p->sub, &plan->grid);
  if (max_rows <= 0) return false;
  p->nsub = nsub;
  p->x = x;
  p->K = int32_t(K);
  p->W = W;
  p->cpr = int(cpr);
  p->spr = int(K / bs);
  if (G > max_rows) G = max_rows;
  p->G = G;
  const int64_t max_nq = int64_t(max_rows) * p->spr;
  const int ng_cap = int((max_nq >> t.ls2) + 2);
  const int res = reserved_smem_per_block();
  if (res <= 0 || res >= 65536 || res % 256 != 0) return false;
  uint32_t off = 0;
  p->off_c2 = off;
  off += 1024;
  p->off_a2 = off;
  off += align_up_u32(uint32_t(ng_cap * 4), 128);
  p->off_xs = off;
  off += align_up_u32(uint32_t(cpr * 4), 128);
  p->off_q = off;
  if (max_nq > int64_t(4) * threads * 16) return false;  // one batch of 16-byte loads
  off += align_up_u32(uint32_t(max_nq + 16), 128);
  p->off_scale = off;
  off += align_up_u32(uint32_t(max_nq * 4), 128);
  p->off_part = off;
  off += align_up_u32(uint32_t(max_rows * W * 4), 128);
  p->off_bias = off;
  if (any_bias(subs, nsub)) off += align_up_u32(uint32_t(max_rows * 4), 128);
  const uint32_t tab = 65536u - uint32_t(res);
  if (off > tab) return false;
  p->off_tab = tab;
  plan->smem_bytes = tab + kTabBytes;
  return plan->smem_bytes <= uint32_t(kMaxSmemPerCta);
}

template <int CB, int NT, int NSUB>
cudaError_t launch_b1(const B1Plan& plan, cudaStream_t stream) {
  auto kern = gemv_b1_kernel<CB, NF4_B1_RPG, NT, NSUB>;
  static PerDeviceCache attr_set;
  const cudaError_t e = set_max_dynamic_smem_once(kern, kMaxSmemPerCta, attr_set);
  if (e != cudaSuccess) return e;
  return launch_k(kern, dim3(unsigned(plan.grid)), dim3(unsigned(NT)), plan.smem_bytes, stream,
                  plan.a);
}


// ---------------------------------------------------------------------------
// Batch 2..8. Same layout as batch 1 (k-stationary, direct weight loads, RPG
// rows per step, three steps in flight, four on 256 threads), with x kept in
// binary32 (bfloat16 widens exactly, so there is no conversion to check): the
// lane's x chunk of every vector stays in registers. The code-pair table holds binary32 pairs
// (lane-private, 256-byte rows, lane l at byte 8l), so one byte permute, one
// 64-bit shared load and one packed fma.rn.f32x2 per vector handle a packed
// byte. The kernel runs BP = 2, 4 or 8 vectors (3 runs as 4, 5..7 as 8 with
// zero vectors that are not written): 16-byte chunks on 512 threads for 2,
// 8-byte chunks on 512 threads for 4 and on 256 threads for 8 (128 x values
// per lane). The block scale is applied inside the warp reduction, once a
// block's lanes are summed. Rows longer than the CTA's lanes are walked in
// column slices; a warp adds its reduced partial of every slice to its own
// (row, vector) slot, so the sums keep a fixed order.

template <int BP, int CB>
struct LaneN {
  uint32_t lanebase8;  // (table address & 0xffff0000) | 8 * lane
  float2 xf[BP][CB];   // x pairs of this lane's chunk, per vector
  bool act;            // this lane owns a real chunk in the current slice
  int scol;            // quantization block of the chunk within a row
};

__device__ __forceinline__ float2 lds_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

// One step (rows r0 .. r0 + rows - 1 of the CTA): per row and vector, the
// lane's dot product; transposed warp reduction over the RPG * BP values,
// with the block scale applied once the lanes of one quantization block
// (32 / CB adjacent lanes: blocks of at least 64 elements) have been summed;
// partial added to (or stored in, for the first slice)
// sPart[(row * BP + vector) * W + warp].
template <int BP, int CB, int RPG>
__device__ __forceinline__ void compute_step_n(const Step<CB, RPG>& st, const LaneN<BP, CB>& L,
                                               const float* sScale, float* sPart, int spr, int W,
                                               int wg, int lane, int r0, int rows, bool first) {
  constexpr int V = RPG * BP;
  // lanes of one 64-element block: 32 / CB (2^kPre); log2(V) transposed steps
  constexpr int kPre = CB == 4 ? 3 : CB == 8 ? 2 : 1;
  constexpr int kSteps = V == 4 ? 2 : V == 8 ? 3 : 4;
  static_assert(RPG == 2 && (CB == 4 || CB == 8 || CB == 16) && (V == 4 || V == 8 || V == 16) &&
                    kPre < kSteps,
                "two rows per step; the block's lanes are summed before the last transposed step");
  float part[V];
#pragma unroll
  for (int r = 0; r < RPG; ++r) {
    float2 acc[BP];
#pragma unroll
    for (int b = 0; b < BP; ++b) acc[b] = make_float2(0.f, 0.f);
    {  // rows past the end are computed from stale registers and dropped
#pragma unroll
      for (int wi = 0; wi < CB / 4; ++wi) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t addr = __byte_perm(st.w[r][wi], L.lanebase8, 0x7604u | (uint32_t(i) << 4));
          const float2 tw = lds_f2(addr);
          const int k = 4 * wi + i;
#pragma unroll
          for (int b = 0; b < BP; ++b) acc[b] = __ffma2_rn(tw, L.xf[b][k], acc[b]);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < BP; ++b) part[r * BP + b] = acc[b].x + acc[b].y;  // lanes past the row have x = 0
  }
  // Transposed steps: the first sends row 1 to the odd lanes; after the
  // steps over the lanes of one block (masks 1 .. 16 / CB) a lane holds
  // V >> kPre values of row (lane & 1), summed over its block's lanes, which
  // take the block scale; the remaining steps and plain butterfly steps
  // combine the blocks.
  auto exchange = [&](int step) {
    const int cnt = V >> step;
    const int m = 1 << step;
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const float send = upper ? part[i] : part[i + cnt / 2];
      const float keep = upper ? part[i + cnt / 2] : part[i];
      part[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  };
#pragma unroll
  for (int step = 0; step < kPre; ++step) exchange(step);
  {
    const int r = lane & 1;  // rows past the end (stale registers) get scale 0
    const float sc = r < rows ? sScale[(r0 + r) * spr + L.scol] : 0.0f;
#pragma unroll
    for (int i = 0; i < (V >> kPre); ++i) part[i] *= sc;
  }
#pragma unroll
  for (int step = kPre; step < kSteps; ++step) exchange(step);
  float red = part[0];
#pragma unroll
  for (int m = V; m < 32; m <<= 1) red += __shfl_xor_sync(0xffffffffu, red, m);
  if (lane < RPG * BP) {
    const int idx = transposed_index<RPG * BP>(lane);
    const int r = idx / BP, b = idx - (idx / BP) * BP;
    if (r < rows) {
      float* d = sPart + ((r0 + r) * BP + b) * W + wg;
      *d = first ? red : *d + red;
    }
  }
}

template <int BP, int CB, int RPG>
__device__ __forceinline__ void consume_n(const uint8_t* lane_src, uint32_t row_bytes,
                                          Step<CB, RPG>& A, Step<CB, RPG>& B, Step<CB, RPG>& C,
                                          const LaneN<BP, CB>& L, const float* sScale, float* sPart,
                                          int spr, int W, int wg, int lane, int rg0, int rg1,
                                          bool first) {
  const int n = rg1 - rg0;
  const int ns = (n + RPG - 1) / RPG;
  auto rows_of = [&](int s) { return (n - s * RPG < RPG) ? n - s * RPG : RPG; };
  auto src_of = [&](int s) { return lane_src + uint32_t(rg0 + s * RPG) * row_bytes; };
  for (int s = 0; s < ns; s += 3) {
    compute_step_n<BP, CB, RPG>(A, L, sScale, sPart, spr, W, wg, lane, rg0 + s * RPG, rows_of(s), first);
    if (s + 3 < ns) load_step<CB, RPG>(A, src_of(s + 3), row_bytes, rows_of(s + 3));
    if (s + 1 < ns) {
      compute_step_n<BP, CB, RPG>(B, L, sScale, sPart, spr, W, wg, lane, rg0 + (s + 1) * RPG,
                                  rows_of(s + 1), first);
      if (s + 4 < ns) load_step<CB, RPG>(B, src_of(s + 4), row_bytes, rows_of(s + 4));
    }
    if (s + 2 < ns) {
      compute_step_n<BP, CB, RPG>(C, L, sScale, sPart, spr, W, wg, lane, rg0 + (s + 2) * RPG,
                                  rows_of(s + 2), first);
      if (s + 5 < ns) load_step<CB, RPG>(C, src_of(s + 5), row_bytes, rows_of(s + 5));
    }
  }
}

// The same loop with four steps in flight (the 256-thread kernel has the
// registers for a fourth step buffer).
template <int BP, int CB, int RPG>
__device__ __forceinline__ void consume_n4(const uint8_t* lane_src, uint32_t row_bytes,
                                           Step<CB, RPG>& A, Step<CB, RPG>& B, Step<CB, RPG>& C,
                                           Step<CB, RPG>& D, const LaneN<BP, CB>& L,
                                           const float* sScale, float* sPart, int spr, int W, int wg,
                                           int lane, int rg0, int rg1, bool first) {
  const int n = rg1 - rg0;
  const int ns = (n + RPG - 1) / RPG;
  auto rows_of = [&](int s) { return (n - s * RPG < RPG) ? n - s * RPG : RPG; };
  auto src_of = [&](int s) { return lane_src + uint32_t(rg0 + s * RPG) * row_bytes; };
  for (int s = 0; s < ns; s += 4) {
    compute_step_n<BP, CB, RPG>(A, L, sScale, sPart, spr, W, wg, lane, rg0 + s * RPG, rows_of(s), first);
    if (s + 4 < ns) load_step<CB, RPG>(A, src_of(s + 4), row_bytes, rows_of(s + 4));
    if (s + 1 < ns) {
      compute_step_n<BP, CB, RPG>(B, L, sScale, sPart, spr, W, wg, lane, rg0 + (s + 1) * RPG,
                                  rows_of(s + 1), first);
      if (s + 5 < ns) load_step<CB, RPG>(B, src_of(s + 5), row_bytes, rows_of(s + 5));
    }
    if (s + 2 < ns) {
      compute_step_n<BP, CB, RPG>(C, L, sScale, sPart, spr, W, wg, lane, rg0 + (s + 2) * RPG,
                                  rows_of(s + 2), first);
      if (s + 6 < ns) load_step<CB, RPG>(C, src_of(s + 6), row_bytes, rows_of(s + 6));
    }
    if (s + 3 < ns) {
      compute_step_n<BP, CB, RPG>(D, L, sScale, sPart, spr, W, wg, lane, rg0 + (s + 3) * RPG,
                                  rows_of(s + 3), first);
      if (s + 7 < ns) load_step<CB, RPG>(D, src_of(s + 7), row_bytes, rows_of(s + 7));
    }
  }
}

// Arguments of the batched kernel (grouped launches as for batch 1).
struct BNArgs {
  SubTensor sub[kMaxSub];
  int nsub;
  const uint16_t* x;
  int32_t K;
  int batch;   // real vectors (<= BP)
  int W;       // warps per row group (per slice)
  int G;       // row groups
  int spr;     // quantization blocks per row
  int cpr;     // column chunks per row
  int slices;  // column slices of W * 32 chunks
  uint32_t off_c2, off_a2, off_q, off_scale, off_part, off_bias, off_tab;
};

template <int BP, int CB, int RPG, int NSUB, int NT>
__global__ void __launch_bounds__(NT, 1) gemv_bn_kernel(const BNArgs p) {
  constexpr int kThreads = NT;
  static_assert(NT >= 256 && NT % 32 == 0, "the prologue loads assume at least 256 threads");
  constexpr int CE = 2 * CB;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  // binary32 pair table at shared window address 64 KB: row e holds
  // (NF4[e >> 4], NF4[e & 15]) at bytes 8l..8l+7 for every lane l.
  unsigned char* const tab = smem + (65536u - smem_u32(smem));
  {
    const float my_code = nf4_code_select(lane & 15);
#pragma unroll
    for (int j = 0; j < 256 * 16 / kThreads; ++j) {
      const int i = tid + j * kThreads;
      const int e = i >> 4, q = i & 15;
      const float hi = __shfl_sync(0xffffffffu, my_code, e >> 4);
      const float lo = __shfl_sync(0xffffffffu, my_code, e & 15);
      *reinterpret_cast<float4*>(tab + e * 256 + q * 16) = make_float4(hi, lo, hi, lo);
    }
  }
  pdl_allow_dependents();

  const SubTensor sb = pick_sub<NSUB>(p.sub, p.nsub, int(blockIdx.x));
  const QuantTensor& t = sb.t;
  const int64_t N = sb.N;
  const int64_t K = p.K;
  float* sC2 = reinterpret_cast<float*>(smem + p.off_c2);
  float* sA2 = reinterpret_cast<float*>(smem + p.off_a2);
  unsigned char* sQ = smem + p.off_q;
  float* sScale = reinterpret_cast<float*>(smem + p.off_scale);
  float* sPart = reinterpret_cast<float*>(smem + p.off_part);
  uint32_t* sBias = reinterpret_cast<uint32_t*>(smem + p.off_bias);

  const int64_t row_bytes = K >> 1;
  const int64_t bid = int64_t(blockIdx.x) - sb.cta0;
  const int64_t row_begin = (bid * N) / sb.ctas;
  const int64_t row_end = ((bid + 1) * N) / sb.ctas;
  const int nrows = int(row_end - row_begin);
  const int64_t b0 = (row_begin * K) >> t.lbs;
  const int nq = nrows * p.spr;
  const int64_t g0 = b0 >> t.ls2;
  const int ng = nq > 0 ? int(((b0 + nq - 1) >> t.ls2) - g0 + 1) : 0;
  const uint8_t* slab = t.packed + row_begin * row_bytes;

  const int g = warp / p.W;
  const int wg = warp - g * p.W;
  const bool consumer = g < p.G;
  const int rg0 = consumer ? group_row0(nrows, p.G, g) : 0;
  const int rg1 = consumer ? group_row0(nrows, p.G, g + 1) : 0;
  pdl_wait_prior_grid();

  // Small loads first (ordered), then the stores that consume them.
  const uint16_t c2v = tid < 256 ? ldg_u16_ordered(t.code2 + tid) : uint16_t(0);
  uint16_t av[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = tid + j * kThreads;
    av[j] = i < ng ? ldg_u16_ordered(t.absmax2 + g0 + i) : uint16_t(0);
  }
  const uintptr_t qa = reinterpret_cast<uintptr_t>(t.absmax_q + b0);
  const int q_lead = int(qa & 15u);
  int q_head = int((16u - (qa & 15u)) & 15u);
  int q_mid_end = int(((qa + uintptr_t(nq)) & ~uintptr_t(15)) - qa);
  if (q_mid_end <= q_head) {
    q_head = nq;
    q_mid_end = nq;
  }
  const int q_vecs = (q_mid_end - q_head) / 16;
  uint4 qm[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = tid + j * kThreads;
    qm[j] = i < q_vecs ? ldg_v4_ordered(reinterpret_cast<const uint4*>(t.absmax_q + b0 + q_head) + i)
                       : make_uint4(0u, 0u, 0u, 0u);
  }
  int qi = -1;
  if (tid < q_head) qi = tid;
  else if (tid >= 32 && tid - 32 < nq - q_mid_end) qi = q_mid_end + (tid - 32);
  const uint8_t qb = qi >= 0 ? ldg_u8_ordered(t.absmax_q + b0 + qi) : uint8_t(0);
  // bias of the CTA's rows, kept (as stored) in shared memory for the end
  const bool has_bias = sb.out.bias != nullptr;
  const uint32_t bias_v = (has_bias && tid < nrows) ? bias_bits_ordered(sb.out, row_begin + tid) : 0u;
  if (tid < 256) sC2[tid] = half_bits_to_float(c2v);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = tid + j * kThreads;
    if (i < ng) sA2[i] = half_bits_to_float(av[j]);
    if (i < q_vecs) *reinterpret_cast<uint4*>(sQ + q_lead + q_head + 16 * i) = qm[j];
  }
  if (qi >= 0) sQ[q_lead + qi] = qb;
  if (has_bias) {
    if (tid < nrows) sBias[tid] = bias_v;
    for (int i = tid + kThreads; i < nrows; i += kThreads) sBias[i] = y_bias_bits(sb.out, row_begin + i);
  }
  for (int base = 4 * kThreads; base < ng; base += 4 * kThreads) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = base + tid + j * kThreads;
      av[j] = i < ng ? ldg_u16_ordered(t.absmax2 + g0 + i) : uint16_t(0);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = base + tid + j * kThreads;
      if (i < ng) sA2[i] = half_bits_to_float(av[j]);
    }
  }
  __syncthreads();
  {
    const uint32_t b0g = uint32_t(b0 & ((int64_t(1) << t.ls2) - 1));
    for (int i = tid; i < nq; i += kThreads)
      sScale[i] = __fadd_rn(__fmul_rn(sC2[sQ[q_lead + i]], sA2[(b0g + uint32_t(i)) >> t.ls2]), t.offset);
  }
  __syncthreads();
  if (!consumer) return;

  LaneN<BP, CB> L;
  L.lanebase8 = (smem_u32(tab) & 0xffff0000u) | (uint32_t(lane) << 3);
  const uint32_t rb = uint32_t(row_bytes);
  const int n_rows = rg1 - rg0;
  const int n_steps = (n_rows + RPG - 1) / RPG;
  auto rows_of = [&](int s) { return (n_rows - s * RPG < RPG) ? n_rows - s * RPG : RPG; };
  for (int sl = 0; sl < p.slices; ++sl) {
    const int c = sl * p.W * 32 + wg * 32 + lane;
    L.act = c < p.cpr;
    const int cc = L.act ? c : p.cpr - 1;
    L.scol = int((int64_t(cc) * CE) >> t.lbs);
    const uint8_t* lane_src = slab + uint32_t(cc) * CB;
    Step<CB, RPG> A, B, C, D;
    if (n_steps > 0) load_step<CB, RPG>(A, lane_src + uint32_t(rg0) * rb, rb, rows_of(0));
    if (n_steps > 1) load_step<CB, RPG>(B, lane_src + uint32_t(rg0 + RPG) * rb, rb, rows_of(1));
    if (n_steps > 2) load_step<CB, RPG>(C, lane_src + uint32_t(rg0 + 2 * RPG) * rb, rb, rows_of(2));
    if (NT == 256 && n_steps > 3)  // a fourth step in flight where the registers allow
      load_step<CB, RPG>(D, lane_src + uint32_t(rg0 + 3 * RPG) * rb, rb, rows_of(3));
    // x chunk of every vector (bfloat16 -> binary32 exactly); missing
    // vectors and lanes past the row are zero
#pragma unroll
    for (int b = 0; b < BP; ++b) {
#pragma unroll
      for (int q = 0; q < CE / 8; ++q) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (L.act && b < p.batch)
          v = __ldg(reinterpret_cast<const uint4*>(p.x + int64_t(b) * K + int64_t(cc) * CE) + q);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          L.xf[b][4 * q + j] = make_float2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u));
      }
    }
    if constexpr (NT == 256)
      consume_n4<BP, CB, RPG>(lane_src, rb, A, B, C, D, L, sScale, sPart, p.spr, p.W, wg, lane, rg0,
                              rg1, sl == 0);
    else
      consume_n<BP, CB, RPG>(lane_src, rb, A, B, C, L, sScale, sPart, p.spr, p.W, wg, lane, rg0, rg1,
                             sl == 0);
  }

  // End of the group: one sum per (row, vector) over the group's warps.
  named_barrier(1 + g, p.W * 32);
  const int gt = tid - g * p.W * 32;
  for (int idx = gt; idx < n_rows * BP; idx += p.W * 32) {
    const int r = rg0 + idx / BP, b = idx - (idx / BP) * BP;
    if (b >= p.batch) continue;
    float v = 0.0f;
    for (int w = 0; w < p.W; ++w) v += sPart[(r * BP + b) * p.W + w];
    y_store(sb.out, int64_t(b) * N + row_begin + r, v, has_bias ? sBias[r] : 0u);
  }
}

// Plan for BP vectors, CB-byte chunks and nt threads (one CTA per SM).
bool plan_bn(const SubTensor* subs, int nsub, int64_t K, const uint16_t* x, int batch, int bp,
             int cb, int nt, int sms, BNArgs* p, int* grid, uint32_t* smem_bytes) {
  const int warps = nt / 32;
  const QuantTensor& t = subs[0].t;
  const int64_t bs = int64_t(1) << t.lbs;
  const int ce = 2 * cb;
  // blocks of at least 64 elements: a block's lanes are adjacent groups of
  // 32 / cb lanes (the scale is applied inside the warp reduction)
  if (K % 32 != 0 || K % bs != 0 || bs < 64) return false;
  const int64_t cpr = K / ce;
  int W = int((cpr + 31) / 32);
  int slices = 1;
  if (W > warps) {
    slices = int((W + warps - 1) / warps);
    W = int((cpr + 32 * slices - 1) / (32 * slices));
  }
  int G = warps / W;
  if (G > kMaxGroups) G = kMaxGroups;
  const int max_rows = assign_ctas(subs, nsub, sms, p->sub, grid);
  if (max_rows <= 0) return false;
  p->nsub = nsub;
  p->x = x;
  p->K = int32_t(K);
  p->batch = batch;
  p->W = W;
  p->cpr = int(cpr);
  p->slices = slices;
  p->spr = int(K / bs);
  if (G > max_rows) G = max_rows;
  if (slices > 1) G = 1;
  p->G = G;
  const int64_t max_nq = int64_t(max_rows) * p->spr;
  if (max_nq > int64_t(4) * nt * 16) return false;
  const int ng_cap = int((max_nq >> t.ls2) + 2);
  const int res = reserved_smem_per_block();
  if (res <= 0 || res >= 65536 || res % 256 != 0) return false;
  uint32_t off = 0;
  p->off_c2 = off;
  off += 1024;
  p->off_a2 = off;
  off += align_up_u32(uint32_t(ng_cap * 4), 128);
  p->off_q = off;
  off += align_up_u32(uint32_t(max_nq + 16), 128);
  p->off_scale = off;
  off += align_up_u32(uint32_t(max_nq * 4), 128);
  p->off_part = off;
  off += align_up_u32(uint32_t(max_rows * bp * W * 4), 128);
  p->off_bias = off;
  if (any_bias(subs, nsub)) off += align_up_u32(uint32_t(max_rows * 4), 128);
  const uint32_t tab = 65536u - uint32_t(res);
  if (off > tab) return false;
  p->off_tab = tab;
  *smem_bytes = tab + kTabBytes;
  return *smem_bytes <= uint32_t(kMaxSmemPerCta);
}

template <int BP, int CB, int NSUB, int NT>
cudaError_t launch_bn(const BNArgs& a, int grid, uint32_t smem_bytes, cudaStream_t stream) {
  auto kern = gemv_bn_kernel<BP, CB, 2, NSUB, NT>;
  static PerDeviceCache attr_set;
  const cudaError_t e = set_max_dynamic_smem_once(kern, kMaxSmemPerCta, attr_set);
  if (e != cudaSuccess) return e;
  return launch_k(kern, dim3(unsigned(grid)), dim3(unsigned(NT)), smem_bytes, stream, a);
}

template <int BP, int CB, int NT>
cudaError_t launch_bn_n(const BNArgs& a, int grid, uint32_t smem_bytes, cudaStream_t stream) {
  return a.nsub == 1 ? launch_bn<BP, CB, 1, NT>(a, grid, smem_bytes, stream)
                     : launch_bn<BP, CB, kMaxSub, NT>(a, grid, smem_bytes, stream);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t try_gemv_b1(const SubTensor* subs, int nsub, int64_t K, const uint16_t* x, int sms,
                        cudaStream_t stream, bool* done) {
  *done = false;
  if (!aligned16(x) || K % 32 != 0) return cudaSuccess;
  for (int j = 0; j < nsub; ++j)
    if (!aligned16(subs[j].t.packed)) return cudaSuccess;
  // chunk width: 16 bytes unless that leaves more than 10% of the lanes idle
  // (measured: more, narrower lanes only add per-row overhead)
  const int64_t cpr16 = K / 32;
  const int cb = (double(cpr16) / double((cpr16 + 31) / 32 * 32) >= 0.9) ? 16 : 8;
  B1Plan p;
  const bool one = nsub == 1;
  if (cb == 16 && plan_b1(subs, nsub, K, x, 16, 512, sms, &p)) {
    *done = true;
    return one ? launch_b1<16, 512, 1>(p, stream) : launch_b1<16, 512, kMaxSub>(p, stream);
  }
  if (plan_b1(subs, nsub, K, x, 8, 512, sms, &p)) {
    *done = true;
    return one ? launch_b1<8, 512, 1>(p, stream) : launch_b1<8, 512, kMaxSub>(p, stream);
  }
  return cudaSuccess;
}

cudaError_t try_gemv_bn(const SubTensor* subs, int nsub, int64_t K, const uint16_t* x, int batch,
                        int sms, cudaStream_t stream, bool* done) {
  *done = false;
  if (batch < 2 || batch > 8 || !aligned16(x)) return cudaSuccess;
  for (int j = 0; j < nsub; ++j)
    if (!aligned16(subs[j].t.packed)) return cudaSuccess;
  // x chunk of all BP vectors in registers: BP * 2 CB binary32 values, 64
  // on 512 threads or 128 on 256
  BNArgs a;
  int grid = 0;
  uint32_t smem = 0;
  if (batch == 2) {
    if (!plan_bn(subs, nsub, K, x, batch, 2, 16, 512, sms, &a, &grid, &smem)) return cudaSuccess;
    *done = true;
    return launch_bn_n<2, 16, 512>(a, grid, smem, stream);
  }
  if (batch <= 4) {
    if (!plan_bn(subs, nsub, K, x, batch, 4, 8, 512, sms, &a, &grid, &smem)) return cudaSuccess;
    *done = true;
    return launch_bn_n<4, 8, 512>(a, grid, smem, stream);
  }
  // 5..8 vectors: 8-byte chunks (128 binary32 x values per lane) on 256
  // threads, half the reduction work per weight of 4-byte chunks on 512
  if (!plan_bn(subs, nsub, K, x, batch, 8, 8, 256, sms, &a, &grid, &smem)) return cudaSuccess;
  *done = true;
  return launch_bn_n<8, 8, 256>(a, grid, smem, stream);
}


}  // namespace nf4
