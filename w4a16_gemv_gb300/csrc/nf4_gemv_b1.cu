// nf4_gemv_b1.cu -- batch-1 decode GEMV y = W_hat x with the NF4 double-quant
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
//     contiguous sub-ranges of whole RPG-row steps, one per row group of W
//     warps; lane l of warp w of a group owns column chunk 32 w + l (CB packed
//     bytes, 2 CB weights) of every row of its sub-range. Warps beyond G * W
//     only help with the prologue.
//   * Weights go straight from global memory into registers with 16-byte
//     streaming loads (a warp reads 512 contiguous bytes of a row), RPG rows
//     per step and two steps in flight, so no shared-memory staging is
//     needed (three steps in flight measured 1-3% slower per layer: the
//     larger burst of loads delays the shared-memory work behind it). (On this GPU a 1-D bulk copy costs about one memory latency of
//     copy-engine time per copy, so copies under ~32 KB cannot stream a CTA's
//     rows at full bandwidth.)
//   * After the grid-dependency wait the small loads (x, code2, absmax2,
//     absmax_q) go out together (as volatile loads, so the compiler keeps them
//     ahead of the weight stream),
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
//     converted chunks, piece-major so that neither the stores nor the
//     per-lane read-back has bank conflicts); a CTA whose x does not convert
//     exactly (dynamic range beyond binary16, NaN/Inf) uses binary32 x with
//     conversions of the codes and packed fma.rn.f32x2 instead. The codes
//     carry a binary16 rounding error of at most 3.3e-4 relative, inside the
//     GEMV tolerance.
//   * Per-warp partial sums of each row go to shared memory; the group's
//     threads add them in warp order (deterministic, no atomics).

#include "nf4_gemv_common.cuh"

namespace nf4 {
namespace {

#ifndef NF4_B1_RPG
#define NF4_B1_RPG 4
#endif


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


template <int CB, bool kFast>
__device__ __forceinline__ float row_dot(const uint32_t (&w)[CB / 4], uint32_t lanebase,
                                         uint32_t tab_s, uint32_t lane4, const uint32_t (&x16)[CB],
                                         const float2 (&xf)[CB]) {
  if constexpr (kFast) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int wi = 0; wi < CB / 4; ++wi) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t addr = __byte_perm(w[wi], lanebase, 0x7604u | (uint32_t(i) << 4));
        const uint32_t h = lds_u32(addr);
        fma2_f16_f32(h, x16[4 * wi + i], a0, a1);
      }
    }
    return a0 + a1;
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
  // The decoded scales of rows r0 .. r0 + RPG - 1 for this lane's block;
  // rows past the CTA's end read the padding after the scale array (their
  // values are dropped at the store, and the reduction never mixes rows).
  const float* srow = L.sScale + (r0 * spr + L.scol);
  float part[RPG];
#pragma unroll
  for (int r = 0; r < RPG; ++r) {
    const float sum = row_dot<CB, kFast>(st.w[r], L.lanebase, L.tab_s, L.lane4, L.x16, L.xf);
    part[r] = L.act ? __fmul_rn(srow[r * spr], L.xs) * sum : 0.0f;
  }
  const float red = transposed_warp_reduce<RPG>(part, lane);
  if (lane < RPG) {
    const int rr = transposed_index<RPG>(lane);
    if (rr < rows) sPart[(r0 + rr) * W + wg] = red;
  }
}

// The consumer loop of one row group: two steps of RPG rows in flight.
template <int CB, int RPG, bool kFast>
__device__ __forceinline__ void consume(const B1Args& p, const uint8_t* lane_src, uint32_t row_bytes,
                                        Step<CB, RPG>& A, Step<CB, RPG>& B, const Lane<CB>& L,
                                        float* sPart, int wg, int lane, int rg0, int rg1) {
  const int n = rg1 - rg0;
  const int ns = (n + RPG - 1) / RPG;
  auto rows_of = [&](int s) { return (n - s * RPG < RPG) ? n - s * RPG : RPG; };
  auto src_of = [&](int s) { return lane_src + uint32_t(rg0 + s * RPG) * row_bytes; };
  for (int s = 0; s < ns; s += 2) {
    compute_step<CB, RPG, kFast>(A, L, sPart, p.spr, p.W, wg, lane, rg0 + s * RPG, rows_of(s));
    if (s + 2 < ns) load_step<CB, RPG>(A, src_of(s + 2), row_bytes, rows_of(s + 2));
    if (s + 1 < ns) {
      compute_step<CB, RPG, kFast>(B, L, sPart, p.spr, p.W, wg, lane, rg0 + (s + 1) * RPG,
                                   rows_of(s + 1));
      if (s + 3 < ns) load_step<CB, RPG>(B, src_of(s + 3), row_bytes, rows_of(s + 3));
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
  int64_t row_begin, row_end;
  cta_rows(bid, sb.ctas, N, &row_begin, &row_end);
  const int nrows = int(row_end - row_begin);
  const int64_t b0 = (row_begin * K) >> t.lbs;  // first quantization block of the CTA
  const int nq = nrows * p.spr;
  const int64_t g0 = b0 >> t.ls2;
  const int ng = nq > 0 ? int(((b0 + nq - 1) >> t.ls2) - g0 + 1) : 0;
  const uint8_t* slab = t.packed + row_begin * row_bytes;

  // This thread's place among the consumers.
  const int g = int(uint32_t(warp) / uint32_t(p.W));
  const int wg = warp - g * p.W;
  const bool consumer = g < p.G;
  const int c = wg * 32 + lane;
  const bool act = consumer && c < p.cpr;
  const int cc = act ? c : p.cpr - 1;
  const int rg0 = consumer ? group_row0<RPG>(nrows, p.G, g) : 0;
  const int rg1 = consumer ? group_row0<RPG>(nrows, p.G, g + 1) : 0;
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
      for (int q = 0; q < 4; ++q) {  // one packed conversion per pair, checked by converting back
        const float f0 = __fmul_rn(__uint_as_float(w[q] << 16), down);
        const float f1 = __fmul_rn(__uint_as_float(w[q] & 0xffff0000u), down);
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h[q]) : "f"(f1), "f"(f0));  // f0 in the low half
        const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&h[q]));
        ex = ex && (back.x == f0) && (back.y == f1);
      }
      if (pc < npieces) {
        const int ch = pc / kPiecesPerChunk;
        const int within = pc - ch * kPiecesPerChunk;
        *reinterpret_cast<uint4*>(tab + x16_slot(ch, within, p.cpr)) =
            make_uint4(h[0], h[1], h[2], h[3]);
        if (within == 0) sXs[ch] = __uint_as_float(uint32_t(127 + e) << 23);
        x_exact = x_exact && ex;
      }
    }
  }
  // The first two weight steps go out once this thread's small loads have
  // arrived and its x pieces are converted: loads queue per SM, so a small
  // load issued next to a weight stream would wait behind it.
  asm volatile("" ::: "memory");  // keep the weight loads after the stores above
  Step<CB, RPG> A, B;
  const int n_rows = rg1 - rg0;
  const int n_steps = (n_rows + RPG - 1) / RPG;
  auto rows_of = [&](int s) { return (n_rows - s * RPG < RPG) ? n_rows - s * RPG : RPG; };
  const uint32_t rb = uint32_t(row_bytes);
  if (n_steps > 0) load_step<CB, RPG>(A, lane_src + uint32_t(rg0) * rb, rb, rows_of(0));
  if (n_steps > 1) load_step<CB, RPG>(B, lane_src + uint32_t(rg0 + RPG) * rb, rb, rows_of(1));

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
      if (act) v = lds_u128(L.tab_s + x16_slot(cc, q, p.cpr));
      L.x16[4 * q + 0] = v.x;
      L.x16[4 * q + 1] = v.y;
      L.x16[4 * q + 2] = v.z;
      L.x16[4 * q + 3] = v.w;
    }
    consume<CB, RPG, true>(p, lane_src, uint32_t(row_bytes), A, B, L, sPart, wg, lane, rg0, rg1);
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
    consume<CB, RPG, false>(p, lane_src, uint32_t(row_bytes), A, B, L, sPart, wg, lane, rg0, rg1);
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


// Shared memory: the pair table (and the binary16 x in the upper halves of
// its rows) at shared window address 64 KB; the small arrays [code2 | absmax2
// | x scales | absmax_q | scales | partial sums | bias] below it when they
// fit, else above it. The dynamic window starts after the per-block reserved
// shared memory (the kernel has no static shared variables).
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
  p->off_scale = off;  // + one step of padding rows (read for dropped rows)
  off += align_up_u32(uint32_t((max_nq + int64_t(NF4_B1_RPG) * p->spr) * 4), 128);
  p->off_part = off;
  off += align_up_u32(uint32_t(max_rows * W * 4), 128);
  p->off_bias = off;
  if (any_bias(subs, nsub)) off += align_up_u32(uint32_t(max_rows * 4), 128);
  const uint32_t tab = 65536u - uint32_t(res);
  uint32_t base = 0;
  if (!place_small_arrays(off, tab, &base, &plan->smem_bytes)) return false;
  p->off_c2 += base;
  p->off_a2 += base;
  p->off_xs += base;
  p->off_q += base;
  p->off_scale += base;
  p->off_part += base;
  p->off_bias += base;
  p->off_tab = tab;
  return true;
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


}  // namespace nf4
