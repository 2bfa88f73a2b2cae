// nf4_gemv_stream.cu -- batch 2..8 decode GEMV y = W_hat x with the NF4
// double-quant dequantization fused, for sm_103a (CUDA cores).
//
// What is computed follows "RTX 4060 上的 LLM 量化实测：4-bit decode 比 FP16 慢在
// 哪里", section "Fused kernel：把反量化搬到片上" (packed codes read once,
// decoded and accumulated on chip, only y written) with the scale formula of
// "NF4 双重量化反量化 CUDA Kernel 实现报告", section 1.3. The work split is the
// k-stationary transpose of the warp-per-row GEMV in "CUDA 进阶手册 / 量化与
// GEMV", section "GEMV kernel 的写法": each thread owns one column chunk of
// every row, so x is read once per CTA and kept in registers.
#include "nf4_gemv_common.cuh"

namespace nf4 {
namespace {

// ---------------------------------------------------------------------------
// Batch 2..8. k-stationary like batch 1, with direct weight loads into
// registers (RPG rows per step, three steps in flight, four on 256 threads)
// instead of a copy ring, and x kept in
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
// sPart[warp * pstride + row * BP + vector] (warp-major: the lanes storing a
// step's partials, and the threads summing a slot over the warps, touch
// consecutive words).
template <int BP, int CB, int RPG>
__device__ __forceinline__ void compute_step_n(const Step<CB, RPG>& st, const LaneN<BP, CB>& L,
                                               const float* sScale, float* sPart, int spr, int pstride,
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
      float* d = sPart + wg * pstride + (r0 + r) * BP + b;
      *d = first ? red : *d + red;
    }
  }
}

template <int BP, int CB, int RPG>
__device__ __forceinline__ void consume_n(const uint8_t* lane_src, uint32_t row_bytes,
                                          Step<CB, RPG>& A, Step<CB, RPG>& B, Step<CB, RPG>& C,
                                          const LaneN<BP, CB>& L, const float* sScale, float* sPart,
                                          int spr, int pstride, int wg, int lane, int rg0, int rg1,
                                          bool first) {
  const int n = rg1 - rg0;
  const int ns = (n + RPG - 1) / RPG;
  auto rows_of = [&](int s) { return (n - s * RPG < RPG) ? n - s * RPG : RPG; };
  auto src_of = [&](int s) { return lane_src + uint32_t(rg0 + s * RPG) * row_bytes; };
  for (int s = 0; s < ns; s += 3) {
    compute_step_n<BP, CB, RPG>(A, L, sScale, sPart, spr, pstride, wg, lane, rg0 + s * RPG, rows_of(s), first);
    if (s + 3 < ns) load_step<CB, RPG>(A, src_of(s + 3), row_bytes, rows_of(s + 3));
    if (s + 1 < ns) {
      compute_step_n<BP, CB, RPG>(B, L, sScale, sPart, spr, pstride, wg, lane, rg0 + (s + 1) * RPG,
                                  rows_of(s + 1), first);
      if (s + 4 < ns) load_step<CB, RPG>(B, src_of(s + 4), row_bytes, rows_of(s + 4));
    }
    if (s + 2 < ns) {
      compute_step_n<BP, CB, RPG>(C, L, sScale, sPart, spr, pstride, wg, lane, rg0 + (s + 2) * RPG,
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
                                           const float* sScale, float* sPart, int spr, int pstride, int wg,
                                           int lane, int rg0, int rg1, bool first) {
  const int n = rg1 - rg0;
  const int ns = (n + RPG - 1) / RPG;
  auto rows_of = [&](int s) { return (n - s * RPG < RPG) ? n - s * RPG : RPG; };
  auto src_of = [&](int s) { return lane_src + uint32_t(rg0 + s * RPG) * row_bytes; };
  for (int s = 0; s < ns; s += 4) {
    compute_step_n<BP, CB, RPG>(A, L, sScale, sPart, spr, pstride, wg, lane, rg0 + s * RPG, rows_of(s), first);
    if (s + 4 < ns) load_step<CB, RPG>(A, src_of(s + 4), row_bytes, rows_of(s + 4));
    if (s + 1 < ns) {
      compute_step_n<BP, CB, RPG>(B, L, sScale, sPart, spr, pstride, wg, lane, rg0 + (s + 1) * RPG,
                                  rows_of(s + 1), first);
      if (s + 5 < ns) load_step<CB, RPG>(B, src_of(s + 5), row_bytes, rows_of(s + 5));
    }
    if (s + 2 < ns) {
      compute_step_n<BP, CB, RPG>(C, L, sScale, sPart, spr, pstride, wg, lane, rg0 + (s + 2) * RPG,
                                  rows_of(s + 2), first);
      if (s + 6 < ns) load_step<CB, RPG>(C, src_of(s + 6), row_bytes, rows_of(s + 6));
    }
    if (s + 3 < ns) {
      compute_step_n<BP, CB, RPG>(D, L, sScale, sPart, spr, pstride, wg, lane, rg0 + (s + 3) * RPG,
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
  int64_t row_begin, row_end;
  cta_rows(bid, sb.ctas, N, &row_begin, &row_end);
  const int nrows = int(row_end - row_begin);
  const int pstride = nrows * BP;  // partial-sum slots of one warp
  const int64_t b0 = (row_begin * K) >> t.lbs;
  const int nq = nrows * p.spr;
  const int64_t g0 = b0 >> t.ls2;
  const int ng = nq > 0 ? int(((b0 + nq - 1) >> t.ls2) - g0 + 1) : 0;
  const uint8_t* slab = t.packed + row_begin * row_bytes;

  const int g = int(uint32_t(warp) / uint32_t(p.W));
  const int wg = warp - g * p.W;
  const bool consumer = g < p.G;
  const int rg0 = consumer ? group_row0<RPG>(nrows, p.G, g) : 0;
  const int rg1 = consumer ? group_row0<RPG>(nrows, p.G, g + 1) : 0;
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
      consume_n4<BP, CB, RPG>(lane_src, rb, A, B, C, D, L, sScale, sPart, p.spr, pstride, wg, lane, rg0,
                              rg1, sl == 0);
    else
      consume_n<BP, CB, RPG>(lane_src, rb, A, B, C, L, sScale, sPart, p.spr, pstride, wg, lane, rg0, rg1,
                             sl == 0);
  }

  // End of the group: one sum per (row, vector) over the group's warps.
  named_barrier(1 + g, p.W * 32);
  const int gt = tid - g * p.W * 32;
  for (int idx = gt; idx < n_rows * BP; idx += p.W * 32) {
    const int r = rg0 + idx / BP, b = idx - (idx / BP) * BP;
    if (b >= p.batch) continue;
    float v = 0.0f;
    for (int w = 0; w < p.W; ++w) v += sPart[w * pstride + r * BP + b];
    y_store(sb.out, int64_t(b) * N + row_begin + r, v, has_bias ? sBias[r] : 0u);
  }
}

// Plan for BP vectors, CB-byte chunks and nt threads (one CTA per SM): the
// binary32 pair table at shared window address 64 KB, the small arrays
// [code2 | absmax2 | absmax_q | scales | partial sums | bias] below it when
// they fit, else above it.
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
  uint32_t base = 0;
  if (!place_small_arrays(off, tab, &base, smem_bytes)) return false;
  p->off_c2 += base;
  p->off_a2 += base;
  p->off_q += base;
  p->off_scale += base;
  p->off_part += base;
  p->off_bias += base;
  p->off_tab = tab;
  return true;
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
}  // namespace

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
