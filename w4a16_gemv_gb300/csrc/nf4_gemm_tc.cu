// nf4_gemm_tc.cu -- the fused GEMV for wide batches (9..64 vectors) on the
// 5th-generation tensor cores: y = W_hat x with the dequantization fused.
//
// At these batches the contraction is dense ("CUDA 进阶手册 / 量化与 GEMV",
// exercise on batch 1/4/32/128: past a few vectors the weights are reused
// enough that the W4A16 path moves to FP16 tensor cores); CUDA-core FMAs
// would make it compute-bound. Per CTA, a tile of 128 weight rows:
//   * the stage's packed weight tile (128 rows x 32 bytes) and x tile go
//     through 8-deep rings in shared memory filled by 2-D tensor copies (TMA;
//     x 128-byte swizzled; rows past the weight or the batch zero-filled)
//     that complete on mbarriers;
//   * sixteen producer warps dequantize in registers: w_hat = fp32(NF4[idx] *
//     s) exactly as the dequantization defines it, split into bfloat16 hi =
//     rn(w_hat) and lo = rn(w_hat - hi) (the residual is exact, so w_hat is
//     represented to about 2^-17 relative), and store both into tensor memory
//     (TMEM lane = weight row) -- the A operand never touches shared memory;
//   * x stays bfloat16 (exact) in shared memory as the B operand, 128-byte
//     swizzled, K-major;
//   * one warp issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32 in TMEM),
//     two per 16-element K step (hi and lo), once the producer warps have
//     signalled the stage's A buffer full; its commit frees the A buffer and
//     the ring slot, which another warp refills with the tile copies. The
//     producers run up to four stages ahead of the MMAs (four A buffers in
//     TMEM);
//   * K is split over a thread-block cluster; each CTA pushes its partial
//     sums into the shared memory of the rank that owns the rows, which adds
//     them in rank order (deterministic) and applies the output stage (bias,
//     rounding to y's type) once. When one CTA per tile would leave many SMs
//     idle, a cluster of three CTAs covers a pair of tiles instead.
// Every wait on an mbarrier is bounded (about one second); a wait that runs
// out sets bit 0 of the device error flags, and the kernel still completes
// its cluster barriers, waits (with the same bound) for its own copies and
// MMAs still in flight, frees its tensor memory and exits. That path reports
// a hang rather than recovering from it: the launch's results are undefined,
// and a copy or MMA that never completes within the second wait may still be
// in flight when the CTA exits. The limit is long enough that only a real
// hang reaches it.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "nf4_internal.cuh"

namespace nf4 {
namespace {

constexpr int kProducerWarps = 16;  // warp w < 16: rows 32 * (w % 4) + lane, K quarter w / 4
constexpr int kMmaWarp = kProducerWarps;       // issues the MMAs
constexpr int kCopyWarp = kProducerWarps + 1;  // starts the tile copies
constexpr int kTcThreads = 32 * (kProducerWarps + 2);
constexpr int kTileM = 128;
constexpr int kStageK = 64;      // elements of K per stage
constexpr int kRing = 8;         // stages of packed weights and x in shared memory
constexpr int kAhead = kRing - 2;  // stages loaded ahead of the one being dequantized
constexpr int kLongStages = 64;  // stages per CTA above which K is split further
constexpr int kNA = 4;               // A buffers in TMEM (the producers' lead over the MMAs)
constexpr uint32_t kTmemCols = 512;  // A: kNA x 64 columns (hi 32 + lo 32); D: from 256, BN (x 2 for a pair)

__device__ unsigned int g_tc_flags = 0;  // bit 0: an mbarrier wait ran out

struct TcArgs {
  QuantTensor t;
  YOut out;
  const uint16_t* x;
  int64_t N;
  int32_t K;
  int batch;
  int splits;  // CTAs per cluster (1, 2, 4 or 8 along K of one tile; 3 for a tile pair)
  int pair;    // 1: a cluster of 3 CTAs covers two tiles (see the kernel)
  uint32_t off_b, off_w, off_recv, off_tab, off_c2, off_bar;
};


__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the leading-byte offset is not used by this layout).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M = 128, N = bn.
__host__ __device__ constexpr uint32_t idesc_bf16(int bn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(bn >> 3) << 17) | (uint32_t(kTileM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Packed binary32 multiply and subtract (two independent IEEE operations,
// round to nearest).
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
__device__ __forceinline__ float2 fsub2_rn(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_rn(float2 v) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(v.y), "f"(v.x));  // element 0 low
  return r;
}
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

template <int BN>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const TcArgs p, const __grid_constant__ CUtensorMap tmx,
                   const __grid_constant__ CUtensorMap tmw) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // tile copies and the swizzled x layout want a 1024-byte aligned base (the
  // host allocates 1024 bytes of slack)
  unsigned char* const smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int kq = warp >> 2;                 // K quarter of a stage (16 elements)
  const int row = (warp & 3) * 32 + lane;   // row of the tile = TMEM lane
  const int cl = int(blockIdx.x) / p.splits;
  const int split = int(blockIdx.x) - cl * p.splits;  // rank in the cluster
  const QuantTensor& t = p.t;
  const int64_t K = p.K;
  const int S = int(K / kStageK);
  // The CTA's work is a range of consecutive (tile, stage) units: split
  // `split` of the stages of tile `cl`, or, for a tile pair, a third of the
  // 2S units of tiles 2 cl and 2 cl + 1. Its units i < ib are stages s0 + i
  // of tile `tile`; units i >= ib (the middle rank of a pair only) are
  // stages i - ib of tile + 1.
  int tile, s0, ns, ib;
  if (p.pair) {
    const int u0 = int(int64_t(split) * 2 * S / 3), u1 = int(int64_t(split + 1) * 2 * S / 3);
    tile = 2 * cl + (u0 >= S ? 1 : 0);
    s0 = u0 >= S ? u0 - S : u0;
    ns = u1 - u0;
    ib = (u0 < S && u1 > S) ? S - u0 : ns;
  } else {
    tile = cl;
    s0 = int(int64_t(split) * S / p.splits);
    ns = int(int64_t(split + 1) * S / p.splits) - s0;
    ib = ns;
  }
  const int64_t r_glob = int64_t(tile) * kTileM + row;
  const bool row_ok = r_glob < p.N;
  const bool row_ok_b = r_glob + kTileM < p.N;  // the same row of the second tile

  const uint32_t sbase = smem_u32(smem);
  const uint32_t b_ring = sbase + p.off_b;                    // kRing slots of BN x 128 B
  const uint32_t w_ring = sbase + p.off_w;                    // kRing slots of 4 KB
  // partial sums received from peers: [src rank][BN][128 / splits] along K,
  // [BN][128] from the middle rank of a tile pair
  float* recv = reinterpret_cast<float*>(smem + p.off_recv);
  float* sC2 = reinterpret_cast<float*>(smem + p.off_c2);
  uint64_t* afull = reinterpret_cast<uint64_t*>(smem + p.off_bar);  // A buffer written (16 warps)
  uint64_t* mdone = afull + kNA;  // MMAs of a stage done (frees its A buffer and ring slot), per slot
  uint64_t* full = mdone + kRing;  // weight and x tiles landed, per slot
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(smem + p.off_bar + 8 * (kNA + 2 * kRing));

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(s_taddr)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int i = 0; i < kNA; ++i) mbar_init(&afull[i], kProducerWarps);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&mdone[i], 1);
      mbar_init(&full[i], 1);
    }
    fence_mbar_init();
  }
  // Programmatic dependent launch: the next kernel may be scheduled now; this
  // one reads no global memory before the grid-dependency wait below (TMEM,
  // barriers and the pair table need none).
  pdl_allow_dependents();

  // Lane-private pair table: row e (256 B) holds (NF4[e >> 4], NF4[e & 15])
  // for lane l at bytes 8l..8l+7 (no bank conflicts).
  {
    const float my_code = nf4_code_select(lane & 15);
    unsigned char* tabp = smem + p.off_tab;
    for (int i = tid; i < 256 * 16; i += kTcThreads) {
      const int e = i >> 4, q = i & 15;
      const float hi = __shfl_sync(0xffffffffu, my_code, e >> 4);
      const float lo = __shfl_sync(0xffffffffu, my_code, e & 15);
      *reinterpret_cast<float4*>(tabp + e * 256 + q * 16) = make_float4(hi, lo, hi, lo);
    }
  }

  // Waits until the MMAs of stage j (and every earlier stage) are done: the
  // commit of stage j arrives on mdone[j % kRing]; a barrier is reused only
  // after every waiter of its previous phase has passed.
  auto wait_mma_done = [&](int j) {
    return mbar_wait_bounded(&mdone[j % kRing], uint32_t((j / kRing) & 1), kWaitLimitCycles);
  };
  const bool producer = warp < kProducerWarps;
  // Small inputs first (their latency hides behind the table build): the
  // code2 entry of this thread, and the block-scale inputs (absmax_q,
  // absmax2) of this row for the first kNA stages; a producer loads those of
  // stages kNA .. kRing - 1 during its first kNA stages, and those of stage
  // i + kRing at stage i, into the registers stage i used (the loop is
  // unrolled over the ring, so no register is copied while its load is in
  // flight).
  pdl_wait_prior_grid();
  const uint16_t c2v = tid < 256 ? __ldg(t.code2 + tid) : uint16_t(0);
  auto load_scale_in = [&](int i, uint32_t& q, uint32_t& a2) {
    q = 0u;
    a2 = 0u;
    const bool second = i >= ib;
    if (producer && i < ns && (second ? row_ok_b : row_ok)) {
      const int64_t e = second ? (r_glob + kTileM) * K + int64_t(i - ib) * kStageK
                               : r_glob * K + int64_t(s0 + i) * kStageK;
      const int64_t blk = e >> t.lbs;
      q = __ldg(t.absmax_q + blk);
      a2 = __ldg(t.absmax2 + (blk >> t.ls2));
    }
  };
  uint32_t qv[kRing], av[kRing];
#pragma unroll
  for (int u = 0; u < kNA; ++u) load_scale_in(u, qv[u], av[u]);
  // The weight and x tiles of stage i into ring slot i % kRing (thread
  // kTcThreads - 32 only).
  auto issue_tiles = [&](int i) {
    const int slot = i % kRing;
    const bool second = i >= ib;
    const int st = second ? i - ib : s0 + i;  // stage within its tile
    mbar_arrive_expect_tx(&full[slot], uint32_t(kTileM * kStageK / 2 + BN * 128));
    tma_load_2d(w_ring + uint32_t(slot) * 4096u, &tmw, st * (kStageK / 2), (tile + (second ? 1 : 0)) * kTileM,
                &full[slot]);
    tma_load_2d(b_ring + uint32_t(slot) * uint32_t(BN * 128), &tmx, st * kStageK, 0, &full[slot]);
  };

  __syncthreads();  // barriers initialised before any copy uses one
  // First phase of the cluster barrier: this CTA is running (its shared
  // memory may receive the peers' partial sums once the phase completes).
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (warp == kCopyWarp && lane == 0)
    for (int i = 0; i < kAhead && i < ns; ++i) issue_tiles(i);

  if (tid < 256) sC2[tid] = half_bits_to_float(c2v);

  tc_fence_before();
  __syncthreads();  // pair table, sC2 and the TMEM address ready
  tc_fence_after();
  const uint32_t tbase = *s_taddr;
  const uint32_t lane_base = tbase + (uint32_t((warp & 3) * 32) << 16);
  const uint32_t d_col = tbase + 64u * kNA;
  const uint32_t tab_lane = sbase + p.off_tab + (uint32_t(lane) << 3);
  constexpr uint32_t kIdesc = idesc_bf16(BN);
  bool ok = true;

  if (producer) {
#pragma unroll 1
    for (int i0 = 0; i0 < ns; i0 += kRing) {
      const uint32_t ph = uint32_t(i0 / kRing) & 1u;  // ring phase of stages i0 .. i0 + kRing - 1
#pragma unroll
      for (int u = 0; u < kRing; ++u) {  // stage i0 + u: ring slot u, A buffer u % kNA
        const int i = i0 + u;
        if (i < ns) {
          if (i >= kNA) {  // the MMAs of stage i - kNA (slot (u - kNA) mod kRing) have read A buffer u % kNA
            const uint32_t ph_prev = u >= kNA ? ph : ph ^ 1u;
            ok = mbar_wait_bounded(&mdone[(u + kRing - kNA) % kRing], ph_prev, kWaitLimitCycles) && ok;
            tc_fence_after();
          }
          // both tiles of the stage landed (the MMAs of the stage read the x
          // tile after this wait, through the A-buffer barrier)
          ok = mbar_wait_bounded(&full[u], ph, kWaitLimitCycles) && ok;

          // block scale fp32(fp32(code2[q] * absmax2[g]) + offset); 0 past the last row
          const float sc = (i >= ib ? row_ok_b : row_ok)
                               ? __fadd_rn(__fmul_rn(sC2[qv[u]], half_bits_to_float(uint16_t(av[u]))), t.offset)
                               : 0.0f;
          load_scale_in(i + kRing, qv[u], av[u]);
          if (u < kRing - kNA && i0 == 0) load_scale_in(u + kNA, qv[u + kNA], av[u + kNA]);
          const float2 sc2 = make_float2(sc, sc);
          // dequantize 16 elements (8 packed bytes) of this row: w_hat = fp32(NF4
          // code * s), split into bfloat16 hi + lo
          uint32_t wd0, wd1;
          asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];"
                       : "=r"(wd0), "=r"(wd1)
                       : "r"(w_ring + uint32_t(u) * 4096u + uint32_t(row) * 32u + uint32_t(kq) * 8u));
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const uint32_t word = b < 4 ? wd0 : wd1;
            const uint32_t addr = tab_lane + (__byte_perm(word, 0u, 0x4440u + uint32_t(b & 3)) << 8);
            float2 c;
            asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(c.x), "=f"(c.y) : "r"(addr));
            const float2 w = fmul2_rn(c, sc2);
            hi[b] = bf16x2_rn(w);
            lo[b] = bf16x2_rn(fsub2_rn(w, bf16x2_to_f2(hi[b])));  // exact residual
          }
          const uint32_t acol = lane_base + uint32_t(u % kNA) * 64u + uint32_t(kq) * 8u;
          tmem_st8(acol, hi);
          tmem_st8(acol + 32u, lo);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&afull[u % kNA]);
        }
      }
    }
  } else if (warp == kMmaWarp && lane == 0) {
    // MMA issue. One thread, sharing its scheduler with producer warps: the
    // per-stage instruction stream is kept short (the loop is unrolled over
    // the ring, so slots, A buffers and phases are compile-time constants;
    // the x-tile descriptor of a slot and K step is the slot-0 descriptor
    // plus a constant in its 16-byte address field). One wait per stage: the
    // producers signal the A buffer only after the stage's tiles landed.
    const uint64_t desc0 = desc_sw128(b_ring);
    constexpr uint32_t kSlotUnits = uint32_t(BN * 128) >> 4;
    static_assert(kRing % kNA == 0, "ring slots and A buffers advance together");
#pragma unroll 1
    for (int i0 = 0; i0 < ns; i0 += kRing) {
      const uint32_t a_ph0 = uint32_t(i0 / kNA) & 1u;
#pragma unroll
      for (int u = 0; u < kRing; ++u) {  // stage i0 + u: slot u, A buffer u % kNA
        if (i0 + u < ns) {
          ok = mbar_wait_bounded(&afull[u % kNA], a_ph0 ^ uint32_t((u / kNA) & 1), kWaitLimitCycles) && ok;
          tc_fence_after();
          const uint32_t a_t = tbase + uint32_t(u % kNA) * 64u;
          const uint64_t bd = desc0 + uint64_t(u * kSlotUnits);
          // the second tile's units accumulate into their own columns
          const int i = i0 + u;
          const uint32_t dc = d_col + (i >= ib ? uint32_t(BN) : 0u);
          mma_bf16(dc, a_t, bd, kIdesc, (i > 0 && i != ib) ? 1u : 0u);
          mma_bf16(dc, a_t + 32u, bd, kIdesc, 1u);
#pragma unroll
          for (int j = 1; j < kStageK / 16; ++j) {  // 32 bytes of K per step
            mma_bf16(dc, a_t + 8u * uint32_t(j), bd + uint64_t(2 * j), kIdesc, 1u);
            mma_bf16(dc, a_t + 32u + 8u * uint32_t(j), bd + uint64_t(2 * j), kIdesc, 1u);
          }
          tc_commit(&mdone[u]);  // frees A buffer u % kNA and ring slot u
        }
      }
    }
  } else if (warp == kCopyWarp && lane == 0) {
    // Tile copies of stage nx into the slot of stage nx - kRing once that
    // stage's MMAs are done (its weight tile was consumed before the
    // producers signalled it).
#pragma unroll 1
    for (int nx = kAhead; nx < ns; ++nx) {
      if (nx >= kRing)
        ok = wait_mma_done(nx - kRing) && ok;
      issue_tiles(nx);
    }
  }
  __syncwarp();
  // all MMAs done (the last commit covers every earlier one)
  if (ns > 0)
    ok = wait_mma_done(ns - 1) && ok;
  tc_fence_after();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every peer is running

  if (p.pair) {
    // Tile pair: rank 0 owns tile 2 cl, rank 2 owns tile 2 cl + 1; the
    // middle rank pushes its partial sums of both tiles (its two
    // accumulators) into the owners' receive buffers, laid out [BN][128].
    // After one cluster barrier each owner adds its own accumulator (two
    // terms, so the order of the operands does not matter) and applies the
    // output stage. Warp (row quarter, K quarter kq) handles columns
    // [kq * BN / 4, (kq + 1) * BN / 4) of its lanes' rows.
    if (split == 1 && producer) {
#pragma unroll
      for (int seg = 0; seg < 2; ++seg) {
        uint32_t dst = smem_u32(recv) + uint32_t(row) * 4u;
        asm volatile("mapa.shared::cluster.u32 %0, %0, %1;" : "+r"(dst) : "r"(uint32_t(seg == 0 ? 0 : 2)));
        uint32_t v[BN / 4];
#pragma unroll
        for (int c0 = 0; c0 < BN / 4; c0 += 4) {
          uint32_t w4[4];
          tmem_ld4(lane_base + 64u * kNA + uint32_t(seg * BN + kq * (BN / 4) + c0), w4);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) v[c0 + jj] = w4[jj];
        }
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int jj = 0; jj < BN / 4; ++jj) asm volatile("" : "+r"(v[jj]));  // uses follow the wait
#pragma unroll
        for (int jj = 0; jj < BN / 4; ++jj) {
          const int n = kq * (BN / 4) + jj;
          const float f = ok ? __uint_as_float(v[jj]) : __uint_as_float(0x7fc00000u);
          asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst + uint32_t(n * kTileM) * 4u), "f"(f)
                       : "memory");
        }
      }
    }
    if (!ok) atomicOr(&g_tc_flags, 1u);
    cluster_sync();  // the middle rank's pushes have landed
    if (split != 1 && producer) {
      uint32_t v[BN / 4];
#pragma unroll
      for (int c0 = 0; c0 < BN / 4; c0 += 4) {
        uint32_t w4[4];
        tmem_ld4(lane_base + 64u * kNA + uint32_t(kq * (BN / 4) + c0), w4);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) v[c0 + jj] = w4[jj];
      }
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
      for (int jj = 0; jj < BN / 4; ++jj) asm volatile("" : "+r"(v[jj]));  // uses follow the wait
      if (row_ok) {
        const uint32_t bias_bits = y_bias_bits(p.out, r_glob);
#pragma unroll
        for (int jj = 0; jj < BN / 4; ++jj) {
          const int n = kq * (BN / 4) + jj;
          if (n < p.batch) {
            const float own = ok ? __uint_as_float(v[jj]) : __uint_as_float(0x7fc00000u);
            y_store(p.out, int64_t(n) * p.N + r_glob, own + recv[n * kTileM + row], bias_bits);
          }
        }
      }
    }
  } else {
    // Split-K: the CTA owning rows [rank * R, (rank + 1) * R) of the tile (R
    // = 128 / splits) receives every rank's partial sums of those rows in its
    // own receive buffer (not used before, so peers may write as soon as their
    // MMAs are done); warp (row quarter, K quarter kq) pushes columns
    // [kq * BN / 4, (kq + 1) * BN / 4) of its lanes' rows.
    const int rows_per = kTileM / p.splits;
    {
      const int owner = row / rows_per;
      const int rl = row - owner * rows_per;
      uint32_t dst = smem_u32(recv) + uint32_t((split * BN) * rows_per + rl) * 4u;
      asm volatile("mapa.shared::cluster.u32 %0, %0, %1;" : "+r"(dst) : "r"(uint32_t(owner)));
      if (producer) {
        // all BN / 4 columns of this warp's quarter, then one wait
        uint32_t v[BN / 4];
  #pragma unroll
        for (int c0 = 0; c0 < BN / 4; c0 += 4) {
          uint32_t w4[4];
          tmem_ld4(lane_base + 64u * kNA + uint32_t(kq * (BN / 4) + c0), w4);
  #pragma unroll
          for (int j = 0; j < 4; ++j) v[c0 + j] = w4[j];
        }
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  #pragma unroll
        for (int j = 0; j < BN / 4; ++j) asm volatile("" : "+r"(v[j]));  // uses follow the wait
  #pragma unroll
        for (int j = 0; j < BN / 4; ++j) {
          const int n = kq * (BN / 4) + j;
          const float f = ok ? __uint_as_float(v[j]) : __uint_as_float(0x7fc00000u);
          asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst + uint32_t(n * rows_per) * 4u), "f"(f)
                       : "memory");
        }
      }
    }
    if (!ok) atomicOr(&g_tc_flags, 1u);
    cluster_sync();  // every rank's pushes have landed

    // Rows [split * R, (split + 1) * R): the sum over ranks in rank order,
    // then the output stage.
    const int lrp = 31 - __clz(rows_per);  // rows_per is a power of two
    const int total = rows_per * p.batch;
    const int64_t rg0 = int64_t(tile) * kTileM + split * rows_per;
    for (int e = tid; e < total; e += kTcThreads) {
      const int b = e >> lrp;
      const int rl = e & (rows_per - 1);
      const int64_t rg = rg0 + rl;
      const float* src = recv + b * rows_per + rl;
      float v = src[0];
  #pragma unroll
      for (int q = 1; q < 8; ++q)
        if (q < p.splits) v += src[q * BN * rows_per];
      if (rg < p.N) y_store(p.out, int64_t(b) * p.N + rg, v, y_bias_bits(p.out, rg));
    }
  }

  // After a wait that ran out, copies or MMAs of this CTA may still be in
  // flight: wait for them (with the same bound) before the tensor memory is
  // freed and the shared memory released. The last commit covers every
  // earlier MMA; a ring slot's last copy is the one of the last stage using it.
  if (__syncthreads_or(!ok) && warp == kCopyWarp && lane == 0) {
    if (ns > 0) wait_mma_done(ns - 1);
    for (int st = ns > kRing ? ns - kRing : 0; st < ns; ++st)
      mbar_wait_bounded(&full[st % kRing], uint32_t((st / kRing) & 1), kWaitLimitCycles);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemCols)
                 : "memory");
  }
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  // initialised once, thread-safely (function-local static)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return PFN_cuTensorMapEncodeTiled_v12000(nullptr);
  }();
  return fn;
}

template <int BN>
cudaError_t launch_tc(const TcArgs& a, const CUtensorMap& tmx, const CUtensorMap& tmw, int grid,
                      uint32_t smem, cudaStream_t stream) {
  auto kern = gemm_tc_kernel<BN>;
  static PerDeviceCache attr_set;
  const cudaError_t e = set_max_dynamic_smem_once(kern, 227 * 1024, attr_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned(kTcThreads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(a.splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = NF4_USE_PDL ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a, tmx, tmw);
}

}  // namespace

cudaError_t try_gemm_tc(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x, int batch,
                        const YOut& out, int sms, cudaStream_t stream, bool* done) {
  *done = false;
  if (batch < 9 || batch > 64 || N <= 0 || K <= 0 || K % kStageK != 0) return cudaSuccess;
  if (K > (int64_t(1) << 30)) return cudaSuccess;  // K and stage coordinates stay in 32 bits
  if (t.lbs < 6 || (K & ((int64_t(1) << t.lbs) - 1)) != 0) return cudaSuccess;  // blocksize >= 64, rows whole blocks
  if ((reinterpret_cast<uintptr_t>(t.packed) & 15u) != 0 || (reinterpret_cast<uintptr_t>(x) & 15u) != 0)
    return cudaSuccess;
  const int BN = (batch + 15) / 16 * 16;
  const int64_t tiles = (N + kTileM - 1) / kTileM;
  const int S = int(K / kStageK);
  if (tiles > (int64_t(1) << 24)) return cudaSuccess;
  // K split over a cluster of up to 8: fill the SMs, keep at least 4 stages
  // per CTA, and split long rows (more than 64 stages, 4096 elements).
  int splits = 1;
  while (splits < 8 && (S + splits - 1) / splits > kLongStages) splits *= 2;
  while (splits < 8 && tiles * splits * 2 <= sms && S / (splits * 2) >= 4) splits *= 2;
  // One CTA per tile leaving more than a third of the SMs idle: clusters of
  // three CTAs over pairs of tiles (two thirds of a tile's stages each).
  const bool pair = splits == 1 && tiles % 2 == 0 && tiles * 3 / 2 <= sms && tiles * 3 < int64_t(sms) * 2 &&
                    S >= 6;
  const int grid = pair ? int(tiles / 2) * 3 : int(tiles) * splits;

  TcArgs a;
  a.t = t;
  a.out = out;
  a.x = x;
  a.N = N;
  a.K = int32_t(K);
  a.batch = batch;
  a.splits = pair ? 3 : splits;
  a.pair = pair ? 1 : 0;
  // Shared memory, from a 1024-aligned base: [weight ring | code2 |
  // barriers | pair table | x ring | split-K receive buffer].
  a.off_w = 0;
  a.off_c2 = uint32_t(kRing * 4096);
  a.off_bar = a.off_c2 + 1024u;
  a.off_tab = a.off_bar + 512u;
  a.off_b = (a.off_tab + 256u * 256u + 1023u) & ~1023u;
  a.off_recv = a.off_b + uint32_t(kRing * BN * 128);  // receive buffer of the split-K sums
  const uint32_t off = a.off_recv + uint32_t(BN * kTileM * 4) + 1024u;  // + slack
  if (off > 227u * 1024u) return cudaSuccess;
  // x as a 2-D tensor (K contiguous, `batch` rows) for the tile copies: box
  // 64 elements (128 bytes, the swizzle span) x BN rows; rows past the batch
  // read as zero.
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaSuccess;
  CUtensorMap tmx;
  const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(batch)};
  const cuuint64_t strides[1] = {cuuint64_t(K) * 2u};
  const cuuint32_t box[2] = {cuuint32_t(kStageK), cuuint32_t(BN)};
  const cuuint32_t estr[2] = {1u, 1u};
  if (encode(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaSuccess;
  // packed weights as a 2-D byte tensor (K / 2 bytes per row, N rows): box
  // 32 bytes x 128 rows; rows past N read as zero
  CUtensorMap tmw;
  const cuuint64_t wdims[2] = {cuuint64_t(K / 2), cuuint64_t(N)};
  const cuuint64_t wstrides[1] = {cuuint64_t(K / 2)};
  const cuuint32_t wbox[2] = {cuuint32_t(kStageK / 2), cuuint32_t(kTileM)};
  if (encode(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(t.packed), wdims, wstrides,
             wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaSuccess;
  *done = true;
  switch (BN) {
    case 16: return launch_tc<16>(a, tmx, tmw, grid, off, stream);
    case 32: return launch_tc<32>(a, tmx, tmw, grid, off, stream);
    case 48: return launch_tc<48>(a, tmx, tmw, grid, off, stream);
    default: return launch_tc<64>(a, tmx, tmw, grid, off, stream);
  }
}

cudaError_t read_and_clear_tc_flags(unsigned int* flags) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flags, g_tc_flags, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_tc_flags, &zero, sizeof(unsigned int));
}

}  // namespace nf4
