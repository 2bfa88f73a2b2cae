// nf4_gemv_common.cuh -- pieces shared by the streaming GEMV kernels
// (batch 1 and batches 2..8): grouped-launch planning, ordered small loads,
// warp reductions, register step buffers and shared-memory helpers.
#pragma once

#include "nf4_internal.cuh"

namespace nf4 {
namespace {

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

// True when any weight of a grouped launch has a bias.
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

// First row (relative to the CTA) of row group g: contiguous ranges of whole
// steps of RPG rows, the last groups taking the remainder. The largest group
// has as many steps as in an even split, and the others compute no padding
// rows (an even split of 27 rows over 4 groups computes 32 row slots, this
// one 28). Unsigned 32-bit division (cheaper than signed).
template <int RPG>
__device__ __forceinline__ int group_row0(int nrows, int G, int g) {
  const uint32_t per = ((uint32_t(nrows) + uint32_t(G) - 1u) / uint32_t(G) + RPG - 1) / RPG * RPG;
  const uint32_t r = per * uint32_t(g);
  return r < uint32_t(nrows) ? int(r) : nrows;
}

// Rows [*first, *end) of CTA `bid` of `ctas` over N rows (balanced split),
// in 32-bit unsigned arithmetic whenever ctas * N fits in 32 bits (a 64-bit
// division costs several times as many instructions). The planners' limit of
// 32768 block scales per CTA keeps every launch of these kernels inside the
// 32-bit branch; the 64-bit one is a guard.
__device__ __forceinline__ void cta_rows(int64_t bid, int ctas, int64_t N, int64_t* first,
                                         int64_t* end) {
  if (N <= int64_t(0xffffffffu) / ctas) {
    const uint32_t b = uint32_t(bid), n = uint32_t(N), c = uint32_t(ctas);
    *first = (b * n) / c;
    *end = ((b + 1u) * n) / c;
  } else {
    *first = (bid * N) / ctas;
    *end = ((bid + 1) * N) / ctas;
  }
}

// Shared offset of piece q (16 bytes: 8 binary16 values) of the binary16 x
// chunk c in the upper 128 bytes of the table rows: 16-byte unit
// m = q * cpr + c, eight units per row half. A warp writing consecutive pieces,
// or reading piece q of consecutive chunks, covers whole 128-byte row halves,
// so neither access has bank conflicts (chunk-major units put every even lane
// of a read on the same four banks). K <= 16384 keeps m below 2048.
__device__ __forceinline__ uint32_t x16_slot(int c, int q, int cpr) {
  const uint32_t m = uint32_t(q) * uint32_t(cpr) + uint32_t(c);
  return (m >> 3) * 256u + 128u + (m & 7u) * 16u;
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

// Where the planners put the small per-CTA arrays (code2, scales, partial
// sums, ...; `bytes` in total, offsets counted from 0): below the pair table
// at shared window address 64 KB (`tab` bytes from the start of dynamic
// shared memory) when they fit there, else right above it. Sets the offset
// to add to each array and the dynamic shared memory of the launch.
bool place_small_arrays(uint32_t bytes, uint32_t tab, uint32_t* base, uint32_t* total) {
  *base = bytes <= tab ? 0u : tab + kTabBytes;
  *total = bytes <= tab ? tab + kTabBytes : *base + bytes;
  return *total <= uint32_t(kMaxSmemPerCta);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace nf4
