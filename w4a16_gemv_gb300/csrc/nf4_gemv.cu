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
                                                             const YOut y) {
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
          for (int b = 0; b < B; ++b)
            y_store(y, int64_t(b) * N + row0 + r, acc[r][b], y_bias_bits(y, row0 + r));
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
      if (row0 + r < N) y_store(y, int64_t(b) * N + row0 + r, v, y_bias_bits(y, row0 + r));
    }
  }
}

// Any even K, any power-of-two block size, any element alignment: one warp
// per row, one packed byte per lane step.
template <int B>
__global__ void __launch_bounds__(kThreads) gemv_generic_kernel(QuantTensor t, int64_t N,
                                                                int64_t K,
                                                                const uint16_t* __restrict__ x,
                                                                const YOut y) {
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
      if (lane == 0) y_store(y, int64_t(b) * N + row, v, y_bias_bits(y, row));
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
                              const uint16_t* x, const YOut& y, cudaStream_t stream) {
  static_assert(kTableBytes <= 48 * 1024, "table fits the default dynamic shared memory");
  const int64_t rows_per_cta = int64_t(kWarps / ks) * R;
  const int64_t blocks = (N + rows_per_cta - 1) / rows_per_cta;
  return launch_k(gemv_fast_kernel<B, CB, R>, dim3(unsigned(blocks)), dim3(kThreads), kTableBytes,
                  stream, t, N, K, ks, x, y);
}

// K == 0: every output is an empty sum (plus the bias, if any).
__global__ void zero_fill_kernel(const YOut y, int64_t N, int64_t count) {
  pdl_allow_dependents();
  pdl_wait_prior_grid();
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += int64_t(gridDim.x) * blockDim.x)
    y_store(y, i, 0.0f, y_bias_bits(y, i % N));
}

template <int B>
cudaError_t launch_generic_typed(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x,
                                 const YOut& y, cudaStream_t stream) {
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

template <int B>
cudaError_t dispatch_batch(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x,
                           const YOut& y, cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  if (K == 0) {
    const int64_t count = int64_t(B) * N;
    int64_t blocks = (count + kThreads - 1) / kThreads;
    if (blocks > int64_t(sms) * 8) blocks = int64_t(sms) * 8;
    return launch_k(zero_fill_kernel, dim3(unsigned(blocks)), dim3(kThreads), 0, stream, y, N, count);
  }
  {
    bool done = false;
    const SubTensor one{t, y, N, 0, 0};
    const cudaError_t ek = (B == 1) ? try_gemv_b1(&one, 1, K, x, sms, stream, &done)
                                    : try_gemv_bn(&one, 1, K, x, B, sms, stream, &done);
    if (done || ek != cudaSuccess) return ek;
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
  // the tensor-core GEMV is the only kernel with waits that can run out
  return read_and_clear_tc_flags(flags);
}

cudaError_t launch_gemv(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x, int batch,
                        const YOut& y, cudaStream_t stream) {
  if (batch > 8) {
    if (K > 0) {
      bool done = false;
      const cudaError_t e = try_gemm_tc(t, N, K, x, batch, y, device_sm_count(), stream, &done);
      if (done || e != cudaSuccess) return e;
    }
    // Otherwise slabs of up to eight vectors, one launch each; after the
    // first slab the weights come from L2.
    const size_t esize = y.dtype == NF4_F32 ? 4 : 2;
    for (int b0 = 0; b0 < batch; b0 += 8) {
      const int nb = batch - b0 < 8 ? batch - b0 : 8;
      YOut ys = y;
      ys.y = static_cast<unsigned char*>(y.y) + size_t(b0) * size_t(N) * esize;
      const cudaError_t e =
          launch_gemv(t, N, K, x == nullptr ? nullptr : x + int64_t(b0) * K, nb, ys, stream);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
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

cudaError_t launch_gemv_group(const QuantTensor* ts, const int64_t* Ns, const YOut* outs, int n,
                              int64_t K, const uint16_t* x, int batch, cudaStream_t stream,
                              bool* done) {
  *done = false;
  if (n < 1 || n > kMaxSub || K <= 0 || batch < 1 || batch > 8) return cudaSuccess;
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  SubTensor subs[kMaxSub];
  for (int j = 0; j < n; ++j) subs[j] = SubTensor{ts[j], outs[j], Ns[j], 0, 0};
  return batch == 1 ? try_gemv_b1(subs, n, K, x, sms, stream, done)
                    : try_gemv_bn(subs, n, K, x, batch, sms, stream, done);
}

}  // namespace nf4
