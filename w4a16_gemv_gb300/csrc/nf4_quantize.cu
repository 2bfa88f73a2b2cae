// nf4_quantize.cu -- NF4 quantization with double quantization on sm_103a.
//
// First level ("NF4反量化算子优化", section "双量化 / 第一层量化"): flatten,
// blocks of `blocksize`, absmax per block, divide, nearest NF4 code, two codes
// per byte (even element in the high nibble). Second level (same section,
// "第二层量化", and "NF4 双重量化反量化 CUDA Kernel 实现报告", section 1.2):
// offset = mean of the block absmax values, absmax2 = binary16 max
// |absmax - offset| per group of `s2_blocksize` blocks, absmax_q = nearest
// code2 index of (absmax - offset) / absmax2.
//
// The decisions that pick an integer (code indices) are taken in the same
// precision and operation order as the library's documented definition
// (binary32 division, binary64 distances, ties to the lower index), and the
// mean uses a fixed summation order (blocks in order within each group, then
// group sums in order), so the output is deterministic bit for bit.
//
// Kernels (none is on the decode hot path):
//   1. absmax_encode: one warp per block -- max |w| (order-free), then each
//      lane encodes its elements; the block absmax goes to the workspace.
//   2. group_sums: one thread per group, binary64 sum of its blocks in order.
//   3. finalize_offset: one thread, binary64 sum of the group sums in order,
//      divided by the block count, rounded to binary32.
//   4. second_level: one warp per group -- absmax2 and absmax_q.

#include "nf4_internal.cuh"

namespace nf4 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

__device__ __forceinline__ int nearest_code(float v, const float* sT) {
  int best = 0;
  double bestd = fabs(__dsub_rn(double(v), double(sT[0])));
#pragma unroll
  for (int j = 1; j < 16; ++j) {
    const double d = fabs(__dsub_rn(double(v), double(sT[j])));
    if (d < bestd) {
      bestd = d;
      best = j;
    }
  }
  return best;
}

__global__ void __launch_bounds__(kThreads) absmax_encode_kernel(const float* __restrict__ w,
                                                                 int64_t n, int lbs,
                                                                 uint8_t* __restrict__ packed,
                                                                 float* __restrict__ absmax) {
  __shared__ float sT[16];
  if (threadIdx.x < 16) sT[threadIdx.x] = nf4_code_select(int(threadIdx.x));
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t bs = int64_t(1) << lbs;
  const int64_t nb = (n + bs - 1) >> lbs;
  const int64_t gwarp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = int64_t(gridDim.x) * kWarps;
  for (int64_t b = gwarp; b < nb; b += nwarps) {
    const int64_t k0 = b << lbs;
    const int64_t k1 = (k0 + bs < n) ? k0 + bs : n;
    float m = 0.0f;
    for (int64_t k = k0 + lane; k < k1; k += 32) m = fmaxf(m, fabsf(w[k]));
    m = warp_max(m);
    if (lane == 0) absmax[b] = m;
    // Each lane encodes whole bytes (element pairs) of the block; a pair never
    // straddles blocks because blocks have an even size.
    for (int64_t k = k0 + 2 * lane; k < k1; k += 64) {
      const float v0 = (m == 0.0f) ? 0.0f : __fdiv_rn(w[k], m);
      const int i0 = nearest_code(v0, sT);
      int i1 = 0;
      if (k + 1 < k1) {
        const float v1 = (m == 0.0f) ? 0.0f : __fdiv_rn(w[k + 1], m);
        i1 = nearest_code(v1, sT);
      }
      packed[k >> 1] = uint8_t((i0 << 4) | i1);
    }
  }
}

__global__ void __launch_bounds__(kThreads) group_sums_kernel(const float* __restrict__ absmax,
                                                              int64_t nb, int ls2,
                                                              double* __restrict__ part) {
  const int64_t ng = (nb + (int64_t(1) << ls2) - 1) >> ls2;
  for (int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; g < ng;
       g += int64_t(gridDim.x) * blockDim.x) {
    const int64_t b0 = g << ls2;
    const int64_t b1 = (b0 + (int64_t(1) << ls2) < nb) ? b0 + (int64_t(1) << ls2) : nb;
    double s = 0.0;
    for (int64_t b = b0; b < b1; ++b) s = __dadd_rn(s, double(absmax[b]));
    part[g] = s;
  }
}

__global__ void finalize_offset_kernel(const double* __restrict__ part, int64_t ng, int64_t nb,
                                       float* __restrict__ offset) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    double total = 0.0;
    for (int64_t g = 0; g < ng; ++g) total = __dadd_rn(total, part[g]);
    *offset = __double2float_rn(__ddiv_rn(total, double(nb)));
  }
}

__global__ void __launch_bounds__(kThreads) second_level_kernel(
    const float* __restrict__ absmax, int64_t nb, int ls2, const uint16_t* __restrict__ code2,
    const float* __restrict__ offset_p, uint16_t* __restrict__ absmax2,
    uint8_t* __restrict__ absmax_q) {
  __shared__ double sC2[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sC2[i] = double(half_bits_to_float(code2[i]));
  __syncthreads();
  const float offset = *offset_p;
  const int lane = threadIdx.x & 31;
  const int64_t s2 = int64_t(1) << ls2;
  const int64_t ng = (nb + s2 - 1) >> ls2;
  const int64_t gwarp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = int64_t(gridDim.x) * kWarps;
  for (int64_t g = gwarp; g < ng; g += nwarps) {
    const int64_t b0 = g << ls2;
    const int64_t b1 = (b0 + s2 < nb) ? b0 + s2 : nb;
    float m = 0.0f;
    for (int64_t b = b0 + lane; b < b1; b += 32) m = fmaxf(m, fabsf(__fsub_rn(absmax[b], offset)));
    m = warp_max(m);
    const uint16_t a2h = __half_as_ushort(__float2half_rn(m));
    if (lane == 0) absmax2[g] = a2h;
    const float a2 = half_bits_to_float(a2h);
    for (int64_t b = b0 + lane; b < b1; b += 32) {
      const float r = (a2 == 0.0f) ? 0.0f : __fdiv_rn(__fsub_rn(absmax[b], offset), a2);
      const double rd = double(r);
      int best = 0;
      double bestd = fabs(__dsub_rn(rd, sC2[0]));
      for (int i = 1; i < 256; ++i) {
        const double d = fabs(__dsub_rn(rd, sC2[i]));
        if (d < bestd) {
          bestd = d;
          best = i;
        }
      }
      absmax_q[b] = uint8_t(best);
    }
  }
}

int64_t grid_for(int64_t work_items, int64_t per_block, int sms) {
  int64_t g = (work_items + per_block - 1) / per_block;
  const int64_t cap = int64_t(sms > 0 ? sms : 1) * 8;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return g;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

size_t quantize_workspace_bytes(int64_t n, int lbs, int ls2) {
  if (n <= 0) return 0;
  const int64_t nb = (n + (int64_t(1) << lbs) - 1) >> lbs;
  const int64_t ng = (nb + (int64_t(1) << ls2) - 1) >> ls2;
  return align_up(size_t(nb) * sizeof(float), 256) + size_t(ng) * sizeof(double);
}

cudaError_t launch_quantize(const float* w, int64_t n, int lbs, int ls2, const uint16_t* code2,
                            uint8_t* packed, uint8_t* absmax_q, uint16_t* absmax2, float* offset,
                            void* workspace, cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int64_t nb = (n + (int64_t(1) << lbs) - 1) >> lbs;
  const int64_t ng = (nb + (int64_t(1) << ls2) - 1) >> ls2;
  float* absmax = static_cast<float*>(workspace);
  double* part = reinterpret_cast<double*>(static_cast<char*>(workspace) +
                                           align_up(size_t(nb) * sizeof(float), 256));
  absmax_encode_kernel<<<dim3(unsigned(grid_for(nb, kWarps, sms))), kThreads, 0, stream>>>(
      w, n, lbs, packed, absmax);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  group_sums_kernel<<<dim3(unsigned(grid_for(ng, kThreads, sms))), kThreads, 0, stream>>>(
      absmax, nb, ls2, part);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  finalize_offset_kernel<<<1, 32, 0, stream>>>(part, ng, nb, offset);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  second_level_kernel<<<dim3(unsigned(grid_for(ng, kWarps, sms))), kThreads, 0, stream>>>(
      absmax, nb, ls2, code2, offset, absmax2, absmax_q);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Fixed scratch for nf4_quantize_noalloc: the same four kernels, with the
// block-absmax / group-sum workspace in a file-scope device array instead of
// caller memory. It serves callers that cannot allocate device memory: hosts
// with no device allocator of their own (plain C programs without a caching
// allocator) and code that must not call cudaMalloc/cudaFree, which may
// synchronise the device and stall work queued on other streams. The array is
// fully overwritten before it is read (every block absmax and every group sum
// is written by the first two kernels), so nothing has to be cleared. It is
// one array per device, shared by every caller: calls that overlap in time
// (different streams, or different host threads without an ordering between
// their streams) race on it and must be serialised by the caller.
namespace {

__device__ __align__(256) unsigned char g_quantize_scratch[NF4_QUANTIZE_NOALLOC_SCRATCH_BYTES];

}  // namespace

// Device address of g_quantize_scratch in the current context, looked up on
// every call (cudaGetSymbolAddress, which may load this translation unit's
// module): nothing is cached, so the address stays right after a
// cudaDeviceReset or when another context is current.
cudaError_t quantize_static_scratch(void** ptr) {
  return cudaGetSymbolAddress(ptr, g_quantize_scratch);
}

}  // namespace nf4
