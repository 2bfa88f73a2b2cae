// nf4_internal.cuh -- definitions shared by the libnf4 translation units
// (device code tables, small device helpers, launcher declarations).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "nf4.h"

namespace nf4 {

// The NF4 code book: the sixteen 8-digit values printed in
// "NF4反量化算子优化", section "NF4 table", as binary32. Code j (0..15) is
// selected from immediates, without touching memory (a first access to
// __constant__ data costs each SM a DRAM round trip).
__device__ __forceinline__ float nf4_code_select(int j) {
  float v = -1.00000000f;
  v = (j == 1) ? -0.69619280f : v;
  v = (j == 2) ? -0.52507305f : v;
  v = (j == 3) ? -0.39491749f : v;
  v = (j == 4) ? -0.28444138f : v;
  v = (j == 5) ? -0.18477343f : v;
  v = (j == 6) ? -0.09105004f : v;
  v = (j == 7) ? 0.00000000f : v;
  v = (j == 8) ? 0.07958030f : v;
  v = (j == 9) ? 0.16093020f : v;
  v = (j == 10) ? 0.24611230f : v;
  v = (j == 11) ? 0.33791524f : v;
  v = (j == 12) ? 0.44070983f : v;
  v = (j == 13) ? 0.56261700f : v;
  v = (j == 14) ? 0.72295684f : v;
  v = (j == 15) ? 1.00000000f : v;
  return v;
}

// Arguments common to every entry point that reads a quantized tensor.
struct QuantTensor {
  const uint8_t* packed;
  const uint8_t* absmax_q;
  const uint16_t* absmax2;
  const uint16_t* code2;
  float offset;
  int lbs;  // log2(blocksize)
  int ls2;  // log2(s2_blocksize)
};

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

// Where a GEMV writes its result. Element (b, r) of y is
// round_dtype(fp32(sum + bias[r])): the binary32 sum, plus the bias widened
// exactly to binary32 (one rounded addition), then one rounding to nearest
// even into the output type. Without a bias the sum is rounded directly.
struct YOut {
  void* y;           // [batch][N] of dtype
  const void* bias;  // [N] of dtype, or nullptr
  int dtype;         // NF4_BF16, NF4_FP16 or NF4_F32
};

// Bias bits of row r as stored (16 or 32 bits), 0 without a bias.
__device__ __forceinline__ uint32_t y_bias_bits(const YOut& o, int64_t r) {
  if (!o.bias) return 0u;
  if (o.dtype == NF4_F32) return __ldg(reinterpret_cast<const uint32_t*>(o.bias) + r);
  return __ldg(reinterpret_cast<const uint16_t*>(o.bias) + r);
}

// Stores element idx of y from the binary32 sum and the row's bias bits.
__device__ __forceinline__ void y_store(const YOut& o, int64_t idx, float sum, uint32_t bias_bits) {
  float v = sum;
  if (o.bias) {
    const float bf = o.dtype == NF4_F32   ? __uint_as_float(bias_bits)
                     : o.dtype == NF4_BF16 ? __uint_as_float(bias_bits << 16)
                                           : half_bits_to_float(uint16_t(bias_bits));
    v = __fadd_rn(v, bf);
  }
  if (o.dtype == NF4_F32)
    reinterpret_cast<float*>(o.y)[idx] = v;
  else if (o.dtype == NF4_BF16)
    reinterpret_cast<__nv_bfloat16*>(o.y)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<__half*>(o.y)[idx] = __float2half_rn(v);
}

// Decoded scale of block b: fp32(fp32(code2[q] * absmax2[g]) + offset), two
// separately rounded operations (no contraction). `code2f` is the table
// already widened to binary32 (exact).
__device__ __forceinline__ float block_scale(const QuantTensor& t, const float* code2f,
                                             int64_t b) {
  const uint8_t q = __ldg(t.absmax_q + b);
  const float a2 = half_bits_to_float(__ldg(t.absmax2 + (b >> t.ls2)));
  return __fadd_rn(__fmul_rn(code2f[q], a2), t.offset);
}

// Read-only 4- and 16-byte global loads that do not allocate in L1.
__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ldg_stream_u128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Per-device values that the host side looks up once (device attributes, a
// kernel attribute already set) and then reads from any host thread. Each
// slot is an atomic: concurrent first calls may each run the (idempotent)
// lookup and store the same value; later calls read it without a lock.
constexpr int kMaxCachedDevices = 64;
class PerDeviceCache {
 public:
  // The stored value for `dev`, else compute(): a result >= 0 is stored, a
  // negative one (an error) is returned and not stored. Devices beyond the
  // cache always compute.
  template <typename F>
  int get(int dev, F&& compute) {
    const bool cached = dev >= 0 && dev < kMaxCachedDevices;
    if (cached) {
      const int v = slot_[dev].load(std::memory_order_acquire);
      if (v > 0) return v - 1;
    }
    const int r = compute();
    if (cached && r >= 0) slot_[dev].store(r + 1, std::memory_order_release);
    return r;
  }

 private:
  std::atomic<int> slot_[kMaxCachedDevices] = {};  // value + 1; 0: not yet known
};

// Raises `kern`'s dynamic shared memory limit to `bytes` once per device.
template <typename Kern>
cudaError_t set_max_dynamic_smem_once(Kern kern, int bytes, PerDeviceCache& done) {
  int dev = 0;
  const cudaError_t ed = cudaGetDevice(&dev);
  if (ed != cudaSuccess) return ed;
  cudaError_t err = cudaSuccess;
  done.get(dev, [&] {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return err == cudaSuccess ? 1 : -1;
  });
  return err;
}

// Per-device properties cached on first use (SM count).
int device_sm_count();

// Launchers (host). Each returns cudaSuccess or the launch error.
cudaError_t launch_dequant(const QuantTensor& t, int64_t n, void* out, nf4_dtype dtype,
                           cudaStream_t stream);
cudaError_t launch_gemv(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x,
                        int batch, const YOut& out, cudaStream_t stream);
size_t quantize_workspace_bytes(int64_t n, int lbs, int ls2);
cudaError_t launch_quantize(const float* w, int64_t n, int lbs, int ls2, const uint16_t* code2,
                            uint8_t* packed, uint8_t* absmax_q, uint16_t* absmax2,
                            float* offset, void* workspace, cudaStream_t stream);
// Device address of the fixed nf4_quantize_noalloc scratch on the current
// device (NF4_QUANTIZE_NOALLOC_SCRATCH_BYTES bytes, 256-byte aligned).
cudaError_t quantize_static_scratch(void** ptr);

}  // namespace nf4

namespace nf4 {

// ---------------------------------------------------------------------------
// Shared-memory mbarriers (the tensor-core GEMV's copy and MMA pipeline).

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the asynchronous proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar`, giving up after about `limit_cycles`
// SM clock cycles. Returns false on timeout (the caller reports it).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit_cycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit_cycles) return false;
  }
  return true;
}

// A wait on the library's own asynchronous copies that exceeds this many SM
// cycles (about one second at 2 GHz) is reported instead of spinning on.
constexpr long long kWaitLimitCycles = 2000000000ll;

// Device-side error flags (bit 0: a bounded wait timed out). Read and cleared
// by nf4_device_error_flags().
cudaError_t read_and_clear_device_flags(unsigned int* flags);

// One weight of a GEMV launch that may serve several weights sharing x.
struct SubTensor {
  QuantTensor t;
  YOut out;
  int64_t N;
  int cta0;  // first CTA serving this weight (set by the planner)
  int ctas;  // CTAs serving it (set by the planner)
};
constexpr int kMaxSub = 4;

// Batch-1 GEMV (k-stationary, direct weight loads) of 1..kMaxSub weights
// sharing x and K, in one launch. Sets *done when it handled the call;
// otherwise the caller uses the general kernels (one launch per weight).
cudaError_t try_gemv_b1(const SubTensor* subs, int nsub, int64_t K, const uint16_t* x, int sms,
                        cudaStream_t stream, bool* done);
// Batch 2..8 GEMV (k-stationary, binary32 x in registers, column slices),
// grouped as for batch 1.
cudaError_t try_gemv_bn(const SubTensor* subs, int nsub, int64_t K, const uint16_t* x, int batch,
                        int sms, cudaStream_t stream, bool* done);
// Batches 9..64 on the tensor cores (tcgen05.mma with the dequantized weights
// in tensor memory); *done is false (nothing launched) when the shape or
// the alignment does not fit (K a multiple of 64, blocksize >= 64 dividing
// K, 16-byte aligned packed weights and x).
cudaError_t try_gemm_tc(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x, int batch,
                        const YOut& out, int sms, cudaStream_t stream, bool* done);
cudaError_t read_and_clear_tc_flags(unsigned int* flags);
// Several weights sharing x and K in one launch of the streaming kernels;
// *done is false (nothing launched) when they cannot share one.
cudaError_t launch_gemv_group(const QuantTensor* ts, const int64_t* Ns, const YOut* outs, int n,
                              int64_t K, const uint16_t* x, int batch, cudaStream_t stream,
                              bool* done);

}  // namespace nf4

namespace nf4 {

// ---------------------------------------------------------------------------
// Programmatic dependent launch. Kernels of this library are launched with
// programmatic stream serialisation allowed, so a kernel can be scheduled
// while the previous kernel in the stream is still finishing. Each kernel
// therefore (1) signals its own dependents early and (2) waits for the
// previous grid's completion and memory flush before its first global
// memory access; work before that point touches only registers, shared
// memory and the constant bank.
#ifndef NF4_USE_PDL
#define NF4_USE_PDL 1
#endif

__device__ __forceinline__ void pdl_wait_prior_grid() {
#if NF4_USE_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

__device__ __forceinline__ void pdl_allow_dependents() {
#if NF4_USE_PDL
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

template <typename... KArgs, typename... Args>
cudaError_t launch_k_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = (NF4_USE_PDL && pdl) ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launch with programmatic stream serialisation allowed.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, Args&&... args) {
  return launch_k_pdl(true, kernel, grid, block, smem, stream, std::forward<Args>(args)...);
}

}  // namespace nf4
