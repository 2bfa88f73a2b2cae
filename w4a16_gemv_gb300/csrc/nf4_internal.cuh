// nf4_internal.cuh -- definitions shared by the libnf4 translation units
// (device code tables, small device helpers, launcher declarations).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nf4.h"

namespace nf4 {

// The NF4 code book: the sixteen 8-digit values printed in
// "NF4反量化算子优化", section "NF4 table", as binary32.
static __constant__ float kCode[16] = {
    -1.00000000f, -0.69619280f, -0.52507305f, -0.39491749f,
    -0.28444138f, -0.18477343f, -0.09105004f, 0.00000000f,
    0.07958030f,  0.16093020f,  0.24611230f,  0.33791524f,
    0.44070983f,  0.56261700f,  0.72295684f,  1.00000000f};

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

// Per-device properties cached on first use (SM count).
int device_sm_count();

// Launchers (host). Each returns cudaSuccess or the launch error.
cudaError_t launch_dequant(const QuantTensor& t, int64_t n, void* out, nf4_dtype dtype,
                           cudaStream_t stream);
cudaError_t launch_gemv(const QuantTensor& t, int64_t N, int64_t K, const uint16_t* x,
                        int batch, float* y, cudaStream_t stream);
size_t quantize_workspace_bytes(int64_t n, int lbs, int ls2);
cudaError_t launch_quantize(const float* w, int64_t n, int lbs, int ls2, const uint16_t* code2,
                            uint8_t* packed, uint8_t* absmax_q, uint16_t* absmax2,
                            float* offset, void* workspace, cudaStream_t stream);

}  // namespace nf4
