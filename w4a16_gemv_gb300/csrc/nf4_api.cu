// nf4_api.cu -- the C ABI of libnf4 (declared in include/nf4.h): host-side
// argument validation, then one launch sequence on the caller's stream.
#include <stdint.h>

#include "nf4_internal.cuh"

namespace nf4 {

int device_sm_count() {
  static PerDeviceCache cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  return cache.get(dev, [dev] {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return -1;
    return sms;
  });
}

}  // namespace nf4

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int64_t kMaxElems = int64_t(1) << 40;

bool is_pow2_log(int32_t v, int32_t lo, int32_t hi, int* log2_out) {
  if (v < lo || v > hi || (v & (v - 1)) != 0) return false;
  int l = 0;
  while ((int32_t(1) << l) < v) ++l;
  *log2_out = l;
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

nf4_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return NF4_OK;
  g_last_cuda_error = int(e);
  return NF4_ERR_CUDA;
}

nf4_status check_block_sizes(int32_t blocksize, int32_t s2_blocksize, int* lbs, int* ls2) {
  if (!is_pow2_log(blocksize, 2, 1 << 20, lbs)) return NF4_ERR_UNSUPPORTED_BLOCKSIZE;
  if (!is_pow2_log(s2_blocksize, 1, 1 << 20, ls2)) return NF4_ERR_UNSUPPORTED_BLOCKSIZE;
  return NF4_OK;
}

nf4_status check_quant_inputs(const uint8_t* packed, const uint8_t* absmax_q,
                              const uint16_t* absmax2, const uint16_t* code2) {
  if (!packed || !absmax_q || !absmax2 || !code2) return NF4_ERR_NULL;
  if (!aligned(absmax2, 2) || !aligned(code2, 2)) return NF4_ERR_MISALIGNED;
  return NF4_OK;
}

}  // namespace

extern "C" {

int nf4_version(void) { return 100; }  // 0.1.0

const char* nf4_status_string(nf4_status status) {
  switch (status) {
    case NF4_OK: return "NF4_OK";
    case NF4_ERR_NULL: return "NF4_ERR_NULL: a required pointer is NULL";
    case NF4_ERR_INVALID_SIZE: return "NF4_ERR_INVALID_SIZE: negative, odd (K) or too large size";
    case NF4_ERR_UNSUPPORTED_BLOCKSIZE:
      return "NF4_ERR_UNSUPPORTED_BLOCKSIZE: block sizes must be powers of two "
             "(blocksize 2..2^20, s2_blocksize 1..2^20)";
    case NF4_ERR_MISALIGNED: return "NF4_ERR_MISALIGNED: pointer not aligned to its element size";
    case NF4_ERR_UNSUPPORTED_DTYPE:
      return "NF4_ERR_UNSUPPORTED_DTYPE: dequant output must be NF4_BF16 or NF4_FP16, "
             "GEMV output NF4_BF16, NF4_FP16 or NF4_F32";
    case NF4_ERR_UNSUPPORTED_BATCH: return "NF4_ERR_UNSUPPORTED_BATCH: batch must be 1..64";
    case NF4_ERR_CUDA: return "NF4_ERR_CUDA: a CUDA runtime call failed (see nf4_last_cuda_error)";
    case NF4_ERR_WORKSPACE: return "NF4_ERR_WORKSPACE: workspace missing or too small";
  }
  return "NF4: unknown status";
}

int nf4_last_cuda_error(void) { return g_last_cuda_error; }

nf4_status nf4_device_error_flags(unsigned int* flags) {
  if (!flags) return NF4_ERR_NULL;
  return cuda_status(nf4::read_and_clear_device_flags(flags));
}

nf4_status nf4_dequant(const uint8_t* packed, const uint8_t* absmax_q, const uint16_t* absmax2,
                       const uint16_t* code2, float offset, int64_t n, int32_t blocksize,
                       int32_t s2_blocksize, void* out, nf4_dtype out_dtype,
                       nf4_stream_t stream) {
  if (n < 0 || n > kMaxElems) return NF4_ERR_INVALID_SIZE;
  int lbs = 0, ls2 = 0;
  nf4_status st = check_block_sizes(blocksize, s2_blocksize, &lbs, &ls2);
  if (st != NF4_OK) return st;
  if (out_dtype != NF4_BF16 && out_dtype != NF4_FP16) return NF4_ERR_UNSUPPORTED_DTYPE;
  if (n == 0) return NF4_OK;
  st = check_quant_inputs(packed, absmax_q, absmax2, code2);
  if (st != NF4_OK) return st;
  if (!out) return NF4_ERR_NULL;
  if (!aligned(out, 2)) return NF4_ERR_MISALIGNED;
  const nf4::QuantTensor t{packed, absmax_q, absmax2, code2, offset, lbs, ls2};
  return cuda_status(nf4::launch_dequant(t, n, out, out_dtype, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace nf4 {

nf4_status check_gemv_args(const uint8_t* packed, const uint8_t* absmax_q,
                           const uint16_t* absmax2, const uint16_t* code2, float offset, int64_t N,
                           int64_t K, int32_t blocksize, int32_t s2_blocksize, const uint16_t* x,
                           int32_t batch, const void* bias, void* y, nf4_dtype y_dtype,
                           QuantTensor* t, YOut* out) {
  if (N < 0 || K < 0 || (K & 1) != 0) return NF4_ERR_INVALID_SIZE;
  if (K > 0 && N > kMaxElems / K) return NF4_ERR_INVALID_SIZE;
  if (N > kMaxElems) return NF4_ERR_INVALID_SIZE;
  int lbs = 0, ls2 = 0;
  nf4_status st = check_block_sizes(blocksize, s2_blocksize, &lbs, &ls2);
  if (st != NF4_OK) return st;
  if (batch < 1 || batch > 64) return NF4_ERR_UNSUPPORTED_BATCH;
  if (y_dtype != NF4_BF16 && y_dtype != NF4_FP16 && y_dtype != NF4_F32)
    return NF4_ERR_UNSUPPORTED_DTYPE;
  if (N == 0) return NF4_OK;
  if (!y) return NF4_ERR_NULL;
  const uintptr_t ysize = y_dtype == NF4_F32 ? 4 : 2;
  if (!aligned(y, ysize) || (bias && !aligned(bias, ysize))) return NF4_ERR_MISALIGNED;
  if (K > 0) {
    st = check_quant_inputs(packed, absmax_q, absmax2, code2);
    if (st != NF4_OK) return st;
    if (!x) return NF4_ERR_NULL;
    if (!aligned(x, 2)) return NF4_ERR_MISALIGNED;
  }
  *t = QuantTensor{packed, absmax_q, absmax2, code2, offset, lbs, ls2};
  *out = YOut{y, bias, int(y_dtype)};
  return NF4_OK;
}

nf4_status status_of(cudaError_t e) { return cuda_status(e); }

}  // namespace nf4

extern "C" {

nf4_status nf4_gemv_ex(const uint8_t* packed, const uint8_t* absmax_q, const uint16_t* absmax2,
                       const uint16_t* code2, float offset, int64_t N, int64_t K,
                       int32_t blocksize, int32_t s2_blocksize, const uint16_t* x,
                       int32_t batch, const void* bias, void* y, nf4_dtype y_dtype,
                       nf4_stream_t stream) {
  nf4::QuantTensor t;
  nf4::YOut out;
  const nf4_status st = nf4::check_gemv_args(packed, absmax_q, absmax2, code2, offset, N, K,
                                             blocksize, s2_blocksize, x, batch, bias, y, y_dtype,
                                             &t, &out);
  if (st != NF4_OK || N == 0) return st;
  return cuda_status(
      nf4::launch_gemv(t, N, K, x, batch, out, reinterpret_cast<cudaStream_t>(stream)));
}

nf4_status nf4_gemv(const uint8_t* packed, const uint8_t* absmax_q, const uint16_t* absmax2,
                    const uint16_t* code2, float offset, int64_t N, int64_t K, int32_t blocksize,
                    int32_t s2_blocksize, const uint16_t* x, int32_t batch, float* y,
                    nf4_stream_t stream) {
  return nf4_gemv_ex(packed, absmax_q, absmax2, code2, offset, N, K, blocksize, s2_blocksize, x,
                     batch, nullptr, y, NF4_F32, stream);
}

size_t nf4_quantize_workspace_size(int64_t n, int32_t blocksize, int32_t s2_blocksize) {
  int lbs = 0, ls2 = 0;
  if (n <= 0 || n > kMaxElems) return 0;
  if (check_block_sizes(blocksize, s2_blocksize, &lbs, &ls2) != NF4_OK) return 0;
  return nf4::quantize_workspace_bytes(n, lbs, ls2);
}

nf4_status nf4_quantize(const float* w, int64_t n, int32_t blocksize, int32_t s2_blocksize,
                        const uint16_t* code2, uint8_t* packed, uint8_t* absmax_q,
                        uint16_t* absmax2, float* offset, void* workspace,
                        size_t workspace_bytes, nf4_stream_t stream) {
  if (n < 0 || n > kMaxElems) return NF4_ERR_INVALID_SIZE;
  int lbs = 0, ls2 = 0;
  nf4_status st = check_block_sizes(blocksize, s2_blocksize, &lbs, &ls2);
  if (st != NF4_OK) return st;
  if (n == 0) return NF4_OK;
  if (!w || !code2 || !packed || !absmax_q || !absmax2 || !offset) return NF4_ERR_NULL;
  if (!aligned(w, 4) || !aligned(code2, 2) || !aligned(absmax2, 2) || !aligned(offset, 4))
    return NF4_ERR_MISALIGNED;
  if (!workspace || workspace_bytes < nf4::quantize_workspace_bytes(n, lbs, ls2) ||
      !aligned(workspace, 8))
    return NF4_ERR_WORKSPACE;
  return cuda_status(nf4::launch_quantize(w, n, lbs, ls2, code2, packed, absmax_q, absmax2, offset,
                                          workspace, reinterpret_cast<cudaStream_t>(stream)));
}

nf4_status nf4_quantize_noalloc(const float* w, int64_t n, int32_t blocksize,
                                int32_t s2_blocksize, const uint16_t* code2, uint8_t* packed,
                                uint8_t* absmax_q, uint16_t* absmax2, float* offset,
                                nf4_stream_t stream) {
  if (n < 0 || n > kMaxElems) return NF4_ERR_INVALID_SIZE;
  int lbs = 0, ls2 = 0;
  nf4_status st = check_block_sizes(blocksize, s2_blocksize, &lbs, &ls2);
  if (st != NF4_OK) return st;
  if (n == 0) return NF4_OK;
  if (!w || !code2 || !packed || !absmax_q || !absmax2 || !offset) return NF4_ERR_NULL;
  if (!aligned(w, 4) || !aligned(code2, 2) || !aligned(absmax2, 2) || !aligned(offset, 4))
    return NF4_ERR_MISALIGNED;
  if (nf4::quantize_workspace_bytes(n, lbs, ls2) > size_t(NF4_QUANTIZE_NOALLOC_SCRATCH_BYTES))
    return NF4_ERR_WORKSPACE;
  void* scratch = nullptr;
  const cudaError_t e = nf4::quantize_static_scratch(&scratch);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(nf4::launch_quantize(w, n, lbs, ls2, code2, packed, absmax_q, absmax2, offset,
                                          scratch, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
