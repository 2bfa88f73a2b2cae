/*
 * nf4.h -- C ABI of libnf4: NF4 (4-bit NormalFloat) weights with double
 * quantization on NVIDIA GB300 (sm_103a).
 *
 * Format (the bitsandbytes-style layout described by the pages):
 *   - Code book: the sixteen NF4 values printed in "NF4反量化算子优化"
 *     (roundaboutt.github.io), section "NF4 table".
 *   - A tensor of n elements is flattened and cut into blocks of `blocksize`
 *     consecutive elements; blocks are grouped by `s2_blocksize`
 *     ("NF4 双重量化反量化 CUDA Kernel 实现报告", section 1.2).
 *   - packed   : uint8 [ceil(n/2)], two 4-bit code indices per byte; element
 *                2t is the HIGH nibble of byte t, element 2t+1 the LOW nibble
 *                (same report, section 2.2). For odd n the last low nibble is
 *                padding.
 *   - absmax_q : uint8 [ceil(n/blocksize)], index into code2 per block.
 *   - absmax2  : binary16 bit patterns [ceil(nblocks/s2_blocksize)], one
 *                second-level scale per group.
 *   - code2    : binary16 bit patterns [256], second-level code table.
 *   - offset   : binary32 scalar added to every decoded block scale.
 *   Dequantization (same report, section 1.3), for element k:
 *     b = k / blocksize, g = b / s2_blocksize,
 *     s = fp32( fp32(code2[absmax_q[b]] * absmax2[g]) + offset ),
 *     out[k] = round16( fp32( NF4[idx(k)] * s ) ),
 *   every operation a separately rounded binary32 operation (no fused
 *   multiply-add), round16 = round-to-nearest-even into bfloat16 or binary16
 *   (subnormals kept).
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them, and keeps no global state beyond
 *     a per-device cache of the SM count and the fixed device scratch array of
 *     nf4_quantize_noalloc.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising.
 *   - Argument checks run on the host before any launch; on failure nothing
 *     is enqueued and an error status is returned. A launch failure returns
 *     NF4_ERR_CUDA (the CUDA error is consumed; nf4_last_cuda_error() returns
 *     it). Kernels never trap.
 *   - Sizes are element counts (int64). Misaligned vector pointers are not an
 *     error: such calls run a slower kernel. Pointers not aligned to their
 *     element size are NF4_ERR_MISALIGNED.
 */
#ifndef NF4_H_
#define NF4_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NF4_API __attribute__((visibility("default")))
#else
#define NF4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* nf4_stream_t;

typedef enum {
  NF4_OK = 0,
  NF4_ERR_NULL = 1,                  /* a required pointer is NULL */
  NF4_ERR_INVALID_SIZE = 2,          /* negative size, odd K, size overflow */
  NF4_ERR_UNSUPPORTED_BLOCKSIZE = 3, /* blocksize / s2_blocksize not a supported power of two */
  NF4_ERR_MISALIGNED = 4,            /* pointer not aligned to its element size */
  NF4_ERR_UNSUPPORTED_DTYPE = 5,     /* output type not accepted by the call */
  NF4_ERR_UNSUPPORTED_BATCH = 6,     /* GEMV batch outside 1..64 */
  NF4_ERR_CUDA = 7,                  /* a CUDA runtime call failed */
  NF4_ERR_WORKSPACE = 8              /* workspace missing or too small */
} nf4_status;

/* Output element types: bfloat16, binary16 (IEEE half), binary32. nf4_dequant
 * writes the two 16-bit types; nf4_gemv_ex writes all three. */
typedef enum { NF4_BF16 = 0, NF4_FP16 = 1, NF4_F32 = 2 } nf4_dtype;

/* Library version as major*10000 + minor*100 + patch. */
NF4_API int nf4_version(void);

/* Static, human-readable name of a status code (never NULL). */
NF4_API const char* nf4_status_string(nf4_status status);

/* The cudaError_t value behind the last NF4_ERR_CUDA returned on this host
 * thread (0 if none). */
NF4_API int nf4_last_cuda_error(void);

/*
 * nf4_device_error_flags -- read and clear the library's device-side error
 * flags. Bit 0 is set when a bounded wait of the tensor-core GEMV (batches
 * 9..64) on its own copy or MMA pipeline ran out (about one second); that
 * launch then writes undefined values to its outputs and finishes instead
 * of hanging. The flags are one word per device, shared by every stream and
 * caller of the library. Synchronises with the device (cudaMemcpyFromSymbol).
 * `flags` is a host pointer.
 * Errors: NF4_ERR_NULL, NF4_ERR_CUDA.
 */
NF4_API nf4_status nf4_device_error_flags(unsigned int* flags);

/*
 * nf4_dequant -- expand n NF4 elements to bfloat16 or binary16.
 * Defined by "NF4 双重量化反量化 CUDA Kernel 实现报告", section 1.3 (formula)
 * and section 2.2 (nibble order); see the format notes above.
 *
 *   packed       uint8  [ceil(n/2)]
 *   absmax_q     uint8  [ceil(n/blocksize)]
 *   absmax2      uint16 [ceil(ceil(n/blocksize)/s2_blocksize)]  (binary16 bits)
 *   code2        uint16 [256]                                   (binary16 bits)
 *   offset       binary32 scalar (by value)
 *   n            number of elements, >= 0 (0 enqueues nothing and returns NF4_OK)
 *   blocksize    power of two, 2 .. 2^20 (64 is the usual value)
 *   s2_blocksize power of two, 1 .. 2^20 (256 is the usual value)
 *   out          [n] 16-bit elements of out_dtype, 2-byte aligned; written
 *                bit-exactly per the formula. Fastest when out is 16-byte
 *                and packed 4-byte aligned.
 *   out_dtype    NF4_BF16 or NF4_FP16
 * Errors: NF4_ERR_NULL, NF4_ERR_INVALID_SIZE (n < 0 or n > 2^40),
 *   NF4_ERR_UNSUPPORTED_BLOCKSIZE, NF4_ERR_MISALIGNED (absmax2, code2, out not
 *   2-byte aligned), NF4_ERR_UNSUPPORTED_DTYPE, NF4_ERR_CUDA.
 */
NF4_API nf4_status nf4_dequant(const uint8_t* packed, const uint8_t* absmax_q,
                       const uint16_t* absmax2, const uint16_t* code2, float offset,
                       int64_t n, int32_t blocksize, int32_t s2_blocksize, void* out,
                       nf4_dtype out_dtype, nf4_stream_t stream);

/*
 * nf4_gemv -- decode GEMV with the dequantization fused: y = W_hat x.
 * The fused form follows "RTX 4060 上的 LLM 量化实测：4-bit decode 比 FP16
 * 慢在哪里", section "Fused kernel：把反量化搬到片上" (unpack, look up, scale
 * and accumulate on chip in fp32; only y is written); the per-warp row
 * structure follows "CUDA 进阶手册 / 量化与 GEMV", section "GEMV kernel 的写法".
 *
 *   packed, absmax_q, absmax2, code2, offset, blocksize, s2_blocksize:
 *                the quantized N x K weight, row-major with K contiguous,
 *                quantized as one flattened tensor of N*K elements
 *                (element (r, k) is flat index r*K + k).
 *   N, K         output and input features; N >= 0, K >= 0 and even.
 *   x            bfloat16 bit patterns [batch][K], 2-byte aligned.
 *   batch        1 .. 64 activation vectors. 9 .. 64 run on the tensor cores
 *                (one launch) when K is a multiple of 64, blocksize >= 64
 *                and packed and x are 16-byte aligned, otherwise in slabs
 *                of up to 8 vectors (one launch each).
 *   y            binary32 [batch][N], 4-byte aligned:
 *                y[b][r] = sum_k W_hat[r][k] * x[b][k], with W_hat[r][k] the
 *                binary32 dequantized weight (before 16-bit rounding) and
 *                binary32 accumulation in an unspecified order. The result
 *                satisfies |y - y_exact| <= 1e-3 * sum_k |W_hat x| + 1e-6.
 *                K == 0 writes zeros.
 * Errors: NF4_ERR_NULL, NF4_ERR_INVALID_SIZE (N < 0, K < 0, K odd, N*K > 2^40),
 *   NF4_ERR_UNSUPPORTED_BLOCKSIZE, NF4_ERR_MISALIGNED,
 *   NF4_ERR_UNSUPPORTED_BATCH, NF4_ERR_CUDA.
 */
NF4_API nf4_status nf4_gemv(const uint8_t* packed, const uint8_t* absmax_q,
                    const uint16_t* absmax2, const uint16_t* code2, float offset,
                    int64_t N, int64_t K, int32_t blocksize, int32_t s2_blocksize,
                    const uint16_t* x, int32_t batch, float* y, nf4_stream_t stream);

/*
 * nf4_gemv_ex -- nf4_gemv with the layer's output stage fused: an optional
 * bias and a 16-bit (or binary32) y. "RTX 4060 上的 LLM 量化实测", section
 * "Fused kernel：把反量化搬到片上", stores each fp32 row sum as binary16 and
 * then adds the layer's bias; here both happen in the epilogue of the same
 * kernel, with a single rounding.
 *
 *   packed .. batch  as for nf4_gemv.
 *   bias         NULL, or [N] elements of y_dtype (device), aligned to its
 *                element size.
 *   y            [batch][N] elements of y_dtype (device), aligned likewise:
 *                y[b][r] = round(fp32(sum_b_r + bias[r])), where sum_b_r is
 *                a binary32 row sum as accurate as nf4_gemv's y (in practice
 *                the same kernel and order), bias[r] is widened
 *                exactly to binary32, the addition is one binary32 operation
 *                and round is round-to-nearest-even into y_dtype (the
 *                identity for NF4_F32). Without a bias, y = round(sum_b_r).
 *                So |y - v| is at most 1e-3 * (sum_k |W_hat x| + |bias[r]|)
 *                + 1e-6 plus half a unit in the last place of y_dtype, with
 *                v the exact value sum_k W_hat x + bias[r].
 *   y_dtype      NF4_BF16, NF4_FP16 or NF4_F32. K == 0 writes round(bias),
 *                or zeros.
 * nf4_gemv(..., y, stream) is nf4_gemv_ex(..., NULL, y, NF4_F32, stream).
 * Errors: as nf4_gemv, plus NF4_ERR_UNSUPPORTED_DTYPE.
 */
NF4_API nf4_status nf4_gemv_ex(const uint8_t* packed, const uint8_t* absmax_q,
                       const uint16_t* absmax2, const uint16_t* code2, float offset,
                       int64_t N, int64_t K, int32_t blocksize, int32_t s2_blocksize,
                       const uint16_t* x, int32_t batch, const void* bias, void* y,
                       nf4_dtype y_dtype, nf4_stream_t stream);

/*
 * Decode step: a fixed sequence of fused GEMV nodes (the linear layers of a
 * decoder's token step), recorded once into a CUDA graph and replayed once
 * per token. "RTX 4060 上的 LLM 量化实测", sections "逐层 profiling：问题出在哪"
 * and "为什么是 k/v projection", finds fixed per-call costs dominating the
 * thin k_proj / v_proj GEMVs of a decode step; a replay pays no host launch
 * cost, and consecutive kernels overlap their start with the previous
 * kernel's end (programmatic dependent launch). Work between the GEMVs of a
 * real decoder (attention, norms, activation) is not part of a step.
 *
 * A node is one nf4_gemv_ex call. Its input is the step's x (input = -1) or
 * the y of an earlier node j (input = j < this node's index), which must be
 * NF4_BF16 with N_j == K. Node i runs after node i-1 (stream order).
 */
typedef struct nf4_gemv_node {
  const uint8_t* packed;    /* the quantized N x K weight, as for nf4_gemv */
  const uint8_t* absmax_q;
  const uint16_t* absmax2;
  const uint16_t* code2;
  float offset;
  int64_t N, K;
  int32_t blocksize, s2_blocksize;
  const void* bias;         /* NULL or [N] of y_dtype */
  int32_t input;            /* -1: the step's x; j >= 0: y of node j */
  void* y;                  /* [batch][N] of y_dtype, caller-owned */
  nf4_dtype y_dtype;
} nf4_gemv_node;

typedef struct nf4_step_st* nf4_step_t;

/*
 * nf4_step_create -- validate the nodes (each as nf4_gemv_ex would, plus the
 * input rules above) and record them into a CUDA graph on the current
 * device. Consecutive nodes with the same input, K and block sizes (up to
 * four, e.g. q/k/v or gate/up) share one launch. All pointers (weights,
 * x [batch][K], biases, every y) are device pointers captured by value: they
 * must stay valid, and their contents are read / written at each
 * nf4_step_launch, not at creation. Nothing is launched here.
 * Each node group is one kernel launch, with programmatic dependent launch
 * between consecutive kernels. The step owns only host-side graph objects
 * (the library allocates no device buffers). Free it with nf4_step_destroy.
 * Errors: NF4_ERR_NULL (step, nodes, or a node's pointers),
 *   NF4_ERR_INVALID_SIZE (n_nodes < 1, a bad input index, K != N of the
 *   input node, or a node's sizes), NF4_ERR_UNSUPPORTED_DTYPE (an input node
 *   whose y is not NF4_BF16, or a bad y_dtype), the other nf4_gemv_ex errors,
 *   NF4_ERR_CUDA (stream capture or graph instantiation failed). On error
 *   *step is NULL.
 */
NF4_API nf4_status nf4_step_create(const nf4_gemv_node* nodes, int32_t n_nodes,
                                   const uint16_t* x, int32_t batch, nf4_step_t* step);

/*
 * nf4_step_launch -- enqueue one replay of the step on `stream` (returns
 * without synchronising). Replays on one stream run one after another; two
 * replays of the same step must not overlap in time (they share every
 * buffer). Errors: NF4_ERR_NULL, NF4_ERR_CUDA (also when the current device
 * is not the one the step was created on).
 */
NF4_API nf4_status nf4_step_launch(nf4_step_t step, nf4_stream_t stream);

/* nf4_step_destroy -- free a step (NULL is a no-op). Synchronises nothing:
 * the caller waits for replays in flight first. */
NF4_API nf4_status nf4_step_destroy(nf4_step_t step);

/*
 * nf4_step_kernel_count -- number of kernel launches one replay of `step`
 * performs (the kernel nodes of its recorded graph), to check how nodes were
 * grouped: the per-call fixed cost that "RTX 4060 上的 LLM 量化实测", section
 * "为什么是 k/v projection", finds dominating thin layers is paid once per
 * launch. `count` is a host pointer; 0 for a step whose nodes were all empty.
 * Errors: NF4_ERR_NULL, NF4_ERR_CUDA.
 */
NF4_API nf4_status nf4_step_kernel_count(nf4_step_t step, int32_t* count);

/*
 * nf4_quantize_workspace_size -- bytes of device workspace nf4_quantize needs
 * for n elements (0 for n <= 0 or unsupported block sizes).
 */
NF4_API size_t nf4_quantize_workspace_size(int64_t n, int32_t blocksize, int32_t s2_blocksize);

/*
 * nf4_quantize -- NF4 quantization with double quantization of a binary32
 * tensor, the encoding that nf4_dequant inverts.
 * First level: "NF4反量化算子优化", section "双量化 / 第一层量化" (flatten,
 * blocks of `blocksize`, per-block absmax, divide, nearest code, two codes per
 * byte). Second level: the same section "第二层量化" and
 * "NF4 双重量化反量化 CUDA Kernel 实现报告", section 1.2 (absmax quantized to
 * uint8 indices into code2, one binary16 absmax2 per group, a binary32 offset).
 * Where the pages leave a step open this library fixes it as follows:
 *   absmax[b]   = max |w| over the elements of block b present;
 *   v           = w / absmax[b] (binary32 division; 0 if absmax[b] == 0);
 *   code index  = argmin_j |v - NF4[j]| in binary64, ties to the lower j;
 *   offset      = binary32( S / nblocks ), S the binary64 sum of absmax taken
 *                 group by group (blocks in order within a group, then the
 *                 group sums in order);
 *   absmax2[g]  = binary16 RNE of max |absmax[b] - offset| (binary32) over the
 *                 blocks of group g;
 *   absmax_q[b] = argmin_i |r - code2[i]| in binary64, ties to the lower i,
 *                 r = binary32 (absmax[b] - offset) / absmax2[g] (0 if absmax2 is 0).
 *
 *   w            binary32 [n], finite values, 4-byte aligned
 *   n, blocksize, s2_blocksize: as for nf4_dequant
 *   code2        binary16 bits [256], increasing (caller-chosen table)
 *   packed, absmax_q, absmax2: outputs, sized as for nf4_dequant
 *   offset       device pointer to ONE binary32 output
 *   workspace    device scratch of at least nf4_quantize_workspace_size() bytes,
 *                8-byte aligned; contents on entry are ignored
 * Errors: NF4_ERR_NULL, NF4_ERR_INVALID_SIZE, NF4_ERR_UNSUPPORTED_BLOCKSIZE,
 *   NF4_ERR_MISALIGNED, NF4_ERR_WORKSPACE, NF4_ERR_CUDA.
 */
NF4_API nf4_status nf4_quantize(const float* w, int64_t n, int32_t blocksize, int32_t s2_blocksize,
                        const uint16_t* code2, uint8_t* packed, uint8_t* absmax_q,
                        uint16_t* absmax2, float* offset, void* workspace,
                        size_t workspace_bytes, nf4_stream_t stream);

/* Size in bytes of the fixed device scratch array of nf4_quantize_noalloc:
 * 16 MiB + 128 KiB, the nf4_quantize workspace of n = 2^28 elements at
 * blocksize 64, s2_blocksize 256. */
#define NF4_QUANTIZE_NOALLOC_SCRATCH_BYTES 16908288

/*
 * nf4_quantize_noalloc -- nf4_quantize with its workspace taken from a fixed
 * device array inside the library instead of caller memory. The pages have no
 * counterpart: it is an interface variant for callers that cannot allocate
 * device memory (hosts with no device allocator of their own, and code that
 * must not call cudaMalloc/cudaFree because they may synchronise the device).
 * It allocates and frees nothing. Results are identical to nf4_quantize.
 *
 *   Arguments, layout and definition: as for nf4_quantize, without
 *   `workspace` / `workspace_bytes`.
 *   Limit: nf4_quantize_workspace_size(n, blocksize, s2_blocksize) must not
 *     exceed NF4_QUANTIZE_NOALLOC_SCRATCH_BYTES (n <= 2^28 at blocksize 64,
 *     s2_blocksize 256); larger inputs return NF4_ERR_WORKSPACE before any
 *     CUDA call.
 *   Set-up: every call looks up the array's device address in the current
 *     context with cudaGetSymbolAddress (nothing is cached, so the entry point
 *     keeps working after cudaDeviceReset or with another context current).
 *     The first call on a device may load the library's module: make one call
 *     before any stream capture.
 *   Concurrency: the array is shared by all callers on a device, so calls
 *     whose kernels may overlap in time (different streams, or host threads
 *     without an ordering between their streams) race on it; the caller
 *     serialises them. Calls on one stream are ordered and safe.
 * Errors: NF4_ERR_NULL, NF4_ERR_INVALID_SIZE, NF4_ERR_UNSUPPORTED_BLOCKSIZE,
 *   NF4_ERR_MISALIGNED, NF4_ERR_WORKSPACE (input too large for the array),
 *   NF4_ERR_CUDA.
 */
NF4_API nf4_status nf4_quantize_noalloc(const float* w, int64_t n, int32_t blocksize,
                                        int32_t s2_blocksize, const uint16_t* code2,
                                        uint8_t* packed, uint8_t* absmax_q, uint16_t* absmax2,
                                        float* offset, nf4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NF4_H_ */
