// nf4_step.cu -- decode step: a fixed sequence of fused GEMV nodes recorded
// once into a CUDA graph and replayed once per generated token.
//
// "RTX 4060 上的 LLM 量化实测", sections "逐层 profiling：问题出在哪" and
// "为什么是 k/v projection", finds the per-call fixed costs dominating the
// thin k_proj / v_proj layers of a decode step. Here the host cost of a
// launch is paid once, at record time; on replay each kernel is scheduled
// while its predecessor drains (programmatic dependent launch: the kernels
// build their shared tables before waiting on the previous grid), so the
// gaps between the layers of a step shrink to the dependent-launch latency.
#include <stdint.h>

#include <new>
#include <vector>

#include "nf4_internal.cuh"

struct nf4_step_st {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int device = -1;
  int32_t n_nodes = 0;
};

namespace nf4 {
nf4_status check_gemv_args(const uint8_t* packed, const uint8_t* absmax_q,
                           const uint16_t* absmax2, const uint16_t* code2, float offset, int64_t N,
                           int64_t K, int32_t blocksize, int32_t s2_blocksize, const uint16_t* x,
                           int32_t batch, const void* bias, void* y, nf4_dtype y_dtype,
                           QuantTensor* t, YOut* out);
nf4_status status_of(cudaError_t e);
}  // namespace nf4

namespace {

void destroy_graph(nf4_step_st* s) {
  if (s->exec) cudaGraphExecDestroy(s->exec);
  if (s->graph) cudaGraphDestroy(s->graph);
  s->exec = nullptr;
  s->graph = nullptr;
}

// Consecutive non-empty nodes from i that read the same input with the same
// K and block sizes (e.g. q/k/v, gate/up), at most kMaxSub.
int32_t group_at(const nf4_gemv_node* nodes, int32_t n_nodes, int32_t i) {
  int32_t n = 1;
  while (n < nf4::kMaxSub && i + n < n_nodes && nodes[i + n].N > 0 &&
         nodes[i + n].input == nodes[i].input && nodes[i + n].K == nodes[i].K &&
         nodes[i + n].blocksize == nodes[i].blocksize &&
         nodes[i + n].s2_blocksize == nodes[i].s2_blocksize)
    ++n;
  return n;
}

// One launch per node group, in node order, with programmatic dependent
// launch between consecutive kernels.
cudaError_t record_nodes(const nf4_gemv_node* nodes, int32_t n_nodes, int32_t batch,
                            const std::vector<nf4::QuantTensor>& ts,
                            const std::vector<nf4::YOut>& outs,
                            const std::vector<const uint16_t*>& xs, nf4_step_st* s,
                            cudaStream_t cs) {
  // Relaxed: first launches of a kernel may set its shared-memory limit.
  cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) return e;
  cudaError_t le = cudaSuccess;
  for (int32_t i = 0; i < n_nodes && le == cudaSuccess;) {
    if (nodes[i].N == 0) {
      ++i;
      continue;
    }
    int32_t n = group_at(nodes, n_nodes, i);
    bool done = false;
    if (n > 1 && nodes[i].K > 0) {
      int64_t Ns[nf4::kMaxSub];
      for (int32_t j = 0; j < n; ++j) Ns[j] = nodes[i + j].N;
      le = nf4::launch_gemv_group(&ts[size_t(i)], Ns, &outs[size_t(i)], int(n), nodes[i].K,
                                  xs[size_t(i)], batch, cs, &done);
    }
    if (!done) n = 1;
    if (le == cudaSuccess && !done)
      le = nf4::launch_gemv(ts[size_t(i)], nodes[i].N, nodes[i].K, xs[size_t(i)], batch,
                            outs[size_t(i)], cs);
    i += n;
  }
  const cudaError_t ee = cudaStreamEndCapture(cs, &s->graph);
  e = le != cudaSuccess ? le : ee;
  if (e == cudaSuccess && s->graph) e = cudaGraphInstantiate(&s->exec, s->graph, 0ull);
  return e;
}

}  // namespace

extern "C" {

nf4_status nf4_step_create(const nf4_gemv_node* nodes, int32_t n_nodes, const uint16_t* x,
                           int32_t batch, nf4_step_t* step) {
  if (!step) return NF4_ERR_NULL;
  *step = nullptr;
  if (n_nodes < 1) return NF4_ERR_INVALID_SIZE;
  if (!nodes) return NF4_ERR_NULL;
  // Validate every node before anything is recorded.
  const size_t count = static_cast<size_t>(n_nodes);
  std::vector<nf4::QuantTensor> ts(count);
  std::vector<nf4::YOut> outs(count);
  std::vector<const uint16_t*> xs(count);
  for (int32_t i = 0; i < n_nodes; ++i) {
    const nf4_gemv_node& n = nodes[i];
    const uint16_t* xi = x;
    if (n.input >= 0) {
      if (n.input >= i) return NF4_ERR_INVALID_SIZE;  // inputs come from earlier nodes
      const nf4_gemv_node& src = nodes[n.input];
      if (src.y_dtype != NF4_BF16) return NF4_ERR_UNSUPPORTED_DTYPE;
      if (src.N != n.K) return NF4_ERR_INVALID_SIZE;
      xi = static_cast<const uint16_t*>(src.y);
    } else if (n.input != -1) {
      return NF4_ERR_INVALID_SIZE;
    }
    const nf4_status st = nf4::check_gemv_args(n.packed, n.absmax_q, n.absmax2, n.code2, n.offset,
                                               n.N, n.K, n.blocksize, n.s2_blocksize, xi, batch,
                                               n.bias, n.y, n.y_dtype, &ts[size_t(i)],
                                               &outs[size_t(i)]);
    if (st != NF4_OK) return st;
    xs[size_t(i)] = xi;
  }

  nf4_step_st* s = new (std::nothrow) nf4_step_st;
  if (!s) return nf4::status_of(cudaErrorMemoryAllocation);
  s->n_nodes = n_nodes;
  cudaError_t e = cudaGetDevice(&s->device);
  cudaStream_t cs = nullptr;
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e == cudaSuccess) {
    e = record_nodes(nodes, n_nodes, batch, ts, outs, xs, s, cs);
    cudaStreamDestroy(cs);
  }
  if (e != cudaSuccess) {
    destroy_graph(s);
    delete s;
    return nf4::status_of(e);
  }
  *step = s;
  return NF4_OK;
}

nf4_status nf4_step_launch(nf4_step_t step, nf4_stream_t stream) {
  if (!step) return NF4_ERR_NULL;
  if (!step->exec) return NF4_OK;  // every node was empty
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return nf4::status_of(e);
  if (dev != step->device) return nf4::status_of(cudaErrorInvalidDevice);
  return nf4::status_of(cudaGraphLaunch(step->exec, reinterpret_cast<cudaStream_t>(stream)));
}

nf4_status nf4_step_kernel_count(nf4_step_t step, int32_t* count) {
  if (!step || !count) return NF4_ERR_NULL;
  *count = 0;
  if (!step->graph) return NF4_OK;
  size_t n = 0;
  cudaError_t e = cudaGraphGetNodes(step->graph, nullptr, &n);
  if (e != cudaSuccess) return nf4::status_of(e);
  std::vector<cudaGraphNode_t> nodes(n);
  if (n > 0) e = cudaGraphGetNodes(step->graph, nodes.data(), &n);
  if (e != cudaSuccess) return nf4::status_of(e);
  int32_t kernels = 0;
  for (size_t i = 0; i < n; ++i) {
    cudaGraphNodeType type;
    e = cudaGraphNodeGetType(nodes[i], &type);
    if (e != cudaSuccess) return nf4::status_of(e);
    if (type == cudaGraphNodeTypeKernel) ++kernels;
  }
  *count = kernels;
  return NF4_OK;
}

nf4_status nf4_step_destroy(nf4_step_t step) {
  if (!step) return NF4_OK;
  destroy_graph(step);
  delete step;
  return NF4_OK;
}

}  // extern "C"
