// A sequence of MatMulNBits projections as one CUDA graph (mnb_graph_*).
//
// A decode step runs its projections back to back; the page "Qwen3 CPU
// Inference Critical Path" (section "Prepared weight-only plan") gives one
// operator call per projection and a session executor around them. On the
// GPU the executor is a CUDA graph: the library records its own launches for
// the whole sequence once (stream capture on a private stream), and every
// step is then one graph launch on the caller's stream, optionally framed by
// the copy of the step's activations in and its outputs out. The launches
// are those of the single-call entry points (programmatic dependent launch
// included), so every projection computes exactly what that call computes.
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/mnb.h"
#include "mnb_common.cuh"
#include "mnb_launch.h"

struct mnb_graph_st {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int device = -1;
  int32_t calls = 0;    // library calls recorded
  int32_t kernels = 0;  // kernel nodes in the graph
};

namespace mnb {
namespace {

// One library call of the sequence: ops [first, first + count) fused over
// one activation row set (count > 1: mnb_matmul_grouped), a gated pair, or a
// single projection.
struct Call {
  int first, count;
  bool paired;
};

std::vector<Call> group_ops(const mnb_chain_op *ops, int32_t n, int64_t M) {
  std::vector<Call> calls;
  for (int j = 0; j < n;) {
    if (ops[j].packed_b_up) {
      calls.push_back({j, 1, true});
      ++j;
      continue;
    }
    int c = 1;
    while (M <= kGemvMaxM && c < kMaxGroup && j + c < n && !ops[j + c].packed_b_up &&
           ops[j + c].A == ops[j].A && ops[j + c].K == ops[j].K)
      ++c;
    calls.push_back({j, c, false});
    j += c;
  }
  return calls;
}

mnb_status record(const mnb_chain_op *ops, const std::vector<Call> &calls, int64_t M, int bs,
                  mnb_dtype a_dtype, mnb_dtype s_dtype, mnb_stream_t s) {
  for (const Call &c : calls) {
    const mnb_chain_op &o = ops[c.first];
    mnb_status st;
    if (c.paired) {
      st = mnb_matmul_gate_up(o.A, o.packed_b, o.packed_scales, o.packed_zp, o.bias,
                              o.packed_b_up, o.packed_scales_up, o.packed_zp_up, o.bias_up, M,
                              o.N, o.K, bs, o.Y, a_dtype, s_dtype, s);
    } else if (c.count == 1) {
      st = mnb_matmul(o.A, o.packed_b, o.packed_scales, o.packed_zp, o.bias, M, o.N, o.K, bs,
                      o.Y, a_dtype, s_dtype, s);
    } else {
      const void *b[kMaxGroup], *sc[kMaxGroup], *z[kMaxGroup];
      const float *bias[kMaxGroup];
      int64_t N[kMaxGroup];
      void *Y[kMaxGroup];
      for (int i = 0; i < c.count; ++i) {
        const mnb_chain_op &q = ops[c.first + i];
        b[i] = q.packed_b;
        sc[i] = q.packed_scales;
        z[i] = q.packed_zp;
        bias[i] = q.bias;
        N[i] = q.N;
        Y[i] = q.Y;
      }
      st = mnb_matmul_grouped(o.A, c.count, b, sc, o.packed_zp ? z : nullptr, bias, N, Y, M,
                              o.K, bs, a_dtype, s_dtype, s);
    }
    if (st != MNB_OK) return st;  // the call's own message stays in mnb_last_error_string
  }
  return MNB_OK;
}

}  // namespace
}  // namespace mnb

using namespace mnb;

extern "C" {

mnb_status mnb_graph_build(const mnb_chain_op *ops, int32_t n_ops, int64_t M, int block_size,
                           mnb_dtype a_dtype, mnb_dtype scale_dtype, mnb_graph *out) {
  if (!ops || !out) return MNB_ERR_NULL;
  *out = nullptr;
  if (n_ops < 1 || n_ops > 65536 || M < 1) return MNB_ERR_SHAPE;
  for (int j = 0; j < n_ops; ++j) {
    const mnb_chain_op &o = ops[j];
    if (!o.A || !o.Y || !o.packed_b || !o.packed_scales) return MNB_ERR_NULL;
    if (!o.packed_b_up && (o.packed_scales_up || o.packed_zp_up || o.bias_up))
      return MNB_ERR_NULL;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return MNB_ERR_CUDA;
  const std::vector<Call> calls = group_ops(ops, n_ops, M);
  // Record on a private stream: the caller's streams stay untouched, and the
  // thread-local capture mode leaves other threads' CUDA calls alone.
  cudaStream_t s = nullptr;
  e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) return MNB_ERR_CUDA;
  cudaGraph_t graph = nullptr;
  mnb_status st = MNB_OK;
  e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) {
    st = record(ops, calls, M, block_size, a_dtype, scale_dtype,
                reinterpret_cast<mnb_stream_t>(s));
    const cudaError_t ee = cudaStreamEndCapture(s, &graph);
    if (st == MNB_OK && ee != cudaSuccess) e = ee;
  }
  cudaStreamDestroy(s);
  if (st != MNB_OK || e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return st != MNB_OK ? st : MNB_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(graph);
    return MNB_ERR_CUDA;
  }
  size_t n_nodes = 0;
  cudaGraphGetNodes(graph, nullptr, &n_nodes);
  std::vector<cudaGraphNode_t> nodes(n_nodes);
  int kernels = 0;
  if (n_nodes && cudaGraphGetNodes(graph, nodes.data(), &n_nodes) == cudaSuccess)
    for (cudaGraphNode_t nd : nodes) {
      cudaGraphNodeType t;
      if (cudaGraphNodeGetType(nd, &t) == cudaSuccess && t == cudaGraphNodeTypeKernel)
        ++kernels;
    }
  mnb_graph g = new (std::nothrow) mnb_graph_st;
  if (!g) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    return MNB_ERR_UNSUPPORTED;
  }
  g->graph = graph;
  g->exec = exec;
  g->device = dev;
  g->calls = static_cast<int32_t>(calls.size());
  g->kernels = kernels;
  *out = g;
  return MNB_OK;
}

mnb_status mnb_graph_info(mnb_graph g, int32_t *calls, int32_t *kernels) {
  if (!g) return MNB_ERR_NULL;
  if (calls) *calls = g->calls;
  if (kernels) *kernels = g->kernels;
  return MNB_OK;
}

mnb_status mnb_graph_run(mnb_graph g, mnb_stream_t stream) {
  if (!g) return MNB_ERR_NULL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != g->device) return MNB_ERR_DEVICE;
  const cudaError_t e = cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MNB_OK : MNB_ERR_CUDA;
}

mnb_status mnb_graph_run_from_host(mnb_graph g, const void *in_host, void *in_dev,
                                   size_t in_bytes, const void *out_dev, void *out_host,
                                   size_t out_bytes, mnb_stream_t stream) {
  if (!g || (in_bytes && (!in_host || !in_dev)) || (out_bytes && (!out_dev || !out_host)))
    return MNB_ERR_NULL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != g->device) return MNB_ERR_DEVICE;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (in_bytes) e = cudaMemcpyAsync(in_dev, in_host, in_bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaGraphLaunch(g->exec, s);
  if (e == cudaSuccess && out_bytes)
    e = cudaMemcpyAsync(out_host, out_dev, out_bytes, cudaMemcpyDeviceToHost, s);
  return e == cudaSuccess ? MNB_OK : MNB_ERR_CUDA;
}

mnb_status mnb_graph_destroy(mnb_graph g) {
  if (!g) return MNB_ERR_NULL;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
  return MNB_OK;
}

}  // extern "C"
