// Library-level entry points: status strings, the whole-layer launcher and
// the layer stack captured as one CUDA graph.
//
// "perf(qwen3.6): fuse decode kernel launches - shared-expert + GDN
// conv/L2-norm" (sparkinfer PR #239), Summary: decode is CUDA-graph and
// launch bound, so every launch per layer costs time; the pages run the
// whole token as one captured graph ("perf(qwen3.6): fused router GEMV+top-k
// + folded residual-norm (decode)", PR #273, Summary item 1). A layer here is
// four kernels (router + top-k, gate/up, down, residual norm) chained with
// programmatic dependent launch, so each kernel's prologue (weights that do
// not depend on the previous kernel) overlaps its predecessor.
#include <stdio.h>

#include <mutex>
#include <new>

#include "common.cuh"
#include "host.hpp"

namespace si {

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

cudaError_t ensure_smem(const void *kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  static std::mutex mu;
  static const void *keys[256];
  static size_t vals[256];
  static int dev_of[256];
  static int n = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (keys[i] == kernel && dev_of[i] == dev && vals[i] >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (n < 256) {
    keys[n] = kernel;
    vals[n] = bytes;
    dev_of[n] = dev;
    ++n;
  }
  return cudaSuccess;
}

struct LayerGeom {
  size_t off_router, off_ffn, off_ids, off_wts, off_routed, off_shared, bytes;
};

static LayerGeom layer_geom(const si_moe_layer &L) {
  LayerGeom g{};
  size_t off = sizeof(WsHeader);
  g.off_router = off;
  off = round_up(off + router_geom(L.n_experts, L.hidden, 1).bytes, 256);
  g.off_ffn = off;
  off = round_up(off + ffn_geom(L).bytes, 256);
  g.off_ids = off;
  off = round_up(off + 8 * sizeof(int32_t), 256);
  g.off_wts = off;
  off = round_up(off + 8 * sizeof(float), 256);
  g.off_routed = off;
  off = round_up(off + static_cast<size_t>(L.hidden) * 2, 256);
  g.off_shared = off;
  off = round_up(off + static_cast<size_t>(L.hidden) * 2, 256);
  g.bytes = off;
  return g;
}

static si_status layer_check(const si_moe_layer &L) {
  const si_status st = ffn_check(L);
  if (st != SI_OK) return st;
  if (L.n_experts < 8 || !L.w_router || !L.w_norm || !(L.eps >= 0.f)) return SI_ERR_INVALID_ARG;
  if (L.router_type != SI_BF16 && L.router_type != SI_F32) return SI_ERR_UNSUPPORTED;
  if (!aligned16(L.w_router) || !aligned16(L.w_norm)) return SI_ERR_INVALID_ARG;
  return SI_OK;
}

// Enqueue one layer on `s` into workspace `ws` (layer_geom layout), device
// errors reported to `status`.
static si_status layer_enqueue(const si_moe_layer &L, const void *x, const void *residual,
                               void *sum_out, void *norm_out, int32_t *ids, float *wts,
                               void *routed, void *shared, void *ws, uint32_t *status,
                               cudaStream_t s) {
  const LayerGeom g = layer_geom(L);
  uint8_t *base = static_cast<uint8_t *>(ws);
  if (!ids) ids = reinterpret_cast<int32_t *>(base + g.off_ids);
  if (!wts) wts = reinterpret_cast<float *>(base + g.off_wts);
  if (!routed) routed = base + g.off_routed;
  if (!shared) shared = base + g.off_shared;
  si_status st = router_launch(x, SI_BF16, L.w_router, L.router_type, L.hidden, L.n_experts,
                               L.top_k, 1, ids, wts, nullptr, base + g.off_router, status, s);
  if (st != SI_OK) return st;
  st = ffn_launch(L, x, nullptr, ids, wts, routed, shared, base + g.off_ffn, status, s);
  if (st != SI_OK) return st;
  if (L.shared_inter > 0)
    return norm_launch(routed, shared, residual, L.w_norm, L.hidden, 1, L.eps, sum_out, norm_out,
                       nullptr, s);
  return norm_launch(routed, residual, nullptr, L.w_norm, L.hidden, 1, L.eps, sum_out, norm_out,
                     nullptr, s);
}

// Test kernel for the bounded wait: one block waits on an mbarrier whose
// expected bytes never arrive (no copy is issued), gives up after budget_ns
// and records SI_ERR_TIMEOUT.
__global__ void wait_timeout_kernel(uint64_t budget_ns, uint32_t *status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive_expect_tx(&bar, 16);
  __syncthreads();
  mbar_wait_bounded(&bar, 0, threadIdx.x == 0 ? status : nullptr, budget_ns);
}

}  // namespace si

using namespace si;

extern "C" si_status si_test_wait_timeout(uint64_t budget_ns, void *workspace, void *stream) {
  if (!workspace || !aligned256(workspace) || budget_ns > 2000000000ull) return SI_ERR_INVALID_ARG;
  return cuda_status(launch_pdl(wait_timeout_kernel, dim3(1), dim3(32), 0,
                                static_cast<cudaStream_t>(stream), budget_ns,
                                static_cast<uint32_t *>(workspace)));
}

struct si_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  int persistent;   // 1: one persistent kernel; 0: four kernels per layer and token
};

extern "C" const char *si_status_string(int status) {
  switch (status) {
    case SI_OK: return "SI_OK";
    case SI_ERR_INVALID_ARG: return "SI_ERR_INVALID_ARG: invalid argument";
    case SI_ERR_UNSUPPORTED: return "SI_ERR_UNSUPPORTED: shape or type combination not supported";
    case SI_ERR_WORKSPACE: return "SI_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case SI_ERR_CUDA: return "SI_ERR_CUDA: a CUDA runtime call failed";
    case SI_ERR_HANDSHAKE: return "SI_ERR_HANDSHAKE: completion counter inconsistent (workspace not zeroed?)";
    case SI_ERR_TIMEOUT: return "SI_ERR_TIMEOUT: a bounded device wait ran out";
    default: return "unknown si_status";
  }
}

extern "C" int si_version(void) { return (1 << 16) | 0; }

extern "C" size_t si_row_bytes(si_dtype type, int64_t k) {
  switch (type) {
    case SI_F32: return static_cast<size_t>(k) * 4;
    case SI_F16:
    case SI_BF16: return static_cast<size_t>(k) * 2;
    case SI_Q8_0: return k % 32 ? 0 : static_cast<size_t>(k / 32) * kQ80Bytes;
    case SI_Q8_1: return k % 32 ? 0 : static_cast<size_t>(k / 32) * kQ81Bytes;
    case SI_Q4_K: return k % 256 ? 0 : static_cast<size_t>(k / 256) * kQ4KBytes;
    case SI_Q5_K: return k % 256 ? 0 : static_cast<size_t>(k / 256) * kQ5KBytes;
    default: return 0;
  }
}

extern "C" size_t si_moe_layer_workspace_bytes(const si_moe_layer *L) {
  if (!L || layer_check(*L) != SI_OK) return 0;
  return layer_geom(*L).bytes;
}

extern "C" si_status si_moe_layer_decode(const si_moe_layer *L, const void *x, const void *residual,
                                         void *sum_out, void *norm_out, int32_t *topk_ids,
                                         float *topk_w, void *routed_out, void *shared_out,
                                         void *workspace, size_t workspace_bytes, void *stream) {
  if (!L || !x || !residual || !sum_out || !norm_out) return SI_ERR_INVALID_ARG;
  const si_status st = layer_check(*L);
  if (st != SI_OK) return st;
  if (!aligned16(x) || !aligned16(residual) || !aligned16(sum_out) || !aligned16(norm_out) ||
      (routed_out && !aligned16(routed_out)) || (shared_out && !aligned16(shared_out)) ||
      (topk_ids && (reinterpret_cast<uintptr_t>(topk_ids) & 3u)) ||
      (topk_w && (reinterpret_cast<uintptr_t>(topk_w) & 3u)))
    return SI_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < layer_geom(*L).bytes)
    return SI_ERR_WORKSPACE;
  return layer_enqueue(*L, x, residual, sum_out, norm_out, topk_ids, topk_w, routed_out, shared_out,
                       workspace, static_cast<uint32_t *>(workspace),
                       static_cast<cudaStream_t>(stream));
}

// Stack workspace: header, then per layer [layer workspace][sum bf16 H][norm bf16 H].
static size_t stack_layer_bytes(const si_moe_layer &L) {
  return round_up(layer_geom(L).bytes + 4 * static_cast<size_t>(L.hidden), 256);
}

extern "C" size_t si_moe_stack_workspace_bytes(const si_moe_layer *layers, int n_layers) {
  if (!layers || n_layers < 1) return 0;
  size_t off = sizeof(WsHeader);
  for (int l = 0; l < n_layers; ++l) {
    if (layer_check(layers[l]) != SI_OK) return 0;
    off += stack_layer_bytes(layers[l]);
  }
  if (stack_supported(layers, n_layers)) {
    const size_t pk = stack_workspace_bytes(layers, n_layers);
    if (pk > off) off = pk;
  }
  return off;
}

extern "C" si_status si_moe_stack_graph_create_mode(const si_moe_layer *layers, int n_layers,
                                                    int n_tokens, const void *x_in, void *y_out,
                                                    void *sum_out, int32_t *ids_out, void *workspace,
                                                    size_t workspace_bytes, int mode, void *stream,
                                                    si_graph **graph_out) {
  if (!layers || n_layers < 1 || n_tokens < 1 || !x_in || !y_out || !graph_out ||
      (mode != SI_STACK_AUTO && mode != SI_STACK_PER_LAYER && mode != SI_STACK_PERSISTENT))
    return SI_ERR_INVALID_ARG;
  *graph_out = nullptr;
  const int H = layers[0].hidden, k = layers[0].top_k;
  for (int l = 0; l < n_layers; ++l) {
    const si_status st = layer_check(layers[l]);
    if (st != SI_OK) return st;
    if (layers[l].hidden != H || layers[l].top_k != k) return SI_ERR_INVALID_ARG;
  }
  if (!aligned16(x_in) || !aligned16(y_out) || (sum_out && !aligned16(sum_out)) ||
      (ids_out && (reinterpret_cast<uintptr_t>(ids_out) & 3u)))
    return SI_ERR_INVALID_ARG;
  // The persistent kernel serves the layers stack_supported takes; the others
  // run as four kernels per layer. A forced persistent graph needs only the
  // persistent kernel's workspace.
  const bool can_persist = stack_supported(layers, n_layers);
  if (mode == SI_STACK_PERSISTENT && !can_persist) return SI_ERR_UNSUPPORTED;
  const size_t need = mode == SI_STACK_PERSISTENT ? stack_workspace_bytes(layers, n_layers)
                                                  : si_moe_stack_workspace_bytes(layers, n_layers);
  if (!workspace || !aligned256(workspace) || workspace_bytes < need) return SI_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (preload_router() != cudaSuccess || preload_ffn() != cudaSuccess ||
      preload_norm() != cudaSuccess || preload_stack() != cudaSuccess)
    return SI_ERR_CUDA;
  cudaStreamCaptureStatus cs;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return SI_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return SI_ERR_INVALID_ARG;
  const bool persistent = can_persist && mode != SI_STACK_PER_LAYER;
  if (persistent) {
    const si_status sp = stack_prepare(layers, n_layers, workspace, s);
    if (sp != SI_OK) return sp;
  }
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return SI_ERR_CUDA;

  uint8_t *base = static_cast<uint8_t *>(workspace);
  uint32_t *status = reinterpret_cast<uint32_t *>(base);
  si_status st = SI_OK;
  if (persistent) {
    st = stack_launch(layers, n_layers, n_tokens, x_in, y_out, sum_out, ids_out, workspace, s);
  } else {
    for (int t = 0; t < n_tokens && st == SI_OK; ++t) {
      const __nv_bfloat16 *xt = static_cast<const __nv_bfloat16 *>(x_in) + static_cast<size_t>(t) * H;
      const void *x = xt, *res = xt;
      size_t off = sizeof(WsHeader);
      for (int l = 0; l < n_layers && st == SI_OK; ++l) {
        const si_moe_layer &L = layers[l];
        uint8_t *lws = base + off;
        const size_t lb = layer_geom(L).bytes;
        void *sum = lws + lb;
        void *y = lws + lb + 2 * static_cast<size_t>(H);
        if (l == n_layers - 1) {
          y = static_cast<__nv_bfloat16 *>(y_out) + static_cast<size_t>(t) * H;
          if (sum_out) sum = static_cast<__nv_bfloat16 *>(sum_out) + static_cast<size_t>(t) * H;
        }
        int32_t *ids = ids_out ? ids_out + (static_cast<size_t>(t) * n_layers + l) * k : nullptr;
        st = layer_enqueue(L, x, res, sum, y, ids, nullptr, nullptr, nullptr, lws, status, s);
        x = y;
        res = sum;
        off += stack_layer_bytes(L);
      }
    }
  }
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(s, &graph);
  if (st != SI_OK || ec != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return st != SI_OK ? st : SI_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  if (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
    cudaGraphDestroy(graph);
    return SI_ERR_CUDA;
  }
  si_graph *g = new (std::nothrow) si_graph{graph, exec, persistent ? 1 : 0};
  if (!g) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    return SI_ERR_CUDA;
  }
  *graph_out = g;
  return SI_OK;
}

extern "C" si_status si_moe_stack_graph_create(const si_moe_layer *layers, int n_layers,
                                               int n_tokens, const void *x_in, void *y_out,
                                               void *sum_out, int32_t *ids_out, void *workspace,
                                               size_t workspace_bytes, void *stream,
                                               si_graph **graph_out) {
  return si_moe_stack_graph_create_mode(layers, n_layers, n_tokens, x_in, y_out, sum_out, ids_out,
                                        workspace, workspace_bytes, SI_STACK_AUTO, stream,
                                        graph_out);
}

// ---------------------------------------------------------------------------
// Batched layer: n_tokens tokens routed independently, their experts grouped
// (si_moe_ffn_batched), then the residual fold of every row.
// ---------------------------------------------------------------------------
namespace si {

struct BLayerGeom {
  size_t off_router, off_ffn, off_ids, off_wts, off_routed, bytes;
};

static BLayerGeom blayer_geom(const si_moe_layer &L, int T) {
  BLayerGeom g{};
  size_t off = sizeof(WsHeader);
  auto take = [&](size_t &field, size_t bytes) {
    field = off;
    off = round_up(off + bytes, 256);
  };
  take(g.off_router, router_geom(L.n_experts, L.hidden, T).bytes);
  take(g.off_ffn, batched_workspace_bytes(L, T));
  take(g.off_ids, sizeof(int32_t) * static_cast<size_t>(T) * L.top_k);
  take(g.off_wts, sizeof(float) * static_cast<size_t>(T) * L.top_k);
  take(g.off_routed, 2u * static_cast<size_t>(T) * L.hidden);
  g.bytes = off;
  return g;
}

static si_status blayer_check(const si_moe_layer &L, int T) {
  const si_status st = batched_validate(L, T);
  if (st != SI_OK) return st;
  if (L.n_experts < 8 || !L.w_router || !L.w_norm || !(L.eps >= 0.f)) return SI_ERR_INVALID_ARG;
  if (L.router_type != SI_BF16 && L.router_type != SI_F32) return SI_ERR_UNSUPPORTED;
  if (!aligned16(L.w_router) || !aligned16(L.w_norm) || L.hidden > 16384) return SI_ERR_INVALID_ARG;
  return SI_OK;
}

static si_status blayer_enqueue(const si_moe_layer &L, int T, int mode, const void *x,
                                const void *residual, void *sum_out, void *norm_out, int32_t *ids,
                                float *wts, void *routed, void *ws, uint32_t *status, cudaStream_t s) {
  const BLayerGeom g = blayer_geom(L, T);
  uint8_t *base = static_cast<uint8_t *>(ws);
  if (!ids) ids = reinterpret_cast<int32_t *>(base + g.off_ids);
  if (!wts) wts = reinterpret_cast<float *>(base + g.off_wts);
  if (!routed) routed = base + g.off_routed;
  si_status st = router_launch(x, SI_BF16, L.w_router, L.router_type, L.hidden, L.n_experts,
                               L.top_k, T, ids, wts, nullptr, base + g.off_router, status, s);
  if (st != SI_OK) return st;
  const BatchedNorm nm{residual, L.w_norm, L.eps, sum_out, norm_out};
  return batched_launch(&L, T, mode, x, ids, wts, routed, base + g.off_ffn, status, s, &nm);
}

// Batched stack workspace: header, then per layer [layer workspace][sum bf16 T x H][norm bf16 T x H].
static size_t bstack_layer_bytes(const si_moe_layer &L, int T) {
  return round_up(blayer_geom(L, T).bytes + 4 * static_cast<size_t>(T) * L.hidden, 256);
}

}  // namespace si

extern "C" size_t si_moe_layer_batched_workspace_bytes(const si_moe_layer *L, int n_tokens) {
  if (!L || blayer_check(*L, n_tokens) != SI_OK) return 0;
  return blayer_geom(*L, n_tokens).bytes;
}

extern "C" si_status si_moe_layer_decode_batched(const si_moe_layer *L, int n_tokens, int mode,
                                                 const void *x, const void *residual, void *sum_out,
                                                 void *norm_out, int32_t *topk_ids, float *topk_w,
                                                 void *routed_out, void *workspace,
                                                 size_t workspace_bytes, void *stream) {
  if (!L || !x || !residual || !sum_out || !norm_out) return SI_ERR_INVALID_ARG;
  if (mode != SI_FFN_AUTO && mode != SI_FFN_INT8 && mode != SI_FFN_TENSOR) return SI_ERR_INVALID_ARG;
  const si_status st = blayer_check(*L, n_tokens);
  if (st != SI_OK) return st;
  if (!aligned16(x) || !aligned16(residual) || !aligned16(sum_out) || !aligned16(norm_out) ||
      (routed_out && !aligned16(routed_out)) ||
      (topk_ids && (reinterpret_cast<uintptr_t>(topk_ids) & 3u)) ||
      (topk_w && (reinterpret_cast<uintptr_t>(topk_w) & 3u)))
    return SI_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < blayer_geom(*L, n_tokens).bytes)
    return SI_ERR_WORKSPACE;
  return blayer_enqueue(*L, n_tokens, mode, x, residual, sum_out, norm_out, topk_ids, topk_w,
                        routed_out, workspace, static_cast<uint32_t *>(workspace),
                        static_cast<cudaStream_t>(stream));
}

extern "C" size_t si_moe_stack_batched_workspace_bytes(const si_moe_layer *layers, int n_layers,
                                                       int n_tokens) {
  if (!layers || n_layers < 1) return 0;
  size_t off = sizeof(WsHeader);
  for (int l = 0; l < n_layers; ++l) {
    if (blayer_check(layers[l], n_tokens) != SI_OK) return 0;
    off += bstack_layer_bytes(layers[l], n_tokens);
  }
  if (n_tokens == 1 && stack_supported(layers, n_layers)) {   // the automatic mode's persistent kernel
    const size_t pk = stack_workspace_bytes(layers, n_layers);
    if (pk > off) off = pk;
  }
  return off;
}

extern "C" si_status si_moe_stack_graph_create_batched(const si_moe_layer *layers, int n_layers,
                                                       int n_tokens, int mode, const void *x_in,
                                                       void *y_out, void *sum_out, int32_t *ids_out,
                                                       void *workspace, size_t workspace_bytes,
                                                       void *stream, si_graph **graph_out) {
  if (!layers || n_layers < 1 || n_tokens < 1 || !x_in || !y_out || !graph_out) return SI_ERR_INVALID_ARG;
  if (mode != SI_FFN_AUTO && mode != SI_FFN_INT8 && mode != SI_FFN_TENSOR) return SI_ERR_INVALID_ARG;
  *graph_out = nullptr;
  const int H = layers[0].hidden, k = layers[0].top_k;
  for (int l = 0; l < n_layers; ++l) {
    const si_status st = blayer_check(layers[l], n_tokens);
    if (st != SI_OK) return st;
    if (layers[l].hidden != H || layers[l].top_k != k) return SI_ERR_INVALID_ARG;
  }
  if (!aligned16(x_in) || !aligned16(y_out) || (sum_out && !aligned16(sum_out)) ||
      (ids_out && (reinterpret_cast<uintptr_t>(ids_out) & 3u)))
    return SI_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) ||
      workspace_bytes < si_moe_stack_batched_workspace_bytes(layers, n_layers, n_tokens))
    return SI_ERR_WORKSPACE;
  // one token: the same results (every path gives every token the bits of
  // the single-token layer) from the persistent kernel when it takes the
  // layers; the ids layout [n_layers][1][k] is the persistent one's [1][n_layers][k]
  if (mode == SI_FFN_AUTO && n_tokens == 1 && stack_supported(layers, n_layers))
    return si_moe_stack_graph_create_mode(layers, n_layers, 1, x_in, y_out, sum_out, ids_out, workspace,
                                          workspace_bytes, SI_STACK_PERSISTENT, stream, graph_out);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (preload_router() != cudaSuccess || preload_batched() != cudaSuccess || preload_norm() != cudaSuccess)
    return SI_ERR_CUDA;
  cudaStreamCaptureStatus cs;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return SI_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return SI_ERR_INVALID_ARG;
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return SI_ERR_CUDA;
  uint8_t *base = static_cast<uint8_t *>(workspace);
  uint32_t *status = reinterpret_cast<uint32_t *>(base);
  si_status st = SI_OK;
  const void *x = x_in, *res = x_in;
  size_t off = sizeof(WsHeader);
  for (int l = 0; l < n_layers && st == SI_OK; ++l) {
    const si_moe_layer &L = layers[l];
    uint8_t *lws = base + off;
    const size_t lb = blayer_geom(L, n_tokens).bytes;
    void *sum = lws + lb;
    void *y = lws + lb + 2 * static_cast<size_t>(n_tokens) * H;
    if (l == n_layers - 1) {
      y = y_out;
      if (sum_out) sum = sum_out;
    }
    int32_t *ids = ids_out ? ids_out + static_cast<size_t>(l) * n_tokens * k : nullptr;
    st = blayer_enqueue(L, n_tokens, mode, x, res, sum, y, ids, nullptr, nullptr, lws, status, s);
    x = y;
    res = sum;
    off += bstack_layer_bytes(L, n_tokens);
  }
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(s, &graph);
  if (st != SI_OK || ec != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return st != SI_OK ? st : SI_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  if (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
    cudaGraphDestroy(graph);
    return SI_ERR_CUDA;
  }
  si_graph *g = new (std::nothrow) si_graph{graph, exec, 0};
  if (!g) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    return SI_ERR_CUDA;
  }
  *graph_out = g;
  return SI_OK;
}

extern "C" int si_graph_is_persistent(const si_graph *graph) {
  return graph ? graph->persistent : -1;
}

extern "C" si_status si_graph_launch(si_graph *graph, void *stream) {
  if (!graph) return SI_ERR_INVALID_ARG;
  return cuda_status(cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)));
}

extern "C" void si_graph_destroy(si_graph *graph) {
  if (!graph) return;
  cudaGraphExecDestroy(graph->exec);
  cudaGraphDestroy(graph->graph);
  delete graph;
}

extern "C" si_status si_workspace_status(const void *workspace, void *stream, int *status_out) {
  if (!workspace || !status_out) return SI_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SI_ERR_CUDA;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SI_ERR_CUDA;
  if (cudaMemsetAsync(const_cast<void *>(workspace), 0, sizeof(uint32_t), s) != cudaSuccess)
    return SI_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SI_ERR_CUDA;
  *status_out = static_cast<int>(v);
  return SI_OK;
}
