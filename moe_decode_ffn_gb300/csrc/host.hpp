// Host-side helpers shared by the C-ABI translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/si_moe.h"

namespace si {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Number of SMs of the current device (queried once per device).
int sm_count();

// Launch with programmatic stream serialization allowed: the kernel may
// start before its predecessor in the stream has finished and must call
// griddepcontrol.wait before reading that predecessor's outputs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline si_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SI_OK : SI_ERR_CUDA; }

// Raise a kernel's dynamic shared memory limit (once per kernel and size;
// the limit is remembered so that launches inside stream capture issue no
// other runtime call).
cudaError_t ensure_smem(const void *kernel, size_t bytes);
template <typename K>
inline cudaError_t allow_smem(K kernel, size_t bytes) {
  return ensure_smem(reinterpret_cast<const void *>(kernel), bytes);
}

// The routed down format of a layer (down_type 0 = expert_type).
inline si_dtype down_type_of(const si_moe_layer &L) {
  return L.down_type == SI_F32 ? L.expert_type : L.down_type;
}

// Load every kernel of the library (called before stream capture starts).
cudaError_t preload_router();
cudaError_t preload_ffn();
cudaError_t preload_norm();

// ---- persistent layer-stack kernel (stack.cu)
// Whether one cooperative launch can run these layers (shapes, formats, SM
// count, shared memory); the workspace it needs; copying the per-layer pointer
// table into that workspace (synchronous, outside capture); the launch.
bool stack_supported(const si_moe_layer *layers, int n_layers);
size_t stack_workspace_bytes(const si_moe_layer *layers, int n_layers);
si_status stack_prepare(const si_moe_layer *layers, int n_layers, void *ws, cudaStream_t s);
si_status stack_launch(const si_moe_layer *layers, int n_layers, int n_tokens, const void *x_in,
                       void *y_out, void *sum_out, int32_t *ids_out, void *ws, cudaStream_t s);
cudaError_t preload_stack();

// ---- router geometry (depends only on the shapes, so the workspace size does too)
struct RouterGeom {
  int row_tiles;     // ceil(E / 8): one warp per expert row
  int splits;        // S: hidden dimension split over thread blocks
  int ctas_per_chunk;
  int tok_per_chunk;
  int n_chunks;
  size_t off_counters, off_flags, off_partials, bytes;
};
RouterGeom router_geom(int n_experts, int hidden, int n_tokens);

// Router on explicit workspace pieces (also used inside the layer launcher).
si_status router_launch(const void *x, si_dtype x_type, const void *w, si_dtype w_type, int hidden,
                        int n_experts, int top_k, int n_tokens, int32_t *ids, float *wts,
                        float *logits, void *ws, uint32_t *status, cudaStream_t s);

// ---- expert FFN workspace (h activations between gate/up and down)
struct FfnGeom {
  int n_slots;         // top_k + (shared ? 1 : 0)
  int n_units;         // 32-row units of h over all slots
  int down_rows;       // output rows per down thread block
  int down_ctas;
  size_t off_hq, off_hd, off_hs, off_hf, bytes;
};
FfnGeom ffn_geom(const si_moe_layer &L);
si_status ffn_check(const si_moe_layer &L);
// e0, e1: the routed experts computed ([0, E) by default: e1 < 0); slot_y
// non-null: per-slot fp32 outputs [k][H] instead of the combined `routed`.
si_status ffn_launch(const si_moe_layer &L, const void *x, const void *x_q8_1, const int32_t *ids,
                     const float *wts, void *routed, void *shared, void *ws, uint32_t *status,
                     cudaStream_t s, bool gateup_only = false, int e0 = 0, int e1 = -1,
                     float *slot_y = nullptr);

// ---- batched routed FFN (batched.cu): shape check, workspace, enqueue
si_status batched_validate(const si_moe_layer &L, int n_tokens);
size_t batched_workspace_bytes(const si_moe_layer &L, int n_tokens);
// The layer's residual norm taken into the combine step (batched layer):
// sum = bf16(routed + residual), norm = RMSNorm(sum) * w_norm.
struct BatchedNorm {
  const void *residual, *w_norm;
  float eps;
  void *sum_out, *norm_out;
};
si_status batched_launch(const si_moe_layer *L, int n_tokens, int mode, const void *x,
                         const int32_t *topk_ids, const float *topk_w, void *routed_out,
                         void *workspace, uint32_t *status, cudaStream_t s,
                         const BatchedNorm *norm = nullptr);
cudaError_t preload_batched();

// ---- test export of the batched helpers' integer block sums (batched.cu)
si_status batched_test_dots(const void *w, int rows, int k, const void *a, int n_vec, int halves,
                            int32_t *out, cudaStream_t s);

// ---- residual norm
si_status norm_launch(const void *a, const void *b, const void *c, const void *w, int n, int rows,
                      float eps, void *sum_out, void *norm_out, void *q8_out, cudaStream_t s);

}  // namespace si
