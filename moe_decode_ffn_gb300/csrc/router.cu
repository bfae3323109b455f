// Fused router: split-K GEMV, grid-completion handshake, top-k + softmax.
//
// "perf(qwen3.6): fused router GEMV+top-k + folded residual-norm (decode)"
// (sparkinfer PR #273), Summary item 1: the router GEMV is split along the
// hidden dimension over thread blocks; each block writes its partial logits,
// then increments a completion counter that wraps back to zero (so a replayed
// CUDA graph needs no reset node); the block that completes the count selects
// the top-k with a tree of warp shuffles (value descending, ties to the lower
// expert index). The softmax over the selected logits is the workload's
// statement.
//
// GB300 layout: one warp per expert row and split; its slice of W_r is loaded
// into registers with 16-byte loads before the kernel waits on its
// predecessor (the router weights do not depend on it), so the weight read
// overlaps the previous kernel's tail. Partial sums go to a [T][S][E]
// workspace and the last block reduces them in split order: no float
// atomics, run-to-run deterministic.
#include <float.h>

#include "common.cuh"
#include "host.hpp"

namespace si {

constexpr int kRouterThreads = 256;
constexpr int kRowsPerCta = kRouterThreads / 32;
constexpr int kMaxTopK = 8;
constexpr int kMaxChunkTokens = 8;

struct RouterParams {
  const void *x;
  const void *w;
  int H, E, k, T;
  int S;             // splits of the hidden dimension
  int tc;            // tokens per chunk
  int cpc;           // CTAs per chunk = row_tiles * S
  int32_t *ids;
  float *wts;
  float *logits;     // nullable
  float *partials;   // [T][S][E]
  uint32_t *counters;
  uint32_t *flags;   // [n_chunks][cpc]
  uint32_t *status;
};

template <typename T> struct Vec;   // 16 bytes of weights
template <> struct Vec<__nv_bfloat16> { static constexpr int n = 8; };
template <> struct Vec<float> { static constexpr int n = 4; };

template <typename WT>
SI_DEV void unpack_w(const uint4 &u, float *v);
template <>
SI_DEV void unpack_w<__nv_bfloat16>(const uint4 &u, float *v) {
  v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
  v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
}
template <>
SI_DEV void unpack_w<float>(const uint4 &u, float *v) {
  v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
  v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
}

template <typename XT, int N>
SI_DEV void load_x(const XT *p, float *v) {
  if constexpr (sizeof(XT) == 2) {
    if constexpr (N == 8) {
      Load8<__nv_bfloat16>::run(p, v);
    } else {  // 4 bf16 = 8 bytes
      uint2 u = *reinterpret_cast<const uint2 *>(p);
      v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
    }
  } else {
    if constexpr (N == 8) {
      Load8<float>::run(p, v);
    } else {
      float4 a = *reinterpret_cast<const float4 *>(p);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    }
  }
}

// Total order used for selection: a before b iff a.v > b.v, or equal values
// and a.i < b.i (so -0 and +0 tie and go by index).
SI_DEV bool before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

SI_DEV void cmpx(float *v, int *id, int i, int j) {  // position i gets the earlier element
  if (before(v[j], id[j], v[i], id[i])) {
    float tv = v[i]; v[i] = v[j]; v[j] = tv;
    int ti = id[i]; id[i] = id[j]; id[j] = ti;
  }
}

// Bitonic sorting network on 8 (value, index) pairs, into selection order.
SI_DEV void sort8(float *v, int *id) {
#pragma unroll
  for (int size = 2; size <= 8; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          if ((i & size) == 0) cmpx(v, id, i, j);
          else cmpx(v, id, j, i);
        }
      }
    }
  }
}

// Butterfly over the 32 lanes: at each of the 5 levels a lane takes its
// partner's sorted 8, keeps the first 8 of the union (elementwise best of
// mine[j] and partner[7-j] is a bitonic sequence holding them) and re-sorts
// with 3 half-cleaner stages. The 16 shuffles of a level are independent.
SI_DEV void warp_top8(float *v, int *id) {
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    float pv[8];
    int pi[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      pv[j] = __shfl_xor_sync(0xffffffffu, v[j], m);
      pi[j] = __shfl_xor_sync(0xffffffffu, id[j], m);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (before(pv[7 - j], pi[7 - j], v[j], id[j])) {
        v[j] = pv[7 - j];
        id[j] = pi[7 - j];
      }
    }
#pragma unroll
    for (int stride = 4; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = i ^ stride;
        if (j > i) cmpx(v, id, i, j);
      }
    }
  }
}

template <typename XT, typename WT, int NCH>
__global__ void __launch_bounds__(kRouterThreads) router_topk_kernel(RouterParams p) {
  constexpr int VEC = Vec<WT>::n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / p.S, split = blockIdx.x % p.S;
  const int chunk = blockIdx.y;
  const int e = tile * kRowsPerCta + warp;
  const int KS = p.H / p.S;
  const int k0 = split * KS;
  const bool row_live = e < p.E;

  // Weight slice of this warp's row into registers (independent of the
  // predecessor kernel).
  uint4 wr[NCH];
  if (row_live) {
    const WT *wrow = static_cast<const WT *>(p.w) + static_cast<size_t>(e) * p.H + k0;
#pragma unroll
    for (int c = 0; c < NCH; ++c)
      wr[c] = __ldg(reinterpret_cast<const uint4 *>(wrow + (c * 32 + lane) * VEC));
  }
  grid_dep_wait();
  grid_dep_launch();

  const int t0 = chunk * p.tc;
  const int t1 = min(p.T, t0 + p.tc);
  if (row_live) {
    for (int t = t0; t < t1; ++t) {
      const XT *xs = static_cast<const XT *>(p.x) + static_cast<size_t>(t) * p.H + k0;
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        float wv[VEC], xv[VEC];
        unpack_w<WT>(wr[c], wv);
        load_x<XT, VEC>(xs + (c * 32 + lane) * VEC, xv);
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc = fmaf(wv[i], xv[i], acc);
      }
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
      if (lane == 0) p.partials[(static_cast<size_t>(t) * p.S + split) * p.E + e] = acc;
    }
  }

  // Completion handshake: publish partials, raise this block's flag, count.
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int me = blockIdx.x;
    atomicExch(&p.flags[static_cast<size_t>(chunk) * p.cpc + me], 1u);
    __threadfence();
    const unsigned prev = atomicInc(&p.counters[chunk], static_cast<unsigned>(p.cpc - 1));
    s_last = (prev == static_cast<unsigned>(p.cpc - 1)) ? 1 : (prev > static_cast<unsigned>(p.cpc - 1) ? 2 : 0);
  }
  __syncthreads();
  if (s_last == 2) {
    // The counter held a value it can never reach: the workspace was not
    // zeroed. Report it and poison this chunk's outputs rather than leave
    // stale ids in place.
    if (threadIdx.x == 0) record_status(p.status, SI_ERR_HANDSHAKE);
    for (int i = threadIdx.x; i < (min(p.T, chunk * p.tc + p.tc) - chunk * p.tc) * p.k; i += kRouterThreads) {
      p.ids[static_cast<size_t>(chunk) * p.tc * p.k + i] = -1;
      p.wts[static_cast<size_t>(chunk) * p.tc * p.k + i] = 0.f;
    }
    return;
  }
  if (!s_last) return;
  __threadfence();

  // Last block of this chunk: every flag must be up, else the counter was
  // not at zero when the run started (workspace not zeroed, or corrupted).
  int missing = 0;
  for (int i = threadIdx.x; i < p.cpc; i += kRouterThreads) {
    uint32_t *f = &p.flags[static_cast<size_t>(chunk) * p.cpc + i];
    if (__ldcg(f) != 1u) missing = 1;
    *f = 0u;
  }
  missing = __syncthreads_or(missing);
  if (missing) {
    if (threadIdx.x == 0) record_status(p.status, SI_ERR_HANDSHAKE);
    for (int i = threadIdx.x; i < (t1 - t0) * p.k; i += kRouterThreads) {
      p.ids[static_cast<size_t>(t0) * p.k + i] = -1;
      p.wts[static_cast<size_t>(t0) * p.k + i] = 0.f;
    }
    return;
  }

  // One warp per token: reduce partials in split order, select, softmax.
  for (int t = t0 + warp; t < t1; t += kRowsPerCta) {
    float v[8];
    int id[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int ex = lane + 32 * c;
      if (ex < p.E) {
        const float *pp = p.partials + static_cast<size_t>(t) * p.S * p.E + ex;
        float l = __ldcg(pp);
        for (int s = 1; s < p.S; ++s) l += __ldcg(pp + static_cast<size_t>(s) * p.E);
        if (p.logits) p.logits[static_cast<size_t>(t) * p.E + ex] = l;
        v[c] = l;
        id[c] = ex;
      } else {
        v[c] = -FLT_MAX;      // never selected: top_k <= n_experts
        id[c] = 0x7fffffff;
      }
    }
    sort8(v, id);
    warp_top8(v, id);
    if (lane == 0) {
      float ex[kMaxTopK];
      float sum = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxTopK; ++r) {
        if (r < p.k) {
          ex[r] = expf(v[r] - v[0]);
          sum += ex[r];
        }
      }
#pragma unroll
      for (int r = 0; r < kMaxTopK; ++r) {
        if (r < p.k) {
          p.ids[static_cast<size_t>(t) * p.k + r] = id[r];
          p.wts[static_cast<size_t>(t) * p.k + r] = __fdiv_rn(ex[r], sum);
        }
      }
    }
  }
}

RouterGeom router_geom(int n_experts, int hidden, int n_tokens) {
  RouterGeom g{};
  g.row_tiles = (n_experts + kRowsPerCta - 1) / kRowsPerCta;
  // Aim at ~2 blocks per SM of a 152-SM GB300; each lane keeps 1..8 16-byte
  // chunks of its row (bf16: hidden/S between 256 and 2048; fp32 halves it).
  const int target = 2 * 152;
  int S = 1;
  while (S * 2 * g.row_tiles <= target) S *= 2;
  const int s_min = (hidden + 1023) / 1024;   // fp32 weights: <= 8 chunks per lane
  const int s_max = hidden / 256;             // bf16 weights: >= 1 chunk per lane
  if (S < s_min) S = s_min;
  if (S > s_max) S = s_max;
  while (hidden % (S * 256) != 0 && S > 1) S /= 2;
  g.splits = S;
  g.ctas_per_chunk = g.row_tiles * S;
  g.tok_per_chunk = n_tokens < kMaxChunkTokens ? n_tokens : kMaxChunkTokens;
  if (g.tok_per_chunk < 1) g.tok_per_chunk = 1;
  g.n_chunks = (n_tokens + g.tok_per_chunk - 1) / g.tok_per_chunk;
  size_t off = sizeof(WsHeader);
  g.off_counters = off;
  off = round_up(off + sizeof(uint32_t) * g.n_chunks, 256);
  g.off_flags = off;
  off = round_up(off + sizeof(uint32_t) * static_cast<size_t>(g.n_chunks) * g.ctas_per_chunk, 256);
  g.off_partials = off;
  off = round_up(off + sizeof(float) * static_cast<size_t>(n_tokens) * S * n_experts, 256);
  g.bytes = off;
  return g;
}

template <typename XT, typename WT>
static cudaError_t launch_router_t(const RouterParams &p, int n_chunks, cudaStream_t s) {
  constexpr int VEC = Vec<WT>::n;
  const int nch = p.H / p.S / (32 * VEC);
  const dim3 grid(p.cpc, n_chunks), block(kRouterThreads);
  switch (nch) {
    case 1: return launch_pdl(router_topk_kernel<XT, WT, 1>, grid, block, 0, s, p);
    case 2: return launch_pdl(router_topk_kernel<XT, WT, 2>, grid, block, 0, s, p);
    case 4: return launch_pdl(router_topk_kernel<XT, WT, 4>, grid, block, 0, s, p);
    case 8: return launch_pdl(router_topk_kernel<XT, WT, 8>, grid, block, 0, s, p);
    default: return cudaErrorInvalidValue;
  }
}

template <typename XT, typename WT>
static cudaError_t preload_router_t() {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, router_topk_kernel<XT, WT, 1>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, router_topk_kernel<XT, WT, 2>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, router_topk_kernel<XT, WT, 4>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, router_topk_kernel<XT, WT, 8>);
  return e;
}

cudaError_t preload_router() {
  cudaError_t e = preload_router_t<__nv_bfloat16, __nv_bfloat16>();
  if (e == cudaSuccess) e = preload_router_t<float, float>();
  if (e == cudaSuccess) e = preload_router_t<float, __nv_bfloat16>();
  if (e == cudaSuccess) e = preload_router_t<__nv_bfloat16, float>();
  return e;
}

si_status router_launch(const void *x, si_dtype x_type, const void *w, si_dtype w_type, int hidden,
                        int n_experts, int top_k, int n_tokens, int32_t *ids, float *wts,
                        float *logits, void *ws, uint32_t *status, cudaStream_t s) {
  const RouterGeom g = router_geom(n_experts, hidden, n_tokens);
  uint8_t *base = static_cast<uint8_t *>(ws);
  RouterParams p{};
  p.x = x; p.w = w; p.H = hidden; p.E = n_experts; p.k = top_k; p.T = n_tokens;
  p.S = g.splits; p.tc = g.tok_per_chunk; p.cpc = g.ctas_per_chunk;
  p.ids = ids; p.wts = wts; p.logits = logits;
  p.partials = reinterpret_cast<float *>(base + g.off_partials);
  p.counters = reinterpret_cast<uint32_t *>(base + g.off_counters);
  p.flags = reinterpret_cast<uint32_t *>(base + g.off_flags);
  p.status = status;
  const int nch_bytes = hidden / g.splits * (w_type == SI_F32 ? 4 : 2) / 16 / 32;
  if (nch_bytes < 1 || nch_bytes > 8 || (nch_bytes & (nch_bytes - 1))) return SI_ERR_UNSUPPORTED;
  cudaError_t e;
  if (x_type == SI_BF16 && w_type == SI_BF16) e = launch_router_t<__nv_bfloat16, __nv_bfloat16>(p, g.n_chunks, s);
  else if (x_type == SI_F32 && w_type == SI_F32) e = launch_router_t<float, float>(p, g.n_chunks, s);
  else if (x_type == SI_F32 && w_type == SI_BF16) e = launch_router_t<float, __nv_bfloat16>(p, g.n_chunks, s);
  else if (x_type == SI_BF16 && w_type == SI_F32) e = launch_router_t<__nv_bfloat16, float>(p, g.n_chunks, s);
  else return SI_ERR_UNSUPPORTED;
  return cuda_status(e);
}

}  // namespace si

using namespace si;

extern "C" size_t si_moe_router_workspace_bytes(int n_experts, int hidden, int n_tokens) {
  if (n_experts < 1 || hidden < 256 || n_tokens < 1) return 0;
  return router_geom(n_experts, hidden, n_tokens).bytes;
}

extern "C" si_status si_moe_router_topk(const void *x, si_dtype x_type, const void *w_router,
                                        si_dtype w_type, int hidden, int n_experts, int top_k,
                                        int n_tokens, int32_t *topk_ids, float *topk_w,
                                        float *logits_out, void *workspace,
                                        size_t workspace_bytes, void *stream) {
  if (!x || !w_router || !topk_ids || !topk_w) return SI_ERR_INVALID_ARG;
  if (hidden < 256 || hidden % 256 != 0 || hidden > 16384) return SI_ERR_INVALID_ARG;
  if (n_experts < 8 || n_experts > 256 || top_k < 1 || top_k > kMaxTopK || top_k > n_experts ||
      n_tokens < 1)
    return SI_ERR_INVALID_ARG;
  if ((x_type != SI_BF16 && x_type != SI_F32) || (w_type != SI_BF16 && w_type != SI_F32))
    return SI_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w_router) || (reinterpret_cast<uintptr_t>(topk_ids) & 3u) ||
      (reinterpret_cast<uintptr_t>(topk_w) & 3u) ||
      (logits_out && (reinterpret_cast<uintptr_t>(logits_out) & 3u)))
    return SI_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) ||
      workspace_bytes < si_moe_router_workspace_bytes(n_experts, hidden, n_tokens))
    return SI_ERR_WORKSPACE;
  return router_launch(x, x_type, w_router, w_type, hidden, n_experts, top_k, n_tokens, topk_ids,
                       topk_w, logits_out, workspace, static_cast<uint32_t *>(workspace),
                       static_cast<cudaStream_t>(stream));
}
