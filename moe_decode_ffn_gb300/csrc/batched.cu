// Batched tokens with per-token routing: grouped experts.
//
// T tokens route independently (top-k ids and weights per token). The
// (token, rank) pairs are grouped by expert so that each selected expert's
// weight rows are read from HBM once and reused for all of its tokens. This
// case is not on the pages (every measurement there is at batch 1); it
// follows the same per-token arithmetic as the single-token path:
//   h = silu(G_e x_t) * (U_e x_t),  y = D_e h,  routed_t = sum_r w_{t,r} y_{t,r}
// ("perf(qwen3.6): fuse decode kernel launches - shared-expert + GDN
// conv/L2-norm", Summary item 1; "Q4_K shared-expert FFN kernels +
// Q8_0/Q5_K->Q4_K requant of the MoE FFN stage", Summary: Q8_1 activations,
// int8 dot products).
//
// Kernels (integer mode, Q4_K experts, no shared expert):
//  prep    block 0 groups the pairs by expert (counts, offsets, stable order
//          by token, the list of active experts); the other blocks quantise
//          every token's x once into a Q8_1 tile record.
//  gate/up one block per (active expert, 32-row unit of h): 32 gate + 32 up
//          rows by TMA bulk copy, the expert's token tiles by bulk copy, h of
//          every token, then Q8_1 of each token's 32 values of h.
//  down    one block per (active expert, 32 output rows): the rows once, then
//          y = D_e h for each of the expert's pairs (fp32 per pair).
//  combine routed[t][j] = sum_r w[t][r] * y[pair(t, r)][j] in rank order.
#include "common.cuh"
#include "host.hpp"

namespace si {

constexpr int kBatchedMaxExperts = 256;
constexpr int kPrepThreads = 512;
constexpr int kGuBThreads = 512;
constexpr int kDownBThreads = 256;
constexpr int kTokChunk = 16;        // token tiles resident per gate/up block at once
constexpr int kDownRows = 32;        // output rows per down block

// Size of one token's Q8_1 tile record: codes at the padded super-block
// stride, then d and s (fp32) per 32-block; a multiple of 16 bytes.
static __host__ __device__ inline int tile_record_bytes(int n) {
  return (n / 256) * kActSbStride + 2 * (n / 32) * 4;
}

struct BatchedParams {
  const __nv_bfloat16 *x;    // [T][H]
  const int32_t *ids;        // [T][k]
  const float *wts;          // [T][k]
  int T, H, E, k, I;
  const uint8_t *wg, *wu, *wd;
  int rb_gu, rb_d;           // row bytes: gate/up rows (H wide), down rows (I wide)
  // workspace
  int *count;                // [E]
  int *offset;               // [E + 1]
  int *active;               // [E] active expert ids, ascending
  int *n_active;             // [1]
  int *pair_token;           // [T*k] token of each grouped pair
  int *pair_of;              // [T*k] grouped position of pair (t, r)
  uint8_t *xrec;             // [T][tile_record_bytes(H)]
  uint8_t *hrec;             // [T*k][tile_record_bytes(I)]
  float *y;                  // [T*k][H]
  __nv_bfloat16 *routed;     // [T][H]
  uint32_t *status;
};

SI_DEV ActTile tile_at(uint8_t *rec, int n) {
  ActTile t;
  t.qs = rec;
  t.d = reinterpret_cast<float *>(rec + (n / 256) * kActSbStride);
  t.s = t.d + n / 32;
  return t;
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPrepThreads) batched_prep_kernel(BatchedParams p) {
  grid_dep_wait();
  grid_dep_launch();
  if (blockIdx.x > 0) {
    // Token tiles: block b quantises token b - 1.
    const int t = blockIdx.x - 1;
    if (t < p.T) {
      ActTile tile = tile_at(p.xrec + static_cast<size_t>(t) * tile_record_bytes(p.H), p.H);
      quantize_to_tile<__nv_bfloat16>(p.x + static_cast<size_t>(t) * p.H, p.H, tile);
    }
    return;
  }
  __shared__ int s_cnt[kBatchedMaxExperts];
  __shared__ int s_off[kBatchedMaxExperts + 1];
  __shared__ int s_e[1024];
  const int P = p.T * p.k;
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  for (int q = threadIdx.x; q < P; q += blockDim.x) {
    int e = p.ids[q];
    if (e < 0 || e >= p.E) {
      record_status(p.status, SI_ERR_INVALID_ARG);
      e = 0;
    }
    if (q < 1024) s_e[q] = e;
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0, na = 0;
    for (int e = 0; e < p.E; ++e) {
      s_off[e] = acc;
      acc += s_cnt[e];
      if (s_cnt[e] > 0) p.active[na++] = e;
    }
    s_off[p.E] = acc;
    *p.n_active = na;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= p.E; e += blockDim.x) {
    p.offset[e] = s_off[e];
    if (e < p.E) p.count[e] = s_cnt[e];
  }
  // Stable position of pair q inside its expert: pairs of that expert with a
  // smaller index come first (token order, then rank order).
  for (int q = threadIdx.x; q < P; q += blockDim.x) {
    const int e = s_e[q];
    int before = 0;
    for (int j = 0; j < q; ++j) before += (s_e[j] == e);
    const int pos = s_off[e] + before;
    p.pair_of[q] = pos;
    p.pair_token[pos] = q / p.k;
  }
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kGuBThreads, 1) gateup_grouped_kernel(BatchedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int units = p.I / 32;
  const int nsb = p.H / kQKK;
  const int xrb = tile_record_bytes(p.H);
  const int hrb = tile_record_bytes(p.I);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);        // 4 weight groups + 1 tokens
  float *h_s = reinterpret_cast<float *>(smem + 64);          // [kTokChunk][32]
  uint8_t *xt = smem + 64 + kTokChunk * 32 * 4;               // [kTokChunk][xrb]
  uint8_t *wbuf = xt + kTokChunk * xrb;                       // gate [32][rb], up [32][rb]
  grid_dep_wait();
  grid_dep_launch();
  const int na = __ldcg(p.n_active);
  if (static_cast<int>(blockIdx.x) >= na * units) return;
  const int e = __ldcg(p.active + blockIdx.x / units);
  const int unit = blockIdx.x % units;
  const int n_e = __ldcg(p.count + e), p0 = __ldcg(p.offset + e);
  const int rb = p.rb_gu;
  uint8_t *gate_buf = wbuf, *up_buf = wbuf + 32 * rb;
  if (threadIdx.x == 0) {
    for (int g = 0; g < 5; ++g) mbar_init(&bars[g], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_first();
    const size_t row0 = static_cast<size_t>(e) * p.I + static_cast<size_t>(unit) * 32;
    const uint32_t bytes = 8u * rb;
    for (int g = 0; g < 4; ++g) {
      mbar_arrive_expect_tx(&bars[g], 2 * bytes);
      bulk_g2s_evict_first(gate_buf + 8 * g * rb, p.wg + (row0 + 8 * g) * rb, bytes, &bars[g], pol);
      bulk_g2s_evict_first(up_buf + 8 * g * rb, p.wu + (row0 + 8 * g) * rb, bytes, &bars[g], pol);
    }
  }
  const int pr = threadIdx.x >> 4, m = (threadIdx.x >> 3) & 1, lane8 = threadIdx.x & 7;
  const uint8_t *row = (m ? up_buf : gate_buf) + pr * rb;
  uint32_t phase = 0;
  bool weights_ready = false;
  for (int c0 = 0; c0 < n_e; c0 += kTokChunk) {
    const int nc = min(kTokChunk, n_e - c0);
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(&bars[4], nc * xrb);
      for (int i = 0; i < nc; ++i) {
        const int t = __ldcg(p.pair_token + p0 + c0 + i);
        bulk_g2s(xt + i * xrb, p.xrec + static_cast<size_t>(t) * xrb, xrb, &bars[4]);
      }
    }
    mbar_wait_bounded(&bars[4], phase, p.status);
    phase ^= 1u;
    if (!weights_ready) {
      mbar_wait_bounded(&bars[pr >> 3], 0, p.status);
      weights_ready = true;
    }
    for (int i = 0; i < nc; ++i) {
      const ActTile a = tile_at(xt + i * xrb, p.H);
      float acc = 0.f;
      for (int sb = lane8; sb < nsb; sb += 8)
        acc += q4k_sb_dot(reinterpret_cast<const uint4 *>(row + sb * kQ4KBytes),
                          reinterpret_cast<const uint4 *>(a.qs + sb * kActSbStride), a.d + 8 * sb,
                          a.s + 8 * sb);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      const float u = __shfl_xor_sync(0xffffffffu, acc, 8);
      if ((threadIdx.x & 15) == 0) h_s[i * 32 + pr] = __fdiv_rn(acc, 1.f + expf(-acc)) * u;
    }
    __syncthreads();
    // Q8_1 of each token's 32 values of h: warp w encodes tokens w, w+16, ...
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < nc; i += kGuBThreads / 32) {
      uint16_t d16, s16;
      const int q = q8_1_encode_warp(h_s[i * 32 + lane], d16, s16);
      ActTile h = tile_at(p.hrec + static_cast<size_t>(p0 + c0 + i) * hrb, p.I);
      const int j0 = unit * 32;   // element offset of this unit inside the pair's h
      h.qs[(j0 / kQKK) * kActSbStride + j0 % kQKK + lane] = static_cast<uint8_t>(q);
      if (lane == 0) {
        h.d[j0 / 32] = half_bits_to_float(d16);
        h.s[j0 / 32] = half_bits_to_float(s16);
      }
    }
    __syncthreads();   // h_s and the token tiles are reused by the next chunk
  }
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kDownBThreads) down_grouped_kernel(BatchedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tiles = p.H / kDownRows;
  const int nsb = p.I / kQKK;
  const int P = 2 * nsb;                 // half super-block pieces per row
  const int hrb = tile_record_bytes(p.I);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);           // weights, tokens
  float *part = reinterpret_cast<float *>(smem + 64);            // [kDownRows][P <= 32]
  uint8_t *ht = smem + 64 + kDownRows * 32 * 4;                  // [kTokChunk][hrb]
  uint8_t *wbuf = ht + kTokChunk * hrb;                          // [kDownRows][rb_d]
  grid_dep_wait();
  grid_dep_launch();
  const int na = __ldcg(p.n_active);
  if (static_cast<int>(blockIdx.x) >= na * tiles) return;
  const int e = __ldcg(p.active + blockIdx.x / tiles);
  const int j0 = (blockIdx.x % tiles) * kDownRows;
  const int n_e = __ldcg(p.count + e), p0 = __ldcg(p.offset + e);
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t bytes = static_cast<uint32_t>(kDownRows) * p.rb_d;
    mbar_arrive_expect_tx(&bars[0], bytes);
    bulk_g2s_evict_first(wbuf, p.wd + (static_cast<size_t>(e) * p.H + j0) * p.rb_d, bytes, &bars[0],
                         policy_evict_first());
  }
  uint32_t phase = 0;
  bool weights_ready = false;
  for (int c0 = 0; c0 < n_e; c0 += kTokChunk) {
    const int nc = min(kTokChunk, n_e - c0);
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(&bars[1], nc * hrb);
      bulk_g2s(ht, p.hrec + static_cast<size_t>(p0 + c0) * hrb, nc * hrb, &bars[1]);
    }
    mbar_wait_bounded(&bars[1], phase, p.status);
    phase ^= 1u;
    if (!weights_ready) {
      mbar_wait_bounded(&bars[0], 0, p.status);
      weights_ready = true;
    }
    for (int i = 0; i < nc; ++i) {
      const ActTile h = tile_at(ht + i * hrb, p.I);
      for (int u = threadIdx.x; u < kDownRows * P; u += blockDim.x) {
        const int jl = u / P, q = u % P, sb = q >> 1;
        part[jl * P + q] = q4k_half_dot(
            reinterpret_cast<const uint4 *>(wbuf + jl * p.rb_d + sb * kQ4KBytes),
            reinterpret_cast<const uint4 *>(h.qs + sb * kActSbStride), h.d + 8 * sb, h.s + 8 * sb,
            q & 1);
      }
      __syncthreads();
      if (threadIdx.x < kDownRows) {
        float y = 0.f;
        for (int q = 0; q < P; ++q) y += part[threadIdx.x * P + q];
        p.y[static_cast<size_t>(p0 + c0 + i) * p.H + j0 + threadIdx.x] = y;
      }
      __syncthreads();
    }
  }
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(BatchedParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= p.T || j >= p.H) return;
  float acc = 0.f;
  for (int r = 0; r < p.k; ++r) {
    const int q = __ldcg(p.pair_of + t * p.k + r);
    acc = fmaf(__ldcg(p.wts + t * p.k + r), __ldcg(p.y + static_cast<size_t>(q) * p.H + j), acc);
  }
  p.routed[static_cast<size_t>(t) * p.H + j] = __float2bfloat16_rn(acc);
}

// ---------------------------------------------------------------------------
struct BatchedGeom {
  size_t off_count, off_offset, off_active, off_nactive, off_pair_token, off_pair_of, off_xrec,
      off_hrec, off_y, bytes;
};

static BatchedGeom batched_geom(const si_moe_layer &L, int T) {
  BatchedGeom g{};
  const size_t P = static_cast<size_t>(T) * L.top_k;
  size_t off = sizeof(WsHeader);
  auto take = [&](size_t &field, size_t bytes) {
    field = off;
    off = round_up(off + bytes, 256);
  };
  take(g.off_count, 4u * L.n_experts);
  take(g.off_offset, 4u * (L.n_experts + 1));
  take(g.off_active, 4u * L.n_experts);
  take(g.off_nactive, 4);
  take(g.off_pair_token, 4 * P);
  take(g.off_pair_of, 4 * P);
  take(g.off_xrec, static_cast<size_t>(T) * tile_record_bytes(L.hidden));
  take(g.off_hrec, P * tile_record_bytes(L.inter));
  take(g.off_y, P * L.hidden * 4);
  g.bytes = off;
  return g;
}

static si_status batched_check(const si_moe_layer &L, int T) {
  if (T < 1 || T > 4096) return SI_ERR_INVALID_ARG;
  if (L.hidden < 256 || L.hidden % 256 || L.hidden > 8192) return SI_ERR_INVALID_ARG;
  if (L.n_experts < 1 || L.n_experts > kBatchedMaxExperts || L.top_k < 1 || L.top_k > 8 ||
      L.top_k > L.n_experts)
    return SI_ERR_INVALID_ARG;
  if (L.inter < 256 || L.inter % 256 || L.inter > 4096) return SI_ERR_INVALID_ARG;
  if (!L.w_gate || !L.w_up || !L.w_down || !aligned16(L.w_gate) || !aligned16(L.w_up) ||
      !aligned16(L.w_down))
    return SI_ERR_INVALID_ARG;
  if (L.expert_type != SI_Q4_K || L.shared_inter != 0) return SI_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * L.top_k > 1024) return SI_ERR_UNSUPPORTED;   // grouping buffer
  return SI_OK;
}

static size_t gateup_grouped_smem(const si_moe_layer &L) {
  return 64 + kTokChunk * 32 * 4 + static_cast<size_t>(kTokChunk) * tile_record_bytes(L.hidden) +
         64u * (L.hidden / 256 * kQ4KBytes);
}
static size_t down_grouped_smem(const si_moe_layer &L) {
  return 64 + kDownRows * 32 * 4 + static_cast<size_t>(kTokChunk) * tile_record_bytes(L.inter) +
         static_cast<size_t>(kDownRows) * (L.inter / 256 * kQ4KBytes);
}

cudaError_t preload_batched() {
  cudaFuncAttributes a;
  const void *ks[] = {reinterpret_cast<const void *>(batched_prep_kernel),
                      reinterpret_cast<const void *>(gateup_grouped_kernel),
                      reinterpret_cast<const void *>(down_grouped_kernel),
                      reinterpret_cast<const void *>(combine_kernel)};
  for (const void *k : ks) {
    const cudaError_t e = cudaFuncGetAttributes(&a, k);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace si

using namespace si;

extern "C" size_t si_moe_ffn_batched_workspace_bytes(const si_moe_layer *L, int n_tokens) {
  if (!L || batched_check(*L, n_tokens) != SI_OK) return 0;
  return batched_geom(*L, n_tokens).bytes;
}

extern "C" si_status si_moe_ffn_batched(const si_moe_layer *L, int n_tokens, int mode,
                                        const void *x, const int32_t *topk_ids,
                                        const float *topk_w, void *routed_out, void *workspace,
                                        size_t workspace_bytes, void *stream) {
  if (!L || !x || !topk_ids || !topk_w || !routed_out) return SI_ERR_INVALID_ARG;
  if (mode != 0 && mode != 1 && mode != 2) return SI_ERR_INVALID_ARG;
  if (mode == 2) return SI_ERR_UNSUPPORTED;   // tensor-core mode: not built yet
  const si_status st = batched_check(*L, n_tokens);
  if (st != SI_OK) return st;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(topk_ids) & 3u) ||
      (reinterpret_cast<uintptr_t>(topk_w) & 3u) || (reinterpret_cast<uintptr_t>(routed_out) & 1u))
    return SI_ERR_INVALID_ARG;
  const BatchedGeom g = batched_geom(*L, n_tokens);
  if (!workspace || !aligned256(workspace) || workspace_bytes < g.bytes) return SI_ERR_WORKSPACE;
  uint8_t *base = static_cast<uint8_t *>(workspace);
  BatchedParams p{};
  p.x = static_cast<const __nv_bfloat16 *>(x);
  p.ids = topk_ids;
  p.wts = topk_w;
  p.T = n_tokens; p.H = L->hidden; p.E = L->n_experts; p.k = L->top_k; p.I = L->inter;
  p.wg = static_cast<const uint8_t *>(L->w_gate);
  p.wu = static_cast<const uint8_t *>(L->w_up);
  p.wd = static_cast<const uint8_t *>(L->w_down);
  p.rb_gu = L->hidden / 256 * kQ4KBytes;
  p.rb_d = L->inter / 256 * kQ4KBytes;
  p.count = reinterpret_cast<int *>(base + g.off_count);
  p.offset = reinterpret_cast<int *>(base + g.off_offset);
  p.active = reinterpret_cast<int *>(base + g.off_active);
  p.n_active = reinterpret_cast<int *>(base + g.off_nactive);
  p.pair_token = reinterpret_cast<int *>(base + g.off_pair_token);
  p.pair_of = reinterpret_cast<int *>(base + g.off_pair_of);
  p.xrec = base + g.off_xrec;
  p.hrec = base + g.off_hrec;
  p.y = reinterpret_cast<float *>(base + g.off_y);
  p.routed = static_cast<__nv_bfloat16 *>(routed_out);
  p.status = reinterpret_cast<uint32_t *>(base);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int units = L->inter / 32, tiles = L->hidden / kDownRows;
  const int max_active = n_tokens * L->top_k < L->n_experts ? n_tokens * L->top_k : L->n_experts;
  const size_t gsm = gateup_grouped_smem(*L), dsm = down_grouped_smem(*L);
  if (gsm > 227 * 1024 || dsm > 227 * 1024) return SI_ERR_UNSUPPORTED;
  cudaError_t e = allow_smem(gateup_grouped_kernel, gsm);
  if (e == cudaSuccess) e = allow_smem(down_grouped_kernel, dsm);
  if (e == cudaSuccess)
    e = launch_pdl(batched_prep_kernel, dim3(1 + n_tokens), dim3(kPrepThreads), 0, s, p);
  if (e == cudaSuccess)
    e = launch_pdl(gateup_grouped_kernel, dim3(max_active * units), dim3(kGuBThreads), gsm, s, p);
  if (e == cudaSuccess)
    e = launch_pdl(down_grouped_kernel, dim3(max_active * tiles), dim3(kDownBThreads), dsm, s, p);
  if (e == cudaSuccess)
    e = launch_pdl(combine_kernel, dim3((L->hidden + 255) / 256, n_tokens), dim3(256), 0, s, p);
  return cuda_status(e);
}
