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
// GB300 layout. Each thread block owns R whole expert rows; the hidden
// dimension of a row is split over W = 8/R warps of the block (the split-K
// reduction stays in shared memory, in a fixed order: deterministic, no
// float atomics). Each warp's slice of W_r goes into registers with 16-byte
// loads before the kernel waits on its predecessor (router weights do not
// depend on it), so the weight read overlaps the previous kernel's tail.
// Logits are written with an epoch tag; one acquire-release atomic per block
// counts completions; the last block checks every tag (a counter that was not
// zero at the start shows up as stale tags) and selects.
//
// Selection: (value, index) pairs are packed into 64-bit keys whose unsigned
// order is the selection order (value descending, -0 == +0, then lower index
// first), so every compare-exchange is a branch-free max/min. Each warp sorts
// 32 keys with a shuffle bitonic network; the first k of every warp are the
// only candidates, and each candidate's rank among them is its final rank.
#include <float.h>

#include <mutex>

#include "common.cuh"
#include "host.hpp"
#include "topk.cuh"

namespace si {

SI_TRACE_BUFFER

constexpr int kRouterThreads = 256;
constexpr int kRouterWarps = kRouterThreads / 32;
constexpr int kMaxTopK = 8;
constexpr int kMaxChunkTokens = 8;
static_assert(kMaxChunkTokens <= kRouterWarps, "the last block selects one token per warp");

struct RouterParams {
  const void *x;
  const void *w;
  int H, E, k, T;
  int R;             // expert rows per block
  int W;             // warps per row (R * W == 8)
  int tc;            // tokens per chunk
  int cpc;           // blocks per chunk = ceil(E / R)
  int32_t *ids;
  float *wts;
  float *logits;     // nullable
  uint2 *tagged;     // [T][E] {logit bits, epoch}
  uint32_t *counters;  // [n_chunks]
  uint32_t *epochs;    // [n_chunks]
  uint32_t *status;
};

template <typename T> struct Vec;   // elements per 16 bytes of weights
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

// VEC activation values as loaded (raw words: the loads go out before any
// of them is converted), then as fp32 exactly as load_x gives them.
template <typename XT, int VEC>
struct XRaw {
  static constexpr int kWords = static_cast<int>(sizeof(XT)) * VEC / 4;   // 2, 4 or 8
  uint32_t w[kWords];
  SI_DEV void load(const XT *p) {
    if constexpr (kWords == 2) {
      const uint2 u = *reinterpret_cast<const uint2 *>(p);
      w[0] = u.x; w[1] = u.y;
    } else {
#pragma unroll
      for (int i = 0; i < kWords / 4; ++i) {
        const uint4 u = reinterpret_cast<const uint4 *>(p)[i];
        w[4 * i] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
      }
    }
  }
  SI_DEV void to_float(float *v) const {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      if constexpr (sizeof(XT) == 2)
        v[i] = (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
      else
        v[i] = __uint_as_float(w[i]);
    }
  }
};

// After a block has written its logits of chunk `chunk` (tokens t0 ..
// t0 + ntok - 1): the chunk's completion count, and in the chunk's last
// block the check of every logit's epoch, the top-k selection and softmax.
SI_DEV void router_chunk_tail(const RouterParams &p, int chunk, int t0, int ntok, uint32_t epoch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Completion count: release this block's logits, acquire everyone's.
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atom_inc_acq_rel(&p.counters[chunk], static_cast<unsigned>(p.cpc - 1));
    s_last = (prev == static_cast<unsigned>(p.cpc - 1)) ? 1 : (prev > static_cast<unsigned>(p.cpc - 1) ? 2 : 0);
  }
  __syncthreads();
  SI_TRACE_MARK(0, 3);
  if (s_last == 0) return;
  int bad = (s_last == 2);

  // Last block of the chunk: every logit must carry this run's epoch.
  __shared__ float s_logit[kMaxChunkTokens][256];
  for (int i = threadIdx.x; i < ntok * p.E; i += kRouterThreads) {
    const uint2 v = __ldcg(&p.tagged[static_cast<size_t>(t0) * p.E + i]);
    if (v.y != epoch) bad = 1;
    s_logit[i / p.E][i % p.E] = __uint_as_float(v.x);
  }
  bad = __syncthreads_or(bad);
  SI_TRACE_MARK(0, 4);
  if (threadIdx.x == 0) p.epochs[chunk] = epoch;
  if (bad) {
    // The counter was not at zero when the run started (workspace not zeroed
    // or corrupted): report, and poison this chunk's outputs rather than
    // leave stale ids in place.
    if (threadIdx.x == 0) record_status(p.status, SI_ERR_HANDSHAKE);
    for (int i = threadIdx.x; i < ntok * p.k; i += kRouterThreads) {
      p.ids[static_cast<size_t>(t0) * p.k + i] = -1;
      p.wts[static_cast<size_t>(t0) * p.k + i] = 0.f;
    }
    return;
  }

  // The selection: top k of the E keys in rank order (keys are unique, so it
  // is one set whatever the method), then the softmax over them in rank
  // order, written by write_selection.
  auto write_selection = [&](int t, const uint64_t sel[kMaxTopK]) {
    const float v0 = key_value(sel[0]);
    float exv[kMaxTopK];
    float sum = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxTopK; ++q) {
      exv[q] = q < p.k ? expf(key_value(sel[q]) - v0) : 0.f;
      sum += exv[q];
    }
    const float inv = __frcp_rn(sum);
#pragma unroll
    for (int q = 0; q < kMaxTopK; ++q) {
      if (q < p.k) {
        p.ids[static_cast<size_t>(t) * p.k + q] = key_index(sel[q]);
        p.wts[static_cast<size_t>(t) * p.k + q] = exv[q] * inv;
      }
    }
  };
  if (ntok == 1) {
    // one token: every warp sorts 32 of its keys; the first k of each warp
    // are the only candidates, and a candidate's rank among them is its
    // rank overall
    __shared__ uint64_t s_cand[kRouterWarps * kMaxTopK];
    __shared__ uint64_t s_sel[kMaxTopK];
    const int ex = threadIdx.x;
    uint64_t key = ex < p.E ? make_key(s_logit[0][ex], ex) : 0ull;   // 0: below every real key
    key = warp_sort32(key, lane);
    if (lane < kMaxTopK) s_cand[warp * kMaxTopK + lane] = key;
    __syncthreads();
    if (threadIdx.x < kRouterWarps * kMaxTopK) {
      const uint64_t me = s_cand[threadIdx.x];
      int rank = 0;
#pragma unroll 8
      for (int j = 0; j < kRouterWarps * kMaxTopK; ++j) rank += s_cand[j] > me;
      if (rank < p.k && me != 0ull) s_sel[rank] = me;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t sel[kMaxTopK];
#pragma unroll
      for (int q = 0; q < kMaxTopK; ++q) sel[q] = q < p.k ? s_sel[q] : 0ull;
      write_selection(t0, sel);
    }
  } else if (warp < ntok) {
    // several tokens, one warp each (warp w takes token t0 + w, all at
    // once): lane l holds the keys of experts l, l + 32, ...; k rounds of a
    // warp-wide maximum take the top k in rank order (each round's maximum
    // sits in one lane, which drops it)
    const int t = t0 + warp;
    uint64_t kk[256 / 32];
#pragma unroll
    for (int i = 0; i < 256 / 32; ++i) {
      const int e = lane + 32 * i;
      kk[i] = e < p.E ? make_key(s_logit[warp][e], e) : 0ull;   // 0: below every real key
    }
    uint64_t sel[kMaxTopK];
#pragma unroll
    for (int q = 0; q < kMaxTopK; ++q) {
      sel[q] = 0ull;
      if (q < p.k) {
        uint64_t m = kk[0];
#pragma unroll
        for (int i = 1; i < 256 / 32; ++i) m = kmax(m, kk[i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = kmax(m, __shfl_xor_sync(0xffffffffu, m, off));
#pragma unroll
        for (int i = 0; i < 256 / 32; ++i)
          if (kk[i] == m) kk[i] = 0ull;
        sel[q] = m;
      }
    }
    if (lane == 0) write_selection(t, sel);
  }
  SI_TRACE_MARK(0, 6);
}

template <typename XT, typename WT, int NCH>
__global__ void __launch_bounds__(kRouterThreads) router_topk_kernel(RouterParams p) {
  constexpr int VEC = Vec<WT>::n;
  SI_TRACE_MARK(0, 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = warp / p.W, wpart = warp % p.W;
  const int e = blockIdx.x * p.R + r;
  const int chunk = blockIdx.y;
  const bool row_live = e < p.E;

  // This warp's part of its row: 16-byte vectors (i * W + wpart) * 32 + lane.
  uint4 wr[NCH];
  if (row_live) {
    const uint4 *wrow = reinterpret_cast<const uint4 *>(static_cast<const WT *>(p.w) +
                                                        static_cast<size_t>(e) * p.H);
#pragma unroll
    for (int c = 0; c < NCH; ++c) wr[c] = __ldg(wrow + (c * p.W + wpart) * 32 + lane);
  }
  grid_dep_wait();
  grid_dep_launch();
  SI_TRACE_MARK(0, 1);

  const int t0 = chunk * p.tc;
  const int t1 = min(p.T, t0 + p.tc);
  const int ntok = t1 - t0;
  const uint32_t epoch = __ldcg(&p.epochs[chunk]) + 1u;
  __shared__ float s_part[kMaxChunkTokens][kRouterWarps];
  // TG tokens at a time: their activation vectors are all requested before
  // the first product (4 vectors per lane in flight, which keeps the kernel
  // at the registers of one token at a time; rows of 4 or more vectors per
  // lane already hold that many loads)
  constexpr int TG = NCH == 1 ? 4 : (NCH == 2 ? 2 : 1);
  for (int tb = t0; tb < t1; tb += TG) {
    XRaw<XT, VEC> xr[TG][NCH];
#pragma unroll
    for (int u = 0; u < TG; ++u) {
      if (row_live && tb + u < t1) {
        const XT *xs = static_cast<const XT *>(p.x) + static_cast<size_t>(tb + u) * p.H;
#pragma unroll
        for (int c = 0; c < NCH; ++c) xr[u][c].load(xs + ((c * p.W + wpart) * 32 + lane) * VEC);
      }
    }
#pragma unroll
    for (int u = 0; u < TG; ++u) {
      if (tb + u < t1) {   // uniform over the block
        float acc = 0.f;
        if (row_live) {
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            float wv[VEC], xv[VEC];
            unpack_w<WT>(wr[c], wv);
            xr[u][c].to_float(xv);
#pragma unroll
            for (int i = 0; i < VEC; ++i) acc = fmaf(wv[i], xv[i], acc);
          }
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (lane == 0) s_part[tb + u - t0][warp] = acc;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < p.R * ntok) {
    const int rr = threadIdx.x % p.R, tt = threadIdx.x / p.R;
    const int ex = blockIdx.x * p.R + rr;
    if (ex < p.E) {
      float l = s_part[tt][rr * p.W];
      for (int w = 1; w < p.W; ++w) l += s_part[tt][rr * p.W + w];
      const size_t o = static_cast<size_t>(t0 + tt) * p.E + ex;
      p.tagged[o] = make_uint2(__float_as_uint(l), epoch);
      if (p.logits) p.logits[o] = l;
    }
  }
  SI_TRACE_MARK(0, 2);

  router_chunk_tail(p, chunk, t0, ntok, epoch);
}

// Sums over the warp of N per-lane values (N a multiple of 32), each lane
// keeping N / 32 of them: lane L ends with outputs L * N / 32 + j. At the
// step of distance d (16, 8, 4, 2, 1) a lane keeps the half of its current
// values that bit d of its index selects and adds its partner's copy of that
// half to its own: every output is the value an xor butterfly over the same
// distances gives it (own value plus partner's at each step), bit for bit,
// with N - 1 shuffles per lane instead of 5 N.
template <int N>
SI_DEV void warp_sums_spread(float v[N], int lane) {
#pragma unroll
  for (int d = 16, m = N / 2; d > 0; d >>= 1, m >>= 1) {
    const bool hi = (lane & d) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float keep = hi ? v[i + m] : v[i];
      const float send = hi ? v[i] : v[i + m];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
    }
  }
}

// Several tokens (a full chunk of up to kMaxChunkTokens) against RT router
// rows per block: warp w, lane l take vectors (c * 8 + w) * 32 + l of every
// row, as router_topk_kernel does with one row per block and 8 warps per
// row, so every logit is the same fma chain, the same butterfly and the same
// sum over the 8 warps: the same bits with RT + kMaxChunkTokens loads per
// lane and chunk instead of one row load per kMaxChunkTokens x loads.
template <typename XT, typename WT, int NCH, int RT>
__global__ void __launch_bounds__(kRouterThreads) router_rows_kernel(RouterParams p) {
  constexpr int VEC = Vec<WT>::n;
  constexpr int C = kMaxChunkTokens;
  constexpr int N = RT * C < 32 ? 32 : RT * C;
  static_assert(kRouterWarps == 8, "8 warps split every row");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * RT;
  const int chunk = blockIdx.y;
  uint4 wr[RT][NCH];
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    const bool live = e0 + r < p.E;
    const uint4 *wrow = reinterpret_cast<const uint4 *>(static_cast<const WT *>(p.w) +
                                                        static_cast<size_t>(live ? e0 + r : 0) * p.H);
#pragma unroll
    for (int c = 0; c < NCH; ++c)
      wr[r][c] = live ? __ldg(wrow + (c * 8 + warp) * 32 + lane) : make_uint4(0u, 0u, 0u, 0u);
  }
  grid_dep_wait();
  grid_dep_launch();
  const int t0 = chunk * p.tc;
  const int ntok = min(p.T, t0 + p.tc) - t0;
  const uint32_t epoch = __ldcg(&p.epochs[chunk]) + 1u;
  float acc[N];
#pragma unroll
  for (int o = 0; o < N; ++o) acc[o] = 0.f;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    XRaw<XT, VEC> xr[C];
#pragma unroll
    for (int u = 0; u < C; ++u)
      if (u < ntok)
        xr[u].load(static_cast<const XT *>(p.x) + static_cast<size_t>(t0 + u) * p.H +
                   ((c * 8 + warp) * 32 + lane) * VEC);
#pragma unroll
    for (int u = 0; u < C; ++u) {
      if (u < ntok) {
        float xv[VEC];
        xr[u].to_float(xv);
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          float wv[VEC];
          unpack_w<WT>(wr[r][c], wv);
#pragma unroll
          for (int i = 0; i < VEC; ++i) acc[r * C + u] = fmaf(wv[i], xv[i], acc[r * C + u]);
        }
      }
    }
  }
  warp_sums_spread<N>(acc, lane);
  __shared__ float s_part[N][kRouterWarps];
#pragma unroll
  for (int j = 0; j < N / 32; ++j) s_part[lane * (N / 32) + j][warp] = acc[j];
  __syncthreads();
  if (threadIdx.x < RT * C) {
    const int r = threadIdx.x / C, u = threadIdx.x % C;
    const int ex = e0 + r;
    if (u < ntok && ex < p.E) {
      float l = s_part[threadIdx.x][0];
#pragma unroll
      for (int w = 1; w < kRouterWarps; ++w) l += s_part[threadIdx.x][w];
      const size_t o = static_cast<size_t>(t0 + u) * p.E + ex;
      p.tagged[o] = make_uint2(__float_as_uint(l), epoch);
      if (p.logits) p.logits[o] = l;
    }
  }
  router_chunk_tail(p, chunk, t0, ntok, epoch);
}

// Rows per block R and warps per row W (R * W = 8): one row per block with
// its 16-byte vectors dealt to the 256 lanes of all 8 warps (vector
// c * 256 + 32 w + lane to lane `lane` of warp w), the order in which the
// persistent stack kernel forms the same dot products, so both give the same
// bits; fewer warps per row only when the row has fewer than 256 vectors.
static void router_shape(int n_experts, int hidden, int vec, int &R, int &W, int &nch) {
  (void)n_experts;
  const int nv = hidden / vec;
  W = 8;
  while (W > 1 && nv % (32 * W) != 0) W /= 2;
  R = 8 / W;
  nch = nv / (32 * W);
}

RouterGeom router_geom(int n_experts, int hidden, int n_tokens) {
  RouterGeom g{};
  int R, W, nch;
  router_shape(n_experts, hidden, 8, R, W, nch);
  g.row_tiles = (n_experts + R - 1) / R;
  g.splits = W;
  g.ctas_per_chunk = g.row_tiles;
  g.tok_per_chunk = n_tokens < kMaxChunkTokens ? n_tokens : kMaxChunkTokens;
  if (g.tok_per_chunk < 1) g.tok_per_chunk = 1;
  g.n_chunks = (n_tokens + g.tok_per_chunk - 1) / g.tok_per_chunk;
  size_t off = sizeof(WsHeader);
  g.off_counters = off;
  off = round_up(off + sizeof(uint32_t) * g.n_chunks, 256);
  g.off_flags = off;   // epochs
  off = round_up(off + sizeof(uint32_t) * g.n_chunks, 256);
  g.off_partials = off;  // tagged logits
  off = round_up(off + sizeof(uint2) * static_cast<size_t>(n_tokens) * n_experts, 256);
  g.bytes = off;
  return g;
}

// Rows per block of the several-chunk kernel: enough rows that each block
// reads fewer bytes than its tokens' activations, few enough that the grid
// still covers the GPU (0: one row per block, router_topk_kernel).
static int rows_per_block(int W, int nch, int tc, int n_chunks) {
  if (W != 8 || nch > 2 || tc != kMaxChunkTokens) return 0;
  return n_chunks >= 8 ? 8 : (n_chunks >= 4 ? 4 : (n_chunks >= 2 ? 2 : 0));
}

template <typename XT, typename WT>
static cudaError_t launch_router_t(RouterParams p, int n_chunks, cudaStream_t s) {
  constexpr int VEC = Vec<WT>::n;
  int nch;
  router_shape(p.E, p.H, VEC, p.R, p.W, nch);
  const int rt = rows_per_block(p.W, nch, p.tc, n_chunks);
  if (rt > 0) {
    p.cpc = (p.E + rt - 1) / rt;
    const dim3 grid(p.cpc, n_chunks), block(kRouterThreads);
    auto k = nch == 1 ? (rt == 8 ? router_rows_kernel<XT, WT, 1, 8>
                                 : rt == 4 ? router_rows_kernel<XT, WT, 1, 4> : router_rows_kernel<XT, WT, 1, 2>)
                      : (rt == 8 ? router_rows_kernel<XT, WT, 2, 8>
                                 : rt == 4 ? router_rows_kernel<XT, WT, 2, 4> : router_rows_kernel<XT, WT, 2, 2>);
    return launch_pdl(k, grid, block, 0, s, p);
  }
  p.cpc = (p.E + p.R - 1) / p.R;
  const dim3 grid(p.cpc, n_chunks), block(kRouterThreads);
  switch (nch) {
    case 1: return launch_pdl(router_topk_kernel<XT, WT, 1>, grid, block, 0, s, p);
    case 2: return launch_pdl(router_topk_kernel<XT, WT, 2>, grid, block, 0, s, p);
    case 4: return launch_pdl(router_topk_kernel<XT, WT, 4>, grid, block, 0, s, p);
    case 8: return launch_pdl(router_topk_kernel<XT, WT, 8>, grid, block, 0, s, p);
    case 16: return launch_pdl(router_topk_kernel<XT, WT, 16>, grid, block, 0, s, p);
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
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, router_topk_kernel<XT, WT, 16>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, router_rows_kernel<XT, WT, 1, 2>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, router_rows_kernel<XT, WT, 1, 4>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, router_rows_kernel<XT, WT, 1, 8>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, router_rows_kernel<XT, WT, 2, 2>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, router_rows_kernel<XT, WT, 2, 4>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, router_rows_kernel<XT, WT, 2, 8>);
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
  p.tc = g.tok_per_chunk;
  p.ids = ids; p.wts = wts; p.logits = logits;
  p.tagged = reinterpret_cast<uint2 *>(base + g.off_partials);
  p.counters = reinterpret_cast<uint32_t *>(base + g.off_counters);
  p.epochs = reinterpret_cast<uint32_t *>(base + g.off_flags);
  p.status = status;
  {
    int R, W, nch;
    router_shape(n_experts, hidden, w_type == SI_F32 ? 4 : 8, R, W, nch);
    if (nch < 1 || nch > 16 || (nch & (nch - 1))) return SI_ERR_UNSUPPORTED;
  }
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

#ifdef SI_TRACE
extern "C" int si_trace_dump_router(void *dst) {
  return cudaMemcpyFromSymbol(dst, si::g_si_trace, sizeof(si::g_si_trace)) == cudaSuccess ? 0 : 4;
}
extern "C" int si_trace_reset_router(void) {
  static uint64_t zeros[si::kTraceKernels * si::kTraceBlocks * si::kTracePhases];
  return cudaMemcpyToSymbol(si::g_si_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : 4;
}
#endif

// ---------------------------------------------------------------------------
// Router with library-owned scratch, for callers that cannot allocate device
// memory. The scratch (status word, completion counters, epochs and the
// tagged logits) lives in this file-scope device array instead of a caller
// workspace; every GPU that loads the library holds it until the process
// exits. It is sized for every accepted shape: n_tokens * n_experts <=
// kNoAllocMaxEntries, with n_experts >= 8, so at most 2048 tokens and 256
// token chunks (status header, counters and epochs of 256 chunks, tagged
// logits of 16384 entries: 133,376 bytes).
// ---------------------------------------------------------------------------
namespace si {
constexpr int kNoAllocMaxEntries = 64 * 256;
constexpr int kNoAllocMaxChunks = kNoAllocMaxEntries / 8 / kMaxChunkTokens;
constexpr size_t kNoAllocScratchBytes = sizeof(WsHeader) + 2 * ((4 * kNoAllocMaxChunks + 255) / 256 * 256) +
                                        sizeof(uint2) * kNoAllocMaxEntries;
static_assert(kNoAllocScratchBytes == 133376, "no-alloc scratch size");
static __device__ __align__(256) uint8_t g_router_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array for the current device. The first call
// on a device looks it up (cudaGetSymbolAddress, with that device current)
// and caches it; later calls only read the cache.
static si_status noalloc_scratch(void **out) {
  static std::mutex mu;
  static void *addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SI_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_router_noalloc_scratch) != cudaSuccess || !p) return SI_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return SI_OK;
}
}  // namespace si

extern "C" si_status si_moe_router_topk_noalloc(const void *x, si_dtype x_type, const void *w_router,
                                                si_dtype w_type, int hidden, int n_experts,
                                                int top_k, int n_tokens, int32_t *topk_ids,
                                                float *topk_w, float *logits_out, void *stream) {
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
  // Larger problems than the fixed scratch holds are refused.
  if (static_cast<int64_t>(n_tokens) * n_experts > kNoAllocMaxEntries) return SI_ERR_UNSUPPORTED;
  const RouterGeom g = router_geom(n_experts, hidden, n_tokens);
  if (g.bytes > kNoAllocScratchBytes) return SI_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  si_status st = noalloc_scratch(&scratch);
  if (st != SI_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the completion counters
  // must start at zero (the epochs may keep counting, and the status word
  // keeps the first device-side error until si_moe_router_noalloc_status
  // reads it).
  if (cudaMemsetAsync(static_cast<uint8_t *>(scratch) + g.off_counters, 0,
                      g.off_flags - g.off_counters, s) != cudaSuccess)
    return SI_ERR_CUDA;
  return router_launch(x, x_type, w_router, w_type, hidden, n_experts, top_k, n_tokens, topk_ids,
                       topk_w, logits_out, scratch, static_cast<uint32_t *>(scratch), s);
}

extern "C" si_status si_moe_router_noalloc_status(void *stream, int *status_out) {
  if (!status_out) return SI_ERR_INVALID_ARG;
  void *scratch = nullptr;
  si_status st = noalloc_scratch(&scratch);
  if (st != SI_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && v != 0) e = cudaMemset(scratch, 0, sizeof(v));
  if (e != cudaSuccess) return SI_ERR_CUDA;
  *status_out = static_cast<int>(v);
  return SI_OK;
}
