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
//          by token) and lists the active experts most tokens first, so the
//          grouped kernels' longest blocks start first and the grid's tail
//          holds the shortest; the other blocks quantise every token's x
//          once into a Q8_1 tile record.
//  gate/up one block per (active expert, 32-row unit of h), two per SM: 32
//          gate + 32 up rows by TMA bulk copy, the expert's token tiles by
//          bulk copy, each weight super-block unpacked once and dotted with
//          every token of the chunk, then Q8_1 of each token's 32 values of h.
//  down    one block per (active expert, 32 output rows): the rows once, then
//          y = D_e h for each of the expert's pairs (fp32 per pair), each
//          weight piece unpacked once per chunk of pairs.
//  combine routed[t][j] = sum_r w[t][r] * y[pair(t, r)][j] in rank order;
//          in the batched layer one block per token also runs the residual
//          norm on it (combine_norm_kernel).
#include "common.cuh"
#include "host.hpp"
#include "norm.cuh"
#include "tc.cuh"

namespace si {

constexpr int kBatchedMaxExperts = 256;
constexpr int kPrepThreads = 512;
static_assert(kBatchedMaxExperts <= kPrepThreads - 32, "prep: the last warp is free of expert rows");
constexpr int kGuBThreads = 256;     // two gate/up blocks per SM: one's copies overlap the other's dots
constexpr int kGuTok = 4;            // token tiles resident per gate/up block at once
constexpr int kDownBThreads = 256;
constexpr int kDnTok = 4;            // token tiles resident per down block at once
// down blocks: 32 R output rows (R = 2 unless the block's shared memory
// would not fit), 32 threads per half super-block of a row (at most 8 warps)

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
  int *active;               // [E] active expert ids by token count, descending (ties: ascending id)
  int *n_active;             // [1]
  int *pair_token;           // [T*k] token of each grouped pair
  int *pair_of;              // [T*k] grouped position of pair (t, r)
  uint8_t *xrec;             // [T][tile_record_bytes(H)]
  uint8_t *hrec;             // [T*k][tile_record_bytes(I)]
  float *y;                  // [T*k][H]
  __nv_bfloat16 *routed;     // [T][H]
  uint32_t *status;
  // tensor-core mode
  int tensor;                // 1: x -> fp16 rows instead of Q8_1 tiles
  __half *xh;                // [T][H] fp16
  __half *hh;                // [T*k][I] fp16
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
    if (t < p.T && p.tensor) {
      for (int i = 8 * threadIdx.x; i < p.H; i += 8 * blockDim.x) {
        float v[8];
        Load8<__nv_bfloat16>::run(p.x + static_cast<size_t>(t) * p.H + i, v);
        *reinterpret_cast<uint4 *>(p.xh + static_cast<size_t>(t) * p.H + i) =
            make_uint4(pack_half2(v[0], v[1]), pack_half2(v[2], v[3]), pack_half2(v[4], v[5]),
                       pack_half2(v[6], v[7]));
      }
    } else if (t < p.T) {
      ActTile tile = tile_at(p.xrec + static_cast<size_t>(t) * tile_record_bytes(p.H), p.H);
      quantize_to_tile<__nv_bfloat16>(p.x + static_cast<size_t>(t) * p.H, p.H, tile);
    }
    return;
  }
  // Group the pairs q = (token q / k, rank q % k) by expert, stably: the
  // position of pair q inside its expert's range is the number of pairs j < q
  // with the same expert. Pairs are taken in chunks of 32 (one warp): within
  // a chunk the lanes with the same expert find each other with a match, and
  // a per-(chunk, expert) count, summed over the earlier chunks, gives the rest.
  __shared__ int s_cnt[kBatchedMaxExperts];
  __shared__ int s_off[kBatchedMaxExperts + 1];
  __shared__ int s_e[1024];
  __shared__ unsigned char s_rank[1024];
  __shared__ __align__(16) unsigned short s_wc[32][kBatchedMaxExperts];   // [chunk][expert]
  // the active list, most tokens first (longest processing time first): an
  // active expert's bucket is b = min(count, 31); its place is the number of
  // experts in higher buckets plus those of lower id in its own (the bit
  // masks of the buckets' experts)
  __shared__ int s_bn[32];
  __shared__ uint32_t s_bmask[32][kBatchedMaxExperts / 32];
  const int P = p.T * p.k;   // <= 1024 (host check)
  const int nchunk = (P + 31) / 32;
  const int lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) s_cnt[e] = 0;
  for (int i = threadIdx.x; i < nchunk * kBatchedMaxExperts / 2; i += blockDim.x)   // the chunks' rows
    reinterpret_cast<uint32_t *>(&s_wc[0][0])[i] = 0u;
  if (threadIdx.x < 32) s_bn[threadIdx.x] = 0;
  if (threadIdx.x < 32 * kBatchedMaxExperts / 32) (&s_bmask[0][0])[threadIdx.x] = 0u;
  __syncthreads();
  for (int q = threadIdx.x; q < 32 * nchunk; q += blockDim.x) {   // whole warps
    int e = -1;
    if (q < P) {
      e = p.ids[q];
      if (e < 0 || e >= p.E) {
        record_status(p.status, SI_ERR_INVALID_ARG);
        e = 0;
      }
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    if (q < P) {
      s_e[q] = e;
      s_rank[q] = static_cast<unsigned char>(__popc(same & ((1u << lane) - 1u)));
      if ((__ffs(same) - 1) == lane) {   // the chunk's first pair of expert e
        s_wc[q >> 5][e] = static_cast<unsigned short>(__popc(same));
        atomicAdd(&s_cnt[e], __popc(same));
      }
    }
  }
  __syncthreads();
  if (static_cast<int>(threadIdx.x) < p.E) {   // counts of the earlier chunks
    const int e = threadIdx.x;
    int acc = 0;
    for (int c = 0; c < nchunk; ++c) {
      const int v = s_wc[c][e];
      s_wc[c][e] = static_cast<unsigned short>(acc);
      acc += v;
    }
    if (acc > 0) {
      const int b = acc < 31 ? acc : 31;
      atomicAdd(&s_bn[b], 1);
      atomicOr(&s_bmask[b][e >> 5], 1u << (e & 31));
    }
  } else if (threadIdx.x >= kPrepThreads - 32) {
    // the last warp: expert offsets (ascending expert), lane L owning
    // experts 8L .. 8L + 7
    int cnt[8], sum = 0, nz = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = 8 * lane + i;
      cnt[i] = e < p.E ? s_cnt[e] : 0;
      sum += cnt[i];
      nz += cnt[i] > 0;
    }
    int incl = sum, incl_nz = nz;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d), onz = __shfl_up_sync(0xffffffffu, incl_nz, d);
      if (lane >= d) {
        incl += o;
        incl_nz += onz;
      }
    }
    int acc = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = 8 * lane + i;
      if (e < p.E) {
        s_off[e] = acc;
        acc += cnt[i];
      }
    }
    if (lane == 31) {
      s_off[p.E] = incl;
      *p.n_active = incl_nz;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= p.E; e += blockDim.x) {
    p.offset[e] = s_off[e];
    if (e < p.E) {
      const int c = s_cnt[e];
      p.count[e] = c;
      if (c > 0) {
        const int b = c < 31 ? c : 31;
        int pos = 0;
#pragma unroll
        for (int v = 1; v < 32; ++v) pos += v > b ? s_bn[v] : 0;
#pragma unroll
        for (int w = 0; w < kBatchedMaxExperts / 32; ++w)
          if (w <= (e >> 5))
            pos += __popc(s_bmask[b][w] & (w < (e >> 5) ? 0xFFFFFFFFu : (1u << (e & 31)) - 1u));
        p.active[pos] = e;
      }
    }
  }
  for (int q = threadIdx.x; q < P; q += blockDim.x) {
    const int e = s_e[q];
    const int pos = s_off[e] + s_wc[q >> 5][e] + s_rank[q];
    p.pair_of[q] = pos;
    p.pair_token[pos] = q / p.k;
  }
}

// ---------------------------------------------------------------------------
// The code words of pair p (sub-blocks 2p, 2p + 1) of a Q4_K super-block,
// split once into their low nibbles (sub-block 2p) and their high nibbles
// left in place (2p + 1, each byte 16 times its code: one mask, no shift),
// and the exact int32 sums of those codes with one token's 64 activation
// codes of the pair (a4: sub-block 2p's 32 codes, then 2p + 1's): the
// integer sums of q4k_pair_isums (the high sum taken as unsigned x signed
// bytes and divided by 16, which is exact).
SI_DEV void q4k_pair_nibbles(const uint4 *wv, int p, uint32_t lo[8], uint32_t hi[8]) {
  uint32_t qw[8];
  q4k_pair_words(wv, p, qw);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    lo[i] = qw[i] & 0x0F0F0F0Fu;
    hi[i] = qw[i] & 0xF0F0F0F0u;   // the high nibbles, times 16
  }
}
// dp4a of unsigned bytes a with signed bytes b
SI_DEV int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
SI_DEV void q4k_pair_nibble_isums(const uint32_t lo[8], const uint32_t hi[8], const uint4 a4[4], int &slo,
                                  int &shi) {
  const uint32_t al[8] = {a4[0].x, a4[0].y, a4[0].z, a4[0].w, a4[1].x, a4[1].y, a4[1].z, a4[1].w};
  const uint32_t ah[8] = {a4[2].x, a4[2].y, a4[2].z, a4[2].w, a4[3].x, a4[3].y, a4[3].z, a4[3].w};
  slo = 0;
  int shi16 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    slo = __dp4a(static_cast<int>(lo[i]), static_cast<int>(al[i]), slo);
    shi16 = dp4a_us(hi[i], ah[i], shi16);
  }
  shi = shi16 >> 4;   // exact: 16 times the sum of the high nibbles' products
}

// Two rows' Q4_K super-blocks w0, w1 (the same super-block sb, shared
// memory) against super-block sb of the first nt token tiles at xt: per
// (row, token) exactly q4k_sb_dot's value (its integer sums, its fmas in
// sub-block order, one rounding per product and one for the difference).
// Each pair of sub-blocks is split into nibbles once for all the tokens and
// each token's activation codes are read once for both rows.
SI_DEV void q4k_sb_dot_2rows_tokens(const uint8_t *w0, const uint8_t *w1, const uint8_t *xt, int xrb, int H,
                                    int sb, int nt, float out[2][kGuTok]) {
  const uint4 *wv[2] = {reinterpret_cast<const uint4 *>(w0), reinterpret_cast<const uint4 *>(w1)};
  uint32_t scp[2][2], mnp[2][2];   // 6-bit scales / mins of sub-blocks 0..3 and 4..7, one per byte
  float d[2], dmin[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint4 hd = wv[r][0];
    scp[r][0] = hd.y & 0x3F3F3F3Fu;
    mnp[r][0] = hd.z & 0x3F3F3F3Fu;
    scp[r][1] = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
    mnp[r][1] = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
    d[r] = half_bits_to_float(static_cast<uint16_t>(hd.x & 0xFFFF));
    dmin[r] = half_bits_to_float(static_cast<uint16_t>(hd.x >> 16));
  }
  float ad[2][kGuTok], am[2][kGuTok];
#pragma unroll
  for (int t = 0; t < kGuTok; ++t) ad[0][t] = ad[1][t] = am[0][t] = am[1][t] = 0.f;
  const int nsb = H / kQKK;
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    uint32_t lo[2][8], hi[2][8];
    q4k_pair_nibbles(wv[0], pp, lo[0], hi[0]);
    q4k_pair_nibbles(wv[1], pp, lo[1], hi[1]);
#pragma unroll
    for (int t = 0; t < kGuTok; ++t) {
      if (t < nt) {
        const uint8_t *rec = xt + t * xrb;
        const uint4 *a = reinterpret_cast<const uint4 *>(rec + sb * kActSbStride) + 4 * pp;
        const uint4 a4[4] = {a[0], a[1], a[2], a[3]};
        const float *da = reinterpret_cast<const float *>(rec + nsb * kActSbStride) + 8 * sb + 2 * pp;
        const float *sa = da + H / 32;
        const float da0 = da[0], da1 = da[1], sa0 = sa[0], sa1 = sa[1];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          int slo, shi;
          q4k_pair_nibble_isums(lo[r], hi[r], a4, slo, shi);
          const int j = 2 * pp;   // sub-blocks j, j + 1 (the same scale word)
          const uint32_t sw = scp[r][j >> 2], mw = mnp[r][j >> 2];
          const int sc0 = static_cast<int>((sw >> (8 * (j & 3))) & 0xFFu);
          const int sc1 = static_cast<int>((sw >> (8 * ((j + 1) & 3))) & 0xFFu);
          const int mn0 = static_cast<int>((mw >> (8 * (j & 3))) & 0xFFu);
          const int mn1 = static_cast<int>((mw >> (8 * ((j + 1) & 3))) & 0xFFu);
          ad[r][t] = fmaf(static_cast<float>(sc0 * slo), da0, ad[r][t]);
          am[r][t] = fmaf(static_cast<float>(mn0), sa0, am[r][t]);
          ad[r][t] = fmaf(static_cast<float>(sc1 * shi), da1, ad[r][t]);
          am[r][t] = fmaf(static_cast<float>(mn1), sa1, am[r][t]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int t = 0; t < kGuTok; ++t)
      if (t < nt) out[r][t] = __fsub_rn(__fmul_rn(d[r], ad[r][t]), __fmul_rn(dmin[r], am[r][t]));
}

// Gate/up, integer mode: one block per (active expert, 32-row unit of h).
// Warp w issues one bulk copy of 8 gate (w < 4) or up rows and, per chunk of
// up to kGuTok of the expert's tokens, the copy of token tile w. Thread
// (row pair prq, gate/up m, lane8) owns super-blocks lane8, lane8 + 8, ... of
// rows prq and prq + 16 and dots both against all the chunk's tokens (each
// pair of sub-blocks split into nibbles once, each token's codes read once
// for both rows); the row dots go to shared memory and warp w forms token
// w's h = silu(gate) * up and its Q8_1 block.
__global__ void __launch_bounds__(kGuBThreads, 2) gateup_grouped_kernel(BatchedParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int units = p.I / 32;
  const int nsb = p.H / kQKK;
  const int xrb = tile_record_bytes(p.H);
  const int hrb = tile_record_bytes(p.I);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);        // 4 weight groups + 1 tokens
  float *s_raw = reinterpret_cast<float *>(smem + 64);        // [kGuTok][gate, up][32] row dots
  uint8_t *xt = smem + 64 + kGuTok * 64 * 4;                  // [kGuTok][xrb]
  uint8_t *wbuf = xt + kGuTok * xrb;                          // gate [32][rb], up [32][rb]
  grid_dep_wait();
  grid_dep_launch();
  const int na = __ldcg(p.n_active);
  if (static_cast<int>(blockIdx.x) >= na * units) return;
  const int e = __ldcg(p.active + blockIdx.x / units);
  const int unit = blockIdx.x % units;
  const int n_e = __ldcg(p.count + e), p0 = __ldcg(p.offset + e);
  const int rb = p.rb_gu;
  uint8_t *gate_buf = wbuf, *up_buf = wbuf + 32 * rb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bytes = 8u * rb;
  if (threadIdx.x == 0) {
    for (int g = 0; g < 5; ++g) mbar_init(&bars[g], 1);
    fence_mbar_init();
    for (int g = 0; g < 4; ++g) mbar_arrive_expect_tx(&bars[g], 2 * bytes);
  }
  __syncthreads();
  if (lane == 0) {
    const uint64_t pol = policy_evict_first();
    const size_t row0 = static_cast<size_t>(e) * p.I + static_cast<size_t>(unit) * 32 + 8 * (warp & 3);
    bulk_g2s_evict_first((warp < 4 ? gate_buf : up_buf) + 8 * (warp & 3) * rb,
                         (warp < 4 ? p.wg : p.wu) + row0 * rb, bytes, &bars[warp & 3], pol);
  }
  const int prq = threadIdx.x >> 4, m = (threadIdx.x >> 3) & 1, lane8 = threadIdx.x & 7;
  uint32_t phase = 0;
  for (int c0 = 0; c0 < n_e; c0 += kGuTok) {
    const int nc = min(kGuTok, n_e - c0);
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&bars[4], nc * xrb);
    __syncthreads();   // armed before any of the chunk's copies is issued
    if (lane == 0 && warp < nc) {
      const int t = __ldcg(p.pair_token + p0 + c0 + warp);
      bulk_g2s(xt + warp * xrb, p.xrec + static_cast<size_t>(t) * xrb, xrb, &bars[4]);
    }
    mbar_wait_bounded(&bars[4], phase, p.status);
    phase ^= 1u;
    // rows prq and prq + 16 of matrix m, together
    if (c0 == 0) {
      mbar_wait_bounded(&bars[prq >> 3], 0, p.status);
      mbar_wait_bounded(&bars[(prq + 16) >> 3], 0, p.status);
    }
    const uint8_t *row0 = (m ? up_buf : gate_buf) + prq * rb;
    float acc[2][kGuTok];
#pragma unroll
    for (int i = 0; i < kGuTok; ++i) acc[0][i] = acc[1][i] = 0.f;
#pragma unroll 1
    for (int sb = lane8; sb < nsb; sb += 8) {
      float dv[2][kGuTok];
      q4k_sb_dot_2rows_tokens(row0 + sb * kQ4KBytes, row0 + 16 * rb + sb * kQ4KBytes, xt, xrb, p.H, sb, nc, dv);
#pragma unroll
      for (int i = 0; i < kGuTok; ++i)
        if (i < nc) {
          acc[0][i] += dv[0][i];
          acc[1][i] += dv[1][i];
        }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int pr = prq + 16 * rr;
#pragma unroll
      for (int i = 0; i < kGuTok; ++i) {
        if (i < nc) {   // nc is uniform over the block
          float v = acc[rr][i];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          if (lane8 == 0) s_raw[(2 * i + m) * 32 + pr] = v;
        }
      }
    }
    __syncthreads();
    // warp w: token w of the chunk; lane j: h_j = silu(gate_j) * up_j, then
    // the Q8_1 block of the token's 32 values of h
    for (int i = warp; i < nc; i += kGuBThreads / 32) {
      const float g = s_raw[(2 * i) * 32 + lane], u = s_raw[(2 * i + 1) * 32 + lane];
      uint16_t d16, s16;
      const int q = q8_1_encode_warp(__fdiv_rn(g, 1.f + expf(-g)) * u, d16, s16);
      ActTile h = tile_at(p.hrec + static_cast<size_t>(p0 + c0 + i) * hrb, p.I);
      const int j0 = unit * 32;   // element offset of this unit inside the pair's h
      h.qs[(j0 / kQKK) * kActSbStride + j0 % kQKK + lane] = static_cast<uint8_t>(q);
      if (lane == 0) {
        h.d[j0 / 32] = half_bits_to_float(d16);
        h.s[j0 / 32] = half_bits_to_float(s16);
      }
    }
    __syncthreads();   // the row dots and the token tiles are reused by the next chunk
  }
}

// ---------------------------------------------------------------------------
// Half h (sub-blocks 4h .. 4h + 3, 128 weights) of super-block sb of R rows
// (w[r], shared memory) against super-block sb of the first nt Q8_1 tiles at
// ht (width I, hrb bytes apart): per (row, token) exactly the single-token
// half dot (the integer sums of q4k_pair_isums, the fmas in sub-block order,
// one rounding per product and one for the difference). Each pair of
// sub-blocks is split into nibbles once and each token's codes are read once
// for all R rows.
template <int R>
SI_DEV void q4k_half_dot_rows_tokens(const uint8_t *const w[R], const uint8_t *ht, int hrb, int I, int sb, int h,
                                     int nt, float out[R][kDnTok]) {
  uint32_t scw[R], mnw[R];   // 6-bit scales / mins of sub-blocks 4h .. 4h + 3, one per byte
  float d[R], dmin[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint4 hd = reinterpret_cast<const uint4 *>(w[r])[0];
    scw[r] = h ? ((hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u)) : (hd.y & 0x3F3F3F3Fu);
    mnw[r] = h ? (((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u)) : (hd.z & 0x3F3F3F3Fu);
    d[r] = half_bits_to_float(static_cast<uint16_t>(hd.x & 0xFFFF));
    dmin[r] = half_bits_to_float(static_cast<uint16_t>(hd.x >> 16));
  }
  float ad[R][kDnTok], am[R][kDnTok];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int t = 0; t < kDnTok; ++t) ad[r][t] = am[r][t] = 0.f;
  const int nsb = I / kQKK;
#pragma unroll
  for (int pp = 0; pp < 2; ++pp) {
    const int pr = 2 * h + pp;   // pair of the super-block
    uint32_t lo[R][8], hi[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) q4k_pair_nibbles(reinterpret_cast<const uint4 *>(w[r]), pr, lo[r], hi[r]);
#pragma unroll
    for (int t = 0; t < kDnTok; ++t) {
      if (t < nt) {
        const uint8_t *rec = ht + t * hrb;
        const uint4 *a = reinterpret_cast<const uint4 *>(rec + sb * kActSbStride) + 4 * pr;
        const uint4 a4[4] = {a[0], a[1], a[2], a[3]};
        const float *da = reinterpret_cast<const float *>(rec + nsb * kActSbStride) + 8 * sb + 2 * pr;
        const float *sa = da + I / 32;
        const float da0 = da[0], da1 = da[1], sa0 = sa[0], sa1 = sa[1];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          int slo, shi;
          q4k_pair_nibble_isums(lo[r], hi[r], a4, slo, shi);
          const int sc0 = static_cast<int>((scw[r] >> (16 * pp)) & 0xFFu);
          const int sc1 = static_cast<int>((scw[r] >> (16 * pp + 8)) & 0xFFu);
          const int mn0 = static_cast<int>((mnw[r] >> (16 * pp)) & 0xFFu);
          const int mn1 = static_cast<int>((mnw[r] >> (16 * pp + 8)) & 0xFFu);
          ad[r][t] = fmaf(static_cast<float>(sc0 * slo), da0, ad[r][t]);
          am[r][t] = fmaf(static_cast<float>(mn0), sa0, am[r][t]);
          ad[r][t] = fmaf(static_cast<float>(sc1 * shi), da1, ad[r][t]);
          am[r][t] = fmaf(static_cast<float>(mn1), sa1, am[r][t]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int t = 0; t < kDnTok; ++t)
      if (t < nt) out[r][t] = __fsub_rn(__fmul_rn(d[r], ad[r][t]), __fmul_rn(dmin[r], am[r][t]));
}

// Down, integer mode: one block per (active expert, 32 R output rows). The
// rows arrive once by bulk copy; per chunk of up to kDnTok of the expert's
// pairs, warp w takes the half super-blocks q = w, w + warps, ... of every
// row (so its lanes read the same activation codes) and lane l the rows l,
// l + 32, ...; then each (pair, row) sums its pieces in order.
template <int R>
__global__ void __launch_bounds__(kDownBThreads, 3) down_grouped_kernel(BatchedParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int kRows = 32 * R;
  const int tiles = p.H / kRows;
  const int nsb = p.I / kQKK;
  const int P = 2 * nsb;                 // half super-block pieces per row
  const int hrb = tile_record_bytes(p.I);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);           // weights, tokens
  float *part = reinterpret_cast<float *>(smem + 64);            // [kDnTok][P][kRows]
  uint8_t *ht = smem + 64 + kDnTok * kRows * P * 4;              // [kDnTok][hrb]
  uint8_t *wbuf = ht + kDnTok * hrb;                             // [kRows][rb_d]
  // The grouping (counts, offsets, active list) comes from the grouping
  // kernel two launches back, which has completed: this grid is launched
  // only once every gate/up block has passed its own wait on it. So this
  // block's weight rows are requested before the wait on the gate/up kernel,
  // whose h tiles it reads after it.
  const int na = __ldcg(p.n_active);
  if (static_cast<int>(blockIdx.x) >= na * tiles) return;
  const int e = __ldcg(p.active + blockIdx.x / tiles);
  const int j0 = (blockIdx.x % tiles) * kRows;
  const int n_e = __ldcg(p.count + e), p0 = __ldcg(p.offset + e);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t bytes = static_cast<uint32_t>(kRows) * p.rb_d;
    mbar_arrive_expect_tx(&bars[0], bytes);
    bulk_g2s_evict_first(wbuf, p.wd + (static_cast<size_t>(e) * p.H + j0) * p.rb_d, bytes, &bars[0],
                         policy_evict_first());
  }
  grid_dep_wait();
  grid_dep_launch();
  uint32_t phase = 0;
  for (int c0 = 0; c0 < n_e; c0 += kDnTok) {
    const int nc = min(kDnTok, n_e - c0);
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(&bars[1], nc * hrb);
      bulk_g2s(ht, p.hrec + static_cast<size_t>(p0 + c0) * hrb, nc * hrb, &bars[1]);
    }
    mbar_wait_bounded(&bars[1], phase, p.status);
    phase ^= 1u;
    if (c0 == 0) mbar_wait_bounded(&bars[0], 0, p.status);
#pragma unroll 1
    for (int q = warp; q < P; q += nw) {   // warp-uniform
      const int sb = q >> 1, h = q & 1;
      const uint8_t *w[R];
#pragma unroll
      for (int r = 0; r < R; ++r) w[r] = wbuf + (lane + 32 * r) * p.rb_d + sb * kQ4KBytes;
      float dv[R][kDnTok];
      q4k_half_dot_rows_tokens<R>(w, ht, hrb, p.I, sb, h, nc, dv);
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int i = 0; i < kDnTok; ++i)
          if (i < nc) part[(i * P + q) * kRows + lane + 32 * r] = dv[r][i];
    }
    __syncthreads();
    for (int v = threadIdx.x; v < nc * kRows; v += blockDim.x) {
      const int i = v / kRows, jl = v % kRows;
      float y = 0.f;
      for (int q = 0; q < P; ++q) y += part[(i * P + q) * kRows + jl];
      p.y[static_cast<size_t>(p0 + c0 + i) * p.H + j0 + jl] = y;
    }
    __syncthreads();   // part and the h tiles are reused by the next chunk
  }
}


// ===========================================================================
// Tensor-core mode (tcgen05, kind::f16): fp16 operands, fp32 accumulators in
// tensor memory. Weights are dequantised from Q4_K (w = d*sc*q - dmin*m in
// fp32, one rounding, then fp16) straight into K-major tiles; activations are
// fp16 (x exactly from bf16, h rounded from fp32).
// ===========================================================================
constexpr int kTcThreads = 256;
constexpr int kTcK = 256;                       // K elements per chunk (one super-block)
constexpr int kTcMaxN = 64;                     // tokens per pass
constexpr int kTcABytes = 128 * kTcK * 2;       // 64 KB
constexpr int kTcBBytes = kTcMaxN * kTcK * 2;   // 32 KB
constexpr int kTcSmem = 2 * kTcABytes + 2 * kTcBBytes + 64;
constexpr int kTcTmemCols = 64;

// Dequantise half `hf` (sub-blocks 4hf..4hf+3) of the Q4_K super-block at
// `sb` (global) into fp16 row `row` of a K-major tile of kTcK columns.
SI_DEV void dequant_half_to_tile(const uint8_t *sb, int hf, uint8_t *tile, int row) {
  const uint4 hd = __ldg(reinterpret_cast<const uint4 *>(sb));
  int sc8[8], mn8[8];
  const uint32_t sw[3] = {hd.y, hd.z, hd.w};
  q4k_unpack_scales(sw, sc8, mn8);
  const float d = half_bits_to_float(static_cast<uint16_t>(hd.x & 0xFFFF));
  const float dmin = half_bits_to_float(static_cast<uint16_t>(hd.x >> 16));
#pragma unroll
  for (int pp = 0; pp < 2; ++pp) {
    const int p = 2 * hf + pp;                        // code pair: sub-blocks 2p, 2p+1
    const int j_lo = 2 * p, j_hi = 2 * p + 1;
    const float s_lo = __fmul_rn(d, static_cast<float>(hf ? sc8[4 + 2 * pp] : sc8[2 * pp]));
    const float s_hi = __fmul_rn(d, static_cast<float>(hf ? sc8[5 + 2 * pp] : sc8[2 * pp + 1]));
    const float m_lo = __fmul_rn(dmin, static_cast<float>(hf ? mn8[4 + 2 * pp] : mn8[2 * pp]));
    const float m_hi = __fmul_rn(dmin, static_cast<float>(hf ? mn8[5 + 2 * pp] : mn8[2 * pp + 1]));
#pragma unroll
    for (int q16 = 0; q16 < 2; ++q16) {
      const uint4 c = __ldg(reinterpret_cast<const uint4 *>(sb + 16 + 32 * p + 16 * q16));
      const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int g = 0; g < 2; ++g) {                   // 8 elements per 16-byte store
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const uint32_t word = cw[2 * g + w];
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const uint32_t b0 = (word >> (16 * b)) & 0xFF, b1 = (word >> (16 * b + 8)) & 0xFF;
            lo[2 * w + b] = pack_half2(__fsub_rn(__fmul_rn(s_lo, static_cast<float>(b0 & 15)), m_lo),
                                       __fsub_rn(__fmul_rn(s_lo, static_cast<float>(b1 & 15)), m_lo));
            hi[2 * w + b] = pack_half2(__fsub_rn(__fmul_rn(s_hi, static_cast<float>(b0 >> 4)), m_hi),
                                       __fsub_rn(__fmul_rn(s_hi, static_cast<float>(b1 >> 4)), m_hi));
          }
        }
        const int e0 = 16 * q16 + 8 * g;              // element inside the sub-block
        *reinterpret_cast<uint4 *>(tile + kmajor_offset(row, 32 * j_lo + e0, kTcK)) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<uint4 *>(tile + kmajor_offset(row, 32 * j_hi + e0, kTcK)) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
      }
    }
  }
}

// Token rows (fp16, K chunk c) into a K-major tile; rows n >= nvalid are zero.
// Source row of tile row n: rows[n] (a global index array) or, when rows is
// null, row_base + n.
SI_DEV void tokens_to_tile(const __half *src, const int *rows, int row_base, int nvalid, int npad,
                           int ld, int k0, uint8_t *tile) {
  for (int idx = threadIdx.x; idx < npad * (kTcK / 8); idx += blockDim.x) {
    const int n = idx / (kTcK / 8), k8 = idx % (kTcK / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < nvalid) {
      const int r = rows ? __ldcg(rows + n) : row_base + n;
      v = __ldcg(reinterpret_cast<const uint4 *>(src + static_cast<size_t>(r) * ld + k0 + 8 * k8));
    }
    *reinterpret_cast<uint4 *>(tile + kmajor_offset(n, 8 * k8, kTcK)) = v;
  }
}

// One 128 x npad x (nchunks * 256) product into tensor memory, A rows given by
// `a_row_ptr(r)` (Q4_K rows, super-block c at +144 c), B rows by `tokens`.
// Double-buffered: the threads dequantise chunk c+1 while the tensor core
// multiplies chunk c. Returns false if a wait ran out.
template <typename RowPtr>
SI_DEV bool tc_product(RowPtr a_row_ptr, const __half *bsrc, const int *brows, int brow_base,
                       int nvalid, int npad, int ldb, int nchunks, uint8_t *smem, uint64_t *bars,
                       uint32_t *phase, uint32_t *pending, uint32_t taddr, uint32_t *status) {
  const uint32_t idesc = umma_idesc_f16_f32(128, npad);
  bool ok = true;
  for (int c = 0; c < nchunks; ++c) {
    const int b = c & 1;
    uint8_t *A = smem + b * kTcABytes;
    uint8_t *B = smem + 2 * kTcABytes + b * kTcBBytes;
    if (pending[b]) {   // uniform over the block
      ok &= mbar_wait_bounded(&bars[b], phase[b], status);
      phase[b] ^= 1u;
      pending[b] = 0;
      // a commit that never arrived: no more tiles, no more MMAs
      if (__syncthreads_or(!ok)) break;
    }
    {
      const int row = threadIdx.x >> 1, hf = threadIdx.x & 1;   // 256 threads: 128 rows x 2 halves
      dequant_half_to_tile(a_row_ptr(row) + c * kQ4KBytes, hf, A, row);
    }
    tokens_to_tile(bsrc, brows, brow_base, nvalid, npad, ldb, c * kTcK, B);
    fence_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      tc_fence_after();
      const uint32_t a0 = smem_addr(A), b0 = smem_addr(B);
#pragma unroll 4
      for (int ks = 0; ks < kTcK / 16; ++ks)
        umma_f16(taddr, umma_desc_kmajor(a0 + 256 * ks, 128, kTcK * 16),
                 umma_desc_kmajor(b0 + 256 * ks, 128, kTcK * 16), idesc, (c > 0 || ks > 0) ? 1u : 0u);
      umma_commit(&bars[b]);
    }
    pending[b] = 1;
  }
  // every commit still outstanding (also after a failed wait: the MMAs
  // already issued must finish before tensor memory is read or released)
  for (int b = 0; b < 2; ++b) {
    if (pending[b]) {
      ok &= mbar_wait_bounded(&bars[b], phase[b], status);
      phase[b] ^= 1u;
      pending[b] = 0;
    }
  }
  tc_fence_after();
  return !__syncthreads_or(!ok);
}

SI_DEV void tc_setup(uint8_t *smem, uint64_t *bars, uint32_t *s_taddr) {
  if (threadIdx.x < 32) {
    tmem_alloc(s_taddr, kTcTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

SI_DEV void tc_teardown(uint32_t taddr) {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(taddr, kTcTmemCols);
}

// gate/up: block = (active expert, 64 rows i0..i0+63): tile rows 0..63 are
// gate rows, 64..127 the same up rows, so lane r and lane r + 64 of the
// accumulator hold g and u of row i0 + r.
__global__ void __launch_bounds__(kTcThreads, 1) tc_gateup_kernel(BatchedParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 2 * kTcABytes + 2 * kTcBBytes);
  uint32_t *s_taddr = reinterpret_cast<uint32_t *>(bars + 2);
  grid_dep_wait();
  grid_dep_launch();
  const int tiles = p.I / 64;
  const int na = __ldcg(p.n_active);
  if (static_cast<int>(blockIdx.x) >= na * tiles) return;
  const int e = __ldcg(p.active + blockIdx.x / tiles);
  const int i0 = (blockIdx.x % tiles) * 64;
  const int n_e = __ldcg(p.count + e), p0 = __ldcg(p.offset + e);
  tc_setup(smem, bars, s_taddr);
  const uint32_t taddr = *s_taddr;
  uint32_t phase[2] = {0, 0}, pending[2] = {0, 0};
  const size_t rowbase = static_cast<size_t>(e) * p.I + i0;
  auto a_row = [&](int r) -> const uint8_t * {
    return r < 64 ? p.wg + (rowbase + r) * p.rb_gu : p.wu + (rowbase + r - 64) * p.rb_gu;
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *U = reinterpret_cast<float *>(smem);     // [64][kTcMaxN], reuses tile A0 after the MMAs
  for (int nc0 = 0; nc0 < n_e; nc0 += kTcMaxN) {
    const int nv = min(kTcMaxN, n_e - nc0), npad = (nv + 15) & ~15;
    // a timed-out commit (recorded in the status word): leave the
    // accumulators unread and the outputs unwritten
    if (!tc_product(a_row, p.xh, p.pair_token + p0 + nc0, 0, nv, npad, p.H, p.H / kTcK, smem, bars,
                    phase, pending, taddr, p.status))
      break;
    // Accumulator rows 64..127 (up) to shared memory, then rows 0..63 (gate) combine.
    if (warp >= 2 && warp < 4) {
      const int r = 32 * warp + lane - 64;
      for (int c8 = 0; c8 < npad; c8 += 8) {
        float v[8];
        tmem_ld8(taddr + (static_cast<uint32_t>(32 * warp) << 16) + c8, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) U[r * kTcMaxN + c8 + i] = v[i];
      }
    }
    __syncthreads();
    if (warp < 2) {
      const int r = 32 * warp + lane;
      for (int c8 = 0; c8 < npad; c8 += 8) {
        float v[8];
        tmem_ld8(taddr + (static_cast<uint32_t>(32 * warp) << 16) + c8, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int n = c8 + i;
          if (n < nv) {
            const float g = v[i], u = U[r * kTcMaxN + n];
            const float h = __fdiv_rn(g, 1.f + expf(-g)) * u;
            p.hh[static_cast<size_t>(p0 + nc0 + n) * p.I + i0 + r] = __float2half_rn(h);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  tc_teardown(taddr);
}

// down: block = (active expert, 128 output rows j0..j0+127).
__global__ void __launch_bounds__(kTcThreads, 1) tc_down_kernel(BatchedParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 2 * kTcABytes + 2 * kTcBBytes);
  uint32_t *s_taddr = reinterpret_cast<uint32_t *>(bars + 2);
  grid_dep_wait();
  grid_dep_launch();
  const int tiles = p.H / 128;
  const int na = __ldcg(p.n_active);
  if (static_cast<int>(blockIdx.x) >= na * tiles) return;
  const int e = __ldcg(p.active + blockIdx.x / tiles);
  const int j0 = (blockIdx.x % tiles) * 128;
  const int n_e = __ldcg(p.count + e), p0 = __ldcg(p.offset + e);
  tc_setup(smem, bars, s_taddr);
  const uint32_t taddr = *s_taddr;
  uint32_t phase[2] = {0, 0}, pending[2] = {0, 0};
  auto a_row = [&](int r) -> const uint8_t * {
    return p.wd + (static_cast<size_t>(e) * p.H + j0 + r) * p.rb_d;
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int nc0 = 0; nc0 < n_e; nc0 += kTcMaxN) {
    const int nv = min(kTcMaxN, n_e - nc0), npad = (nv + 15) & ~15;
    // h rows of this expert's pairs are contiguous: p0 + nc0 + n.
    if (!tc_product(a_row, p.hh, nullptr, p0 + nc0, nv, npad, p.I, p.I / kTcK, smem, bars, phase,
                    pending, taddr, p.status))
      break;
    if (warp < 4) {
      const int r = 32 * warp + lane;
      for (int c8 = 0; c8 < npad; c8 += 8) {
        float v[8];
        tmem_ld8(taddr + (static_cast<uint32_t>(32 * warp) << 16) + c8, v);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (c8 + i < nv) p.y[static_cast<size_t>(p0 + nc0 + c8 + i) * p.H + j0 + r] = v[i];
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  tc_teardown(taddr);
}

// Test: D = A * B^T for one 128 x n x k block (fp16 row-major inputs, k a
// multiple of 16 up to 256, n a multiple of 16 up to 64), through the same
// descriptors, MMA, commit and tensor-memory loads as the kernels above.
__global__ void __launch_bounds__(kTcThreads, 1) tc_test_kernel(const __half *a, const __half *b,
                                                               int n, int k, float *out,
                                                               uint32_t *status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 2 * kTcABytes + 2 * kTcBBytes);
  uint32_t *s_taddr = reinterpret_cast<uint32_t *>(bars + 2);
  tc_setup(smem, bars, s_taddr);
  const uint32_t taddr = *s_taddr;
  for (int idx = threadIdx.x; idx < 128 * (k / 8); idx += blockDim.x) {
    const int r = idx / (k / 8), k8 = idx % (k / 8);
    *reinterpret_cast<uint4 *>(smem + kmajor_offset(r, 8 * k8, kTcK)) =
        *reinterpret_cast<const uint4 *>(a + r * k + 8 * k8);
  }
  for (int idx = threadIdx.x; idx < n * (k / 8); idx += blockDim.x) {
    const int r = idx / (k / 8), k8 = idx % (k / 8);
    *reinterpret_cast<uint4 *>(smem + 2 * kTcABytes + kmajor_offset(r, 8 * k8, kTcK)) =
        *reinterpret_cast<const uint4 *>(b + r * k + 8 * k8);
  }
  fence_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    tc_fence_after();
    const uint32_t idesc = umma_idesc_f16_f32(128, n);
    for (int ks = 0; ks < k / 16; ++ks)
      umma_f16(taddr, umma_desc_kmajor(smem_addr(smem) + 256 * ks, 128, kTcK * 16),
               umma_desc_kmajor(smem_addr(smem + 2 * kTcABytes) + 256 * ks, 128, kTcK * 16), idesc,
               ks > 0 ? 1u : 0u);
    umma_commit(&bars[0]);
  }
  const bool ok = !__syncthreads_or(!mbar_wait_bounded(&bars[0], 0, status));
  tc_fence_after();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (ok && warp < 4) {   // a timed-out commit leaves the accumulator unread
    for (int c8 = 0; c8 < n; c8 += 8) {
      float v[8];
      tmem_ld8(taddr + (static_cast<uint32_t>(32 * warp) << 16) + c8, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) out[(32 * warp + lane) * n + c8 + i] = v[i];
    }
  }
  tc_teardown(taddr);
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(BatchedParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= p.T || j >= p.H) return;
  // the token's pair positions and weights, then its k rows all in flight,
  // then the fma chain in rank order
  int q[8];
  float w[8], yv[8];
#pragma unroll
  for (int r = 0; r < 8; ++r)
    if (r < p.k) {
      q[r] = __ldcg(p.pair_of + t * p.k + r);
      w[r] = __ldcg(p.wts + t * p.k + r);
    }
#pragma unroll
  for (int r = 0; r < 8; ++r)
    if (r < p.k) yv[r] = __ldcg(p.y + static_cast<size_t>(q[r]) * p.H + j);
  float acc = 0.f;
#pragma unroll
  for (int r = 0; r < 8; ++r)
    if (r < p.k) acc = fmaf(w[r], yv[r], acc);
  p.routed[static_cast<size_t>(t) * p.H + j] = __float2bfloat16_rn(acc);
}

// The batched layer's combine and residual norm in one pass: block t forms
// routed[t] (the combine kernel's fma chain in rank order and its bf16
// rounding; written out too) slice by slice as the norm row's input a, with
// b = the residual: the bits of the combine kernel followed by the norm
// kernel.
__global__ void __launch_bounds__(kNormThreads) combine_norm_kernel(BatchedParams p, BatchedNorm nm) {
  extern __shared__ float s_sum[];   // [H]
  __shared__ float s_red[kNormThreads / 32];
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.x;
  int q[8];
  float w[8];
#pragma unroll
  for (int r = 0; r < 8; ++r)
    if (r < p.k) {
      q[r] = __ldcg(p.pair_of + t * p.k + r);
      w[r] = __ldcg(p.wts + t * p.k + r);
    }
  __nv_bfloat16 *routed = p.routed + static_cast<size_t>(t) * p.H;
  auto load_routed = [&](int i0, float va[8]) {
    float4 yv[8][2];
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < p.k) {
        const float4 *src = reinterpret_cast<const float4 *>(p.y + static_cast<size_t>(q[r]) * p.H + i0);
        yv[r][0] = __ldcg(src);
        yv[r][1] = __ldcg(src + 1);
      }
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < p.k) {
        const float v[8] = {yv[r][0].x, yv[r][0].y, yv[r][0].z, yv[r][0].w,
                            yv[r][1].x, yv[r][1].y, yv[r][1].z, yv[r][1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(w[r], v[i], acc[i]);
      }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) va[i] = bf16_round(acc[i]);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = bf16_bits(va[2 * i]) | (static_cast<uint32_t>(bf16_bits(va[2 * i + 1])) << 16);
    *reinterpret_cast<uint4 *>(routed + i0) = make_uint4(o[0], o[1], o[2], o[3]);
  };
  add_rmsnorm_row(load_routed, static_cast<const __nv_bfloat16 *>(nm.residual), nullptr,
                  static_cast<const __nv_bfloat16 *>(nm.w_norm), p.H, nm.eps, t,
                  static_cast<__nv_bfloat16 *>(nm.sum_out), static_cast<__nv_bfloat16 *>(nm.norm_out), nullptr,
                  s_sum, s_red);
}

// Test export: the exact integer block sums of the batched helpers for
// n_vec activation vectors (the "tokens"), each super-block's code words
// loaded once for all of them, as the grouped kernels do: whole super-blocks
// (gate/up) or halves (down). out int32 [n_vec][rows][k / 32].
__global__ void tokens_block_dots_kernel(const uint8_t *w, int rows, int k, const uint8_t *a,
                                         int n_vec, int halves, int32_t *out) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int nsb = k / kQKK, nb = k / 32, rec = tile_record_bytes(k);
  for (int t = 0; t < n_vec; ++t)
    tile_from_q8_1(a + static_cast<size_t>(t) * nb * kQ81Bytes, k, tile_at(smem + t * rec, k));
  const int r = blockIdx.x;
  for (int sb = threadIdx.x; sb < nsb; sb += blockDim.x) {
    const uint4 *wv = reinterpret_cast<const uint4 *>(w + (static_cast<size_t>(r) * nsb + sb) * kQ4KBytes);
    int32_t *o = out + static_cast<size_t>(r) * nb + 8 * sb;
    if (!halves) {
#pragma unroll 1
      for (int pp = 0; pp < 4; ++pp) {
        uint32_t lo[8], hi[8];
        q4k_pair_nibbles(wv, pp, lo, hi);
        for (int t = 0; t < n_vec; ++t) {
          const uint4 *a = reinterpret_cast<const uint4 *>(smem + t * rec + sb * kActSbStride) + 4 * pp;
          const uint4 a4[4] = {a[0], a[1], a[2], a[3]};
          int slo, shi;
          q4k_pair_nibble_isums(lo, hi, a4, slo, shi);
          o[static_cast<size_t>(t) * rows * nb + 2 * pp] = slo;
          o[static_cast<size_t>(t) * rows * nb + 2 * pp + 1] = shi;
        }
      }
    } else {
      // halves: the same nibble functions, pair by pair as the down kernel
#pragma unroll 1
      for (int pp = 0; pp < 4; ++pp) {
        uint32_t lo[8], hi[8];
        q4k_pair_nibbles(wv, pp, lo, hi);
        for (int t = 0; t < n_vec; ++t) {
          const uint4 *a = reinterpret_cast<const uint4 *>(smem + t * rec + sb * kActSbStride) + 4 * pp;
          const uint4 a4[4] = {a[0], a[1], a[2], a[3]};
          int slo, shi;
          q4k_pair_nibble_isums(lo, hi, a4, slo, shi);
          o[static_cast<size_t>(t) * rows * nb + 2 * pp] = slo;
          o[static_cast<size_t>(t) * rows * nb + 2 * pp + 1] = shi;
        }
      }
    }
  }
}

si_status batched_test_dots(const void *w, int rows, int k, const void *a, int n_vec, int halves,
                            int32_t *out, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(n_vec) * tile_record_bytes(k);
  cudaError_t e = allow_smem(tokens_block_dots_kernel, smem);
  if (e == cudaSuccess)
    e = launch_pdl(tokens_block_dots_kernel, dim3(rows), dim3(128), smem, s,
                   static_cast<const uint8_t *>(w), rows, k, static_cast<const uint8_t *>(a), n_vec,
                   halves, out);
  return cuda_status(e);
}

// ---------------------------------------------------------------------------
struct BatchedGeom {
  size_t off_count, off_offset, off_active, off_nactive, off_pair_token, off_pair_of, off_xrec,
      off_hrec, off_y, off_xh, off_hh, bytes;
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
  take(g.off_xh, static_cast<size_t>(T) * L.hidden * 2);
  take(g.off_hh, P * L.inter * 2);
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
  if (L.expert_type != SI_Q4_K || down_type_of(L) != SI_Q4_K || L.shared_inter != 0)
    return SI_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * L.top_k > 1024) return SI_ERR_UNSUPPORTED;   // grouping buffer
  return SI_OK;
}

static size_t gateup_grouped_smem(const si_moe_layer &L) {
  return 64 + kGuTok * 64 * 4 + static_cast<size_t>(kGuTok) * tile_record_bytes(L.hidden) +
         64u * (L.hidden / 256 * kQ4KBytes);
}
static size_t down_grouped_smem(const si_moe_layer &L, int R) {
  const int P = 2 * (L.inter / 256), rows = 32 * R;
  return 64 + static_cast<size_t>(kDnTok) * rows * P * 4 +
         static_cast<size_t>(kDnTok) * tile_record_bytes(L.inter) +
         static_cast<size_t>(rows) * (L.inter / 256 * kQ4KBytes);
}
static int down_rows_per_lane(const si_moe_layer &L) {
  return down_grouped_smem(L, 2) <= 227 * 1024 ? 2 : 1;
}

cudaError_t preload_batched() {
  cudaFuncAttributes a;
  const void *ks[] = {reinterpret_cast<const void *>(batched_prep_kernel),
                      reinterpret_cast<const void *>(gateup_grouped_kernel),
                      reinterpret_cast<const void *>(down_grouped_kernel<1>),
                      reinterpret_cast<const void *>(down_grouped_kernel<2>),
                      reinterpret_cast<const void *>(tc_gateup_kernel),
                      reinterpret_cast<const void *>(tc_down_kernel),
                      reinterpret_cast<const void *>(combine_kernel),
                      reinterpret_cast<const void *>(combine_norm_kernel)};
  for (const void *k : ks) {
    const cudaError_t e = cudaFuncGetAttributes(&a, k);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

size_t batched_workspace_bytes(const si_moe_layer &L, int n_tokens) {
  return batched_geom(L, n_tokens).bytes;
}
si_status batched_validate(const si_moe_layer &L, int n_tokens) { return batched_check(L, n_tokens); }

// The combine step: alone, or with the layer's residual norm.
static cudaError_t launch_combine(const BatchedParams &p, const BatchedNorm *norm, cudaStream_t s) {
  if (!norm) return launch_pdl(combine_kernel, dim3((p.H + 255) / 256, p.T), dim3(256), 0, s, p);
  return launch_pdl(combine_norm_kernel, dim3(p.T), dim3(kNormThreads), sizeof(float) * p.H, s, p, *norm);
}

// Enqueue the batched routed FFN (arguments checked by the caller) into
// workspace `workspace`, device errors reported to `status`.
si_status batched_launch(const si_moe_layer *L, int n_tokens, int mode, const void *x,
                         const int32_t *topk_ids, const float *topk_w, void *routed_out,
                         void *workspace, uint32_t *status, cudaStream_t s, const BatchedNorm *norm) {
  // AUTO takes the integer path: measured faster than the tensor-core path at
  // every supported batch (1..128 tokens over 128 experts leave at most ~8
  // tokens per selected expert, so dequantising the weights to fp16 costs more
  // than the MMA saves).
  const bool tensor = mode == 2;
  const BatchedGeom g = batched_geom(*L, n_tokens);
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
  p.status = status;
  p.tensor = tensor ? 1 : 0;
  p.xh = reinterpret_cast<__half *>(base + g.off_xh);
  p.hh = reinterpret_cast<__half *>(base + g.off_hh);
  if (tensor) {
    if (L->hidden % 128 || L->inter % 256) return SI_ERR_UNSUPPORTED;
    const int max_active = n_tokens * L->top_k < L->n_experts ? n_tokens * L->top_k : L->n_experts;
    cudaError_t e = allow_smem(tc_gateup_kernel, kTcSmem);
    if (e == cudaSuccess) e = allow_smem(tc_down_kernel, kTcSmem);
    if (e == cudaSuccess)
      e = launch_pdl(batched_prep_kernel, dim3(1 + n_tokens), dim3(kPrepThreads), 0, s, p);
    if (e == cudaSuccess)
      e = launch_pdl(tc_gateup_kernel, dim3(max_active * (L->inter / 64)), dim3(kTcThreads),
                     kTcSmem, s, p);
    if (e == cudaSuccess)
      e = launch_pdl(tc_down_kernel, dim3(max_active * (L->hidden / 128)), dim3(kTcThreads),
                     kTcSmem, s, p);
    if (e == cudaSuccess)
      e = launch_combine(p, norm, s);
    return cuda_status(e);
  }
  const int R = down_rows_per_lane(*L);
  const int units = L->inter / 32, tiles = L->hidden / (32 * R);
  const int max_active = n_tokens * L->top_k < L->n_experts ? n_tokens * L->top_k : L->n_experts;
  const size_t gsm = gateup_grouped_smem(*L), dsm = down_grouped_smem(*L, R);
  if (gsm > 227 * 1024 || dsm > 227 * 1024) return SI_ERR_UNSUPPORTED;
  auto down = R == 2 ? down_grouped_kernel<2> : down_grouped_kernel<1>;
  const int P = 2 * (L->inter / 256);
  const int down_threads = 32 * (P < kDownBThreads / 32 ? P : kDownBThreads / 32);
  cudaError_t e = allow_smem(gateup_grouped_kernel, gsm);
  if (e == cudaSuccess) e = allow_smem(down, dsm);
  if (e == cudaSuccess)
    e = launch_pdl(batched_prep_kernel, dim3(1 + n_tokens), dim3(kPrepThreads), 0, s, p);
  if (e == cudaSuccess)
    e = launch_pdl(gateup_grouped_kernel, dim3(max_active * units), dim3(kGuBThreads), gsm, s, p);
  if (e == cudaSuccess)
    e = launch_pdl(down, dim3(max_active * tiles), dim3(down_threads), dsm, s, p);
  if (e == cudaSuccess)
    e = launch_combine(p, norm, s);
  return cuda_status(e);
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
  const si_status st = batched_check(*L, n_tokens);
  if (st != SI_OK) return st;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(topk_ids) & 3u) ||
      (reinterpret_cast<uintptr_t>(topk_w) & 3u) || (reinterpret_cast<uintptr_t>(routed_out) & 1u))
    return SI_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < batched_geom(*L, n_tokens).bytes)
    return SI_ERR_WORKSPACE;
  return batched_launch(L, n_tokens, mode, x, topk_ids, topk_w, routed_out, workspace,
                        static_cast<uint32_t *>(workspace), static_cast<cudaStream_t>(stream));
}

extern "C" si_status si_test_umma_f16(const void *a, const void *b, int n, int k, float *out,
                                      void *workspace, void *stream) {
  if (!a || !b || !out || !workspace || !aligned16(a) || !aligned16(b)) return SI_ERR_INVALID_ARG;
  if (n < 16 || n > kTcMaxN || n % 16 || k < 16 || k > kTcK || k % 16) return SI_ERR_INVALID_ARG;
  cudaError_t e = allow_smem(tc_test_kernel, kTcSmem);
  if (e == cudaSuccess)
    e = launch_pdl(tc_test_kernel, dim3(1), dim3(kTcThreads), kTcSmem,
                   static_cast<cudaStream_t>(stream), static_cast<const __half *>(a),
                   static_cast<const __half *>(b), n, k, out, static_cast<uint32_t *>(workspace));
  return cuda_status(e);
}
