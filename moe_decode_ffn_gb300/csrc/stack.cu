// Persistent layer-stack kernel: every layer of every token in one
// cooperative launch, one resident block per SM.
//
// "perf(qwen3.6): fuse decode kernel launches - shared-expert + GDN
// conv/L2-norm" (sparkinfer PR #239), Summary: decode is launch bound. Here
// one kernel body loops over tokens and layers; a layer's three all-to-all
// exchanges go through epoch-tagged lines in global memory instead of kernel
// boundaries:
//   X1 router logits  - every block writes the logits of its expert rows;
//                       every block gathers all of them and runs the top-k
//                       and softmax itself (same bits everywhere), so the
//                       grid completion handshake of "perf(qwen3.6): fused
//                       router GEMV+top-k + folded residual-norm (decode)"
//                       (PR #273, Summary item 1) becomes one gather;
//   X2 h codes        - each gate/up unit writes its 32 Q8_1 codes + scales;
//                       every block with down rows gathers all of them;
//   X3 output rows    - each block writes bf16(routed + shared) of its rows;
//                       every block gathers all rows and folds the residual +
//                       RMSNorm of the next layer itself (Summary item 2 of
//                       the same page).
// A line element is 8 bytes, {payload word, tag}, written and read as single
// 64-bit accesses, so a reader that sees the tag of this iteration also sees
// its payload: one load both proves readiness and delivers the data (no
// counter, flag or fence round trip). Every writer owns whole 128-byte slots
// and fills its slot with one coalesced store: slots shared by several
// writers, polled by every block, made those writes wait behind the polls. Tags are epoch + iteration + 1, the
// epoch advancing by the iteration count at the end of every launch, so lines
// left by an earlier launch never match. Lines are double-buffered by
// iteration parity: a block writes buffer (i & 1) at iteration i only after it
// has gathered every block's X3 line of iteration i - 1, which each block
// writes after it has finished reading everything of iteration i - 2.
//
// Weights that do not depend on the routing are requested ahead, by warps
// that are idle at that moment: the next layer's router rows, shared-gate
// vector and norm weights and this layer's shared down rows while the logits
// are gathered; the next shared-expert gate/up unit as soon as this one is
// consumed. Only the routed experts' bytes wait for the selection.
//
// Per-thread index arithmetic is hoisted out of the loop; the per-row
// arithmetic is the multi-kernel path's, so both give identical bits.
#include "common.cuh"
#include "host.hpp"
#include "topk.cuh"

namespace si {

SI_TRACE_BUFFER

constexpr int kStkThreads = 512;
constexpr int kSlot = 16;           // u64 elements per 128-byte slot
constexpr int kStkFixedBytes = 2048;
constexpr int kArmT = 480;          // the thread that arms every barrier (warp 15, lane 0)

struct StackLayerPtrs {             // 80 bytes
  const __nv_bfloat16 *w_router, *w_sg, *w_norm;
  const uint8_t *wg, *wu, *wd, *wsg, *wsu, *wsd;
  const void *pad;
};
static_assert(sizeof(StackLayerPtrs) == 80, "layer table entry is 80 bytes");

// Byte offsets into dynamic shared memory (after the fixed kStkFixedBytes).
struct StackSmem {
  uint32_t layers, resid, y, tbuf, part, xt_qs, xt_d, xt_s, ht_qs, ht_d, ht_s, pbuf, pbuf_stride, gu,
      dn, sd, bytes;
};

struct StackParams {
  const StackLayerPtrs *layers;
  int n_layers, n_tokens;
  int H, E, k, I, Is;         // Is == 0: no shared expert
  int rb, rbd, rbsd;          // row bytes: gate/up rows (H), routed down rows (I), shared down rows
  int J;                      // down output rows per block (even)
  int W;                      // router: warps per expert row
  int nch;                    // router: 16-byte vectors per lane
  int np3;                    // X3: pairs of elements per block slot (ceil(J / 4))
  float eps;
  StackSmem sm;
  const __nv_bfloat16 *x_in;  // [T][H]
  __nv_bfloat16 *y_out, *sum_out;   // [T][H]
  int32_t *ids_out;           // [T][L][k] or null
  uint32_t *status;
  uint32_t *epoch;            // tag base
  uint64_t *lg;               // X1 [2][G][kSlot]: {logit row c, logit row c + G}
  uint64_t *hl;               // X2 [2][units][kSlot]: 8 code words, {d16 | s16 << 16}, pad
  uint64_t *ol;               // X3 [2][G][kSlot]: bf16 pairs of this block's rows
};

// ---- tagged lines ----------------------------------------------------------
SI_DEV uint64_t tagged(uint32_t tag, uint32_t payload) {
  return (static_cast<uint64_t>(tag) << 32) | payload;
}
SI_DEV bool tag_ok(uint64_t v, uint32_t tag) { return static_cast<uint32_t>(v >> 32) == tag; }
SI_DEV void st_tag1(uint64_t *p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
SI_DEV void st_tag2(uint64_t *p, uint64_t a, uint64_t b) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
// Two elements (16-byte aligned); each 64-bit element is read atomically.
SI_DEV void ld_tag2(const uint64_t *p, uint64_t &a, uint64_t &b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p)
               : "memory");
}
SI_DEV bool pair_ok(uint64_t a, uint64_t b, uint32_t tag) { return tag_ok(a, tag) && tag_ok(b, tag); }

// Re-read the pair at p until both elements carry `tag`, at most
// kWaitBudgetNs; records SI_ERR_TIMEOUT and returns false if they never do.
static __device__ __noinline__ bool poll_pair(const uint64_t *p, uint32_t tag, uint64_t &a,
                                              uint64_t &b, uint32_t *status,
                                              uint64_t budget_ns = kWaitBudgetNs) {
  const uint64_t t0 = now_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i) {
      ld_tag2(p, a, b);
      if (pair_ok(a, b, tag)) return true;
    }
    if (now_ns() - t0 > budget_ns) {
      record_status(status, SI_ERR_TIMEOUT);
      return false;
    }
  }
}
// a, b: the pair as loaded already; polls only if it is not there yet.
SI_DEV bool get_pair(const uint64_t *p, uint32_t tag, uint64_t &a, uint64_t &b, uint32_t *status) {
  return pair_ok(a, b, tag) || poll_pair(p, tag, a, b, status);
}

// Q8_1 of 32 values held 4 per lane by 8 consecutive lanes: d = amax / 127,
// q = round-half-away(v / d) clamped to +-127, d16 = fp16(d),
// s16 = fp16(d * sum q) (the definition every encoder of the library follows).
SI_DEV uint32_t q8_1_encode_8lanes(const float v[4], uint16_t &d16, uint16_t &s16) {
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  const float d = __fdiv_rn(amax, 127.0f);
  const bool live = d > 0.f;
  const float dd = live ? d : 1.0f;
  uint32_t packed = 0u;
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float r = fminf(fmaxf(roundf(__fdiv_rn(v[i], dd)), -127.f), 127.f);
    const int q = live ? static_cast<int>(r) : 0;
    sum += q;
    packed |= static_cast<uint32_t>(q & 0xFF) << (8 * i);
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  sum += __shfl_xor_sync(0xffffffffu, sum, 4);
  d16 = float_to_half_bits(d);
  s16 = float_to_half_bits(__fmul_rn(d, static_cast<float>(sum)));
  return packed;
}

// y (n floats, bf16 values, shared memory) -> Q8_1 activation tile, 4 values
// per thread. Ends with __syncthreads.
SI_DEV void quantize_y(const float *y, int n, ActTile t) {
#pragma unroll 1
  for (int g = threadIdx.x; g < n / 4; g += blockDim.x) {   // n / 4 is a multiple of blockDim
    const float4 v4 = *reinterpret_cast<const float4 *>(y + 4 * g);
    const float v[4] = {v4.x, v4.y, v4.z, v4.w};
    uint16_t d16, s16;
    const uint32_t q = q8_1_encode_8lanes(v, d16, s16);
    const int blk = g >> 3, part = g & 7;
    *reinterpret_cast<uint32_t *>(t.qs + (blk >> 3) * kActSbStride + (blk & 7) * 32 + part * 4) = q;
    if (part == 0) {
      t.d[blk] = half_bits_to_float(d16);
      t.s[blk] = half_bits_to_float(s16);
    }
  }
  __syncthreads();
}

// sum_h w_sg[h] * y[h], the same thread mapping and order as the down
// kernel's block_dot_bf16 over 512 threads.
SI_DEV float sigma_dot(const __nv_bfloat16 *w, const float *y, int n, float *red) {
  float acc = 0.f;
#pragma unroll 1
  for (int i0 = 8 * threadIdx.x; i0 < n; i0 += 8 * blockDim.x) {
    float wv[8];
    Load8<__nv_bfloat16>::run(w + i0, wv);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(wv[i], y[i0 + i], acc);
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  float tot = 0.f;
#pragma unroll 1
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) tot += red[i];
  __syncthreads();
  return tot;
}

// ---- copies ---------------------------------------------------------------------
// Issuing one bulk copy occupies the issuing thread for a few hundred cycles
// whatever its size, so copies are few and large, and are issued one per
// warp (lane 0) by warps that have nothing else to do at that moment. One
// thread (kArmT) arms every barrier (arrive + expected bytes) before a
// __syncthreads that precedes the copies.
SI_DEV void arm(uint64_t *bars, int b, uint32_t bytes, uint32_t &armed, uint32_t &used) {
  mbar_arrive_expect_tx(&bars[b], bytes);
  armed ^= 1u << b;
  used |= 1u << b;
}

// Gather X3 (t = bf16(routed + shared) per row) into `tbuf`, then fold it
// into the residual: s = bf16(t + resid), y = bf16((s * rsqrt(mean(s^2) +
// eps)) * w), the norm kernel's arithmetic and order (the first 256 threads
// own rows 8i..8i+7 of every 2048-row slice). Thread i reads pairs i and
// i + 512 of the slots: f_src = element offset, f_row = first row, f_n = rows
// of this block in the pair (0 for a pair that only proves presence).
// `resid` holds the residual on entry and s on exit. Returns false (in every
// thread) if a slot did not arrive in time.
SI_DEV bool fold_norm(const StackParams &p, const uint64_t *ol, uint32_t tag, float *resid,
                      const __nv_bfloat16 *w, float *y, float *tbuf, float *red,
                      const int f_src[2], const int f_row[2], const int f_n[2]) {
  const int H = p.H;
  bool ok = true;
  uint64_t v[2][2];
#pragma unroll
  for (int s = 0; s < 2; ++s)
    if (f_src[s] >= 0) ld_tag2(ol + f_src[s], v[s][0], v[s][1]);
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    if (f_src[s] < 0) continue;
    ok &= get_pair(ol + f_src[s], tag, v[s][0], v[s][1], p.status);
    SI_TRACE_LATEST(0, 13);
    const uint32_t w0 = static_cast<uint32_t>(v[s][0]), w1 = static_cast<uint32_t>(v[s][1]);
    const float tv[4] = {bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1)};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < f_n[s]) tbuf[f_row[s] + e] = tv[e];
  }
  if (__syncthreads_or(!ok)) return false;
  if (threadIdx.x < 256) {
    float ss = 0.f;
#pragma unroll 1
    for (int r0 = 8 * threadIdx.x; r0 < H; r0 += 2048) {
      const float4 t0 = *reinterpret_cast<const float4 *>(tbuf + r0);
      const float4 t1 = *reinterpret_cast<const float4 *>(tbuf + r0 + 4);
      const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float sv = bf16_round(tv[e] + resid[r0 + e]);
        ss = fmaf(sv, sv, ss);
        resid[r0 + e] = sv;
      }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  }
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += red[i];
  const float r = rsqrtf(__fdiv_rn(tot, static_cast<float>(H)) + p.eps);
#pragma unroll 1
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    y[i] = bf16_round(__fmul_rn(__fmul_rn(resid[i], r), __bfloat162float(w[i])));
  __syncthreads();
  return true;
}

template <int SFMT>
__global__ void __launch_bounds__(kStkThreads, 1) stack_kernel(StackParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr bool kShared = SFMT != 0;
  const int G = gridDim.x, c = blockIdx.x;
  const int H = p.H, I = p.I, Is = kShared ? p.Is : 0, k = p.k, E = p.E;
  const int nsb = H / kQKK;
  const int n_slots = k + (kShared ? 1 : 0);
  const int units_r = k * I / 32, units = units_r + Is / 32;
  const int nsb_r = I / kQKK, nsb_s = Is / kQKK;
  const int P_r = 2 * nsb_r, P_s = kShared ? 2 * nsb_s : 1, P_max = P_r > P_s ? P_r : P_s;
  const int n_iters = p.n_tokens * p.n_layers;
  const int J = p.J;

  // ---- shared memory --------------------------------------------------------
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);   // 0,1 prefetch groups; 2..5 gate/up groups; 6 routed down; 7 shared down
  uint32_t *s_base = reinterpret_cast<uint32_t *>(smem + 128);
  float *red = reinterpret_cast<float *>(smem + 144);
  float *s_part = reinterpret_cast<float *>(smem + 208);
  float *s_wts = reinterpret_cast<float *>(smem + 240);
  uint64_t *s_sel = reinterpret_cast<uint64_t *>(smem + 304);
  uint64_t *s_cand = reinterpret_cast<uint64_t *>(smem + 368);
  float *h_s = reinterpret_cast<float *>(smem + 880);
  float *s_logit = reinterpret_cast<float *>(smem + 1024);
  StackLayerPtrs *s_layers = reinterpret_cast<StackLayerPtrs *>(smem + p.sm.layers);
  float *resid = reinterpret_cast<float *>(smem + p.sm.resid);
  float *y = reinterpret_cast<float *>(smem + p.sm.y);
  float *tbuf = reinterpret_cast<float *>(smem + p.sm.tbuf);
  float *part = reinterpret_cast<float *>(smem + p.sm.part);
  const ActTile xt{smem + p.sm.xt_qs, reinterpret_cast<float *>(smem + p.sm.xt_d),
                   reinterpret_cast<float *>(smem + p.sm.xt_s)};
  const ActTile ht{smem + p.sm.ht_qs, reinterpret_cast<float *>(smem + p.sm.ht_d),
                   reinterpret_cast<float *>(smem + p.sm.ht_s)};
  uint8_t *pbuf = smem + p.sm.pbuf;   // [2]: router rows (2 x H bf16), w_sg (H), w_norm (H)
  const uint32_t pstr = p.sm.pbuf_stride;
  uint8_t *gu_buf = smem + p.sm.gu;   // gate [32] + up [32] rows
  uint8_t *dn_buf = smem + p.sm.dn;   // [k][J] routed down rows
  uint8_t *sd_buf = smem + p.sm.sd;   // [J] shared down rows

  // ---- static assignment ----------------------------------------------------
  const int my_unit = c < units ? c : -1;
  const bool shared_unit = kShared && my_unit >= units_r;
  const int j0 = c * J;
  const int nrows = j0 < H ? min(J, H - j0) : 0;
  const int row_a = c, row_b = c + G;   // router rows of this block
  const int nrr = (row_a < E ? 1 : 0) + (p.W == 4 && row_b < E ? 1 : 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rs = warp / p.W, wpart = warp % p.W;               // router: row, K part
  const int pr = threadIdx.x >> 4, gm = (threadIdx.x >> 3) & 1, lane8 = threadIdx.x & 7;   // gate/up
  const uint64_t pol = policy_evict_first();
  // X2 gather: pair q (5 per unit slot: 4 code pairs, 1 scale pair) ->
  // element offset g_q and shared memory destination g_dst (byte offset of 8
  // codes, or -(unit + 1) for the scales)
  int g_q[2], g_dst[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int q = static_cast<int>(threadIdx.x) + s * kStkThreads;
    const int u = q / 5, sub = q - 5 * (q / 5);
    g_q[s] = q < units * 5 ? u * kSlot + 2 * sub : -1;   // element offset of the pair
    const int base_sb = u < units_r ? (u / (I / 32)) * nsb_r : k * nsb_r;
    const int hb = u < units_r ? u % (I / 32) : u - units_r;
    g_dst[s] = sub < 4 ? static_cast<int>(p.sm.ht_qs) + (base_sb + hb / 8) * kActSbStride + (hb % 8) * 32 + 8 * sub
                       : -(u + 1);
  }
  // down: item (slot r, row jl, half-super-block qq) of this thread
  int d_row[2], d_act[2], d_blk[2], d_h[2], d_part[2];
  {
    const int items_r = k * J * P_r;
    const int items = items_r + (kShared ? J * P_s : 0);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int u = static_cast<int>(threadIdx.x) + s * kStkThreads;
      int r, jl, qq;
      if (u < items_r) {
        r = u / (J * P_r);
        const int rem = u - r * (J * P_r);
        jl = rem / P_r;
        qq = rem - jl * P_r;
      } else {
        r = k;
        jl = (u - items_r) / P_s;
        qq = (u - items_r) - jl * P_s;
      }
      const bool sh = kShared && r == k;
      const int sb = qq >> 1;
      d_part[s] = (u < items && jl < nrows) ? (r * J + jl) * P_max + qq : -1;
      d_row[s] = (sh ? static_cast<int>(p.sm.sd) + jl * p.rbsd
                     : static_cast<int>(p.sm.dn) + (r * J + jl) * p.rbd) + sb * kQ4KBytes;
      d_act[s] = static_cast<int>(p.sm.ht_qs) + (r * nsb_r + sb) * kActSbStride;
      d_blk[s] = (r * I) / 32 + 8 * sb;
      d_h[s] = qq & 1;
    }
  }
  // X3 gather: pair q = (block b, m) holds rows b * J + 4m .. + 3
  int f_src[2], f_row[2], f_n[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int q = static_cast<int>(threadIdx.x) + s * kStkThreads;
    const int b = q / p.np3, m = q - b * p.np3;
    const int r0 = b * J + 4 * m;
    f_src[s] = q < G * p.np3 ? b * kSlot + 2 * m : -1;
    f_row[s] = r0;
    f_n[s] = max(0, min(min(4, J - 4 * m), H - r0));
  }
  // combine: slot tr, row tj
  const int tr = static_cast<int>(threadIdx.x) / J, tj = static_cast<int>(threadIdx.x) - tr * J;
  const bool tlive = static_cast<int>(threadIdx.x) < n_slots * J && tj < nrows;
  const int tPP = (kShared && tr == k) ? P_s : P_r;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    *s_base = __ldcg(p.epoch);
  }
  {
    const unsigned long long *src = reinterpret_cast<const unsigned long long *>(p.layers);
    unsigned long long *dst = reinterpret_cast<unsigned long long *>(s_layers);
#pragma unroll 1
    for (int i = threadIdx.x; i < p.n_layers * 10; i += blockDim.x) dst[i] = __ldg(src + i);
  }
  __syncthreads();
  const uint32_t base = *s_base;

  // Thread kArmT: `armed` holds, per barrier, the parity of the number of
  // phases armed so far, `used` which barriers were ever armed. On an error
  // exit it waits for the last armed phase of each, so no copy is left in
  // flight.
  uint32_t armed = 0u, used = 0u;
  int t = 0, l = 0;   // token and layer of iteration it
  const uint32_t gbytes = static_cast<uint32_t>((nrr + (kShared ? 1 : 0) + 1) * H * 2);
  const uint32_t gubytes = 8u * p.rb;    // one group: 8 gate (or up) rows
  if (threadIdx.x == kArmT && n_iters > 0) {
    // iteration 0's routing-independent bytes and shared gate/up unit
    const StackLayerPtrs &L0 = s_layers[0];
    arm(bars, 0, gbytes, armed, used);
    if (nrr > 0) bulk_g2s(pbuf, L0.w_router + static_cast<size_t>(row_a) * H, H * 2, &bars[0]);
    if (nrr > 1) bulk_g2s(pbuf + 2 * H, L0.w_router + static_cast<size_t>(row_b) * H, H * 2, &bars[0]);
    if (kShared) bulk_g2s(pbuf + 4 * H, L0.w_sg, H * 2, &bars[0]);
    bulk_g2s(pbuf + 6 * H, L0.w_norm, H * 2, &bars[0]);
    if (shared_unit) {
      const size_t row0 = static_cast<size_t>(my_unit - units_r) * 32;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        arm(bars, 2 + g, 2 * gubytes, armed, used);
        bulk_g2s_evict_first(gu_buf + g * gubytes, L0.wsg + (row0 + 8 * g) * p.rb, gubytes, &bars[2 + g], pol);
        bulk_g2s_evict_first(gu_buf + (4 + g) * gubytes, L0.wsu + (row0 + 8 * g) * p.rb, gubytes,
                             &bars[2 + g], pol);
      }
    }
  }

  for (int it = 0;; ++it) {
    const uint32_t tag = base + static_cast<uint32_t>(it) + 1u, par = it & 1u;
    SI_TRACE_MARK(0, 0);
    if (threadIdx.x == kArmT && it < n_iters) {   // copies issued during this iteration's logit gather
      if (it + 1 < n_iters) arm(bars, (it + 1) & 1, gbytes, armed, used);
      if (kShared && nrows > 0) arm(bars, 7, static_cast<uint32_t>(nrows) * p.rbsd, armed, used);
    }
    // [N] FFN input: the fold of the previous iteration's outputs (at a
    // token's first layer, those are the previous token's results), or x_in.
    if (it > 0) {
      const uint8_t *pb = pbuf + ((it - 1) & 1) * pstr;
      if (!fold_norm(p, p.ol + static_cast<size_t>((it - 1) & 1) * G * kSlot, tag - 1u, resid,
                     reinterpret_cast<const __nv_bfloat16 *>(pb + 6 * H), y, tbuf, red, f_src, f_row,
                     f_n))
        goto fail;
      if (l == 0) {
#pragma unroll 1
        for (int i = threadIdx.x; i < nrows; i += blockDim.x) {
          p.y_out[static_cast<size_t>(t - 1) * H + j0 + i] = __float2bfloat16_rn(y[j0 + i]);
          if (p.sum_out)
            p.sum_out[static_cast<size_t>(t - 1) * H + j0 + i] = __float2bfloat16_rn(resid[j0 + i]);
        }
        __syncthreads();   // y and resid are overwritten below
      }
    }
    if (it == n_iters) break;
    if (l == 0) {
#pragma unroll 1
      for (int i = threadIdx.x; i < H; i += blockDim.x) {
        const float v = __bfloat162float(p.x_in[static_cast<size_t>(t) * H + i]);
        resid[i] = v;
        y[i] = v;
      }
      __syncthreads();
    }
    SI_TRACE_MARK(0, 1);

    // [R] router rows: W warps per row, vector (i * W + wpart) * 32 + lane
    {
      const bool ok = mbar_wait_bounded(&bars[par], (it >> 1) & 1, p.status);
      if (ok && rs < nrr) {
        const uint4 *wrow = reinterpret_cast<const uint4 *>(pbuf + par * pstr + rs * 2 * H);
        float acc = 0.f;
#pragma unroll 1
        for (int i = 0; i < p.nch; ++i) {
          const int v = (i * p.W + wpart) * 32 + lane;
          const uint4 u = wrow[v];
          float wv[8];
          Load8<__nv_bfloat16>::run(&u, wv);
          const float4 y0 = *reinterpret_cast<const float4 *>(y + 8 * v);
          const float4 y1 = *reinterpret_cast<const float4 *>(y + 8 * v + 4);
          acc = fmaf(wv[0], y0.x, acc);
          acc = fmaf(wv[1], y0.y, acc);
          acc = fmaf(wv[2], y0.z, acc);
          acc = fmaf(wv[3], y0.w, acc);
          acc = fmaf(wv[4], y1.x, acc);
          acc = fmaf(wv[5], y1.y, acc);
          acc = fmaf(wv[6], y1.z, acc);
          acc = fmaf(wv[7], y1.w, acc);
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (lane == 0) s_part[rs * p.W + wpart] = acc;
      }
      if (__syncthreads_or(!ok)) goto fail;
      if (threadIdx.x == 0) {
        float lg[2] = {0.f, 0.f};
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
          if (rr < nrr) {
            lg[rr] = s_part[rr * p.W];
#pragma unroll 1
            for (int w = 1; w < p.W; ++w) lg[rr] += s_part[rr * p.W + w];
          }
        st_tag2(p.lg + (static_cast<size_t>(par) * G + c) * kSlot, tagged(tag, __float_as_uint(lg[0])),
                tagged(tag, __float_as_uint(lg[1])));
      }
    }
    // the gate/up activations, while the logits travel
    quantize_y(y, H, xt);   // ends with __syncthreads
    SI_TRACE_MARK(0, 2);

    // [S] gather every logit; top-k + softmax in every block
    {
      bool ok = true;
      if (static_cast<int>(threadIdx.x) < G && static_cast<int>(threadIdx.x) < E) {
        const uint64_t *q = p.lg + (static_cast<size_t>(par) * G + threadIdx.x) * kSlot;
        uint64_t a, b;
        ld_tag2(q, a, b);
        ok = get_pair(q, tag, a, b, p.status);
        SI_TRACE_LATEST(0, 8);
        s_logit[threadIdx.x] = __uint_as_float(static_cast<uint32_t>(a));
        if (static_cast<int>(threadIdx.x) + G < E)
          s_logit[threadIdx.x + G] = __uint_as_float(static_cast<uint32_t>(b));
      } else if (lane == 0) {
        // warps without a slot to poll: the next iteration's router rows,
        // shared-gate vector and norm weights; this iteration's shared down
        // rows; and the arming of this iteration's routed copies
        if (threadIdx.x == kArmT) {
          if (my_unit >= 0 && !shared_unit)
#pragma unroll 1
            for (int g = 0; g < 4; ++g) arm(bars, 2 + g, 2 * gubytes, armed, used);
          if (nrows > 0) arm(bars, 6, static_cast<uint32_t>(k * nrows * p.rbd), armed, used);
        }
        const StackLayerPtrs &Ln = s_layers[l + 1 == p.n_layers ? 0 : l + 1];
        uint8_t *dst = pbuf + ((it + 1) & 1) * pstr;
        uint64_t *bar = &bars[(it + 1) & 1];
        const bool next = it + 1 < n_iters;
        if (warp == 12 && next && nrr > 0)
          bulk_g2s(dst, Ln.w_router + static_cast<size_t>(row_a) * H, H * 2, bar);
        if (warp == 13 && next && nrr > 1)
          bulk_g2s(dst + 2 * H, Ln.w_router + static_cast<size_t>(row_b) * H, H * 2, bar);
        if (warp == 14 && next && kShared) bulk_g2s(dst + 4 * H, Ln.w_sg, H * 2, bar);
        if (warp == 15 && next) bulk_g2s(dst + 6 * H, Ln.w_norm, H * 2, bar);
        if (warp == 11 && kShared && nrows > 0)
          bulk_g2s_evict_first(sd_buf, s_layers[l].wsd + static_cast<size_t>(j0) * p.rbsd,
                               static_cast<uint32_t>(nrows) * p.rbsd, &bars[7], pol);
      }
      if (__syncthreads_or(!ok)) goto fail;
    }
    SI_TRACE_MARK(0, 3);
    if (warp < 8) {
      const int ex = threadIdx.x;
      const uint64_t key = warp_sort32(ex < E ? make_key(s_logit[ex], ex) : 0ull, lane);
      if (lane < 8) s_cand[warp * 8 + lane] = key;
    }
    SI_TRACE_MARK(0, 9);
    __syncthreads();
    {
      // rank of candidate tid / 8 among the 64: 8 threads compare 8 each
      const uint64_t me = s_cand[threadIdx.x >> 3];
      const int j0c = 8 * (threadIdx.x & 7);
      int rank = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) rank += s_cand[j0c + j] > me;
      rank += __shfl_xor_sync(0xffffffffu, rank, 1);
      rank += __shfl_xor_sync(0xffffffffu, rank, 2);
      rank += __shfl_xor_sync(0xffffffffu, rank, 4);
      if ((threadIdx.x & 7) == 0 && rank < k && me != 0ull) s_sel[rank] = me;
    }
    __syncthreads();
    SI_TRACE_MARK(0, 10);
    // routed bytes, one copy per warp: warps 0..7 this block's gate/up unit
    // (warp w: group w & 3 of the gate (w < 4) or up rows, 8 rows each),
    // warps 8 .. 8 + k - 1 its down rows of each selected expert; a block with
    // a gate/up unit issues the down rows only once it has consumed its own
    // gate/up rows, so that they do not compete with the more urgent bytes
    if (lane == 0) {
      const StackLayerPtrs &Lp = s_layers[l];
      if (warp < 8 && my_unit >= 0 && !shared_unit) {
        const int slot = my_unit / (I / 32), hb = my_unit - slot * (I / 32);
        int e = key_index(s_sel[slot]);
        if (e < 0 || e >= E) e = 0;
        const size_t row0 = static_cast<size_t>(e) * I + static_cast<size_t>(hb) * 32 + 8 * (warp & 3);
        bulk_g2s_evict_first(gu_buf + warp * gubytes, (warp < 4 ? Lp.wg : Lp.wu) + row0 * p.rb,
                             gubytes, &bars[2 + (warp & 3)], pol);
      }
      if (warp >= 8 && warp < 8 + k && nrows > 0 && my_unit < 0) {
        int e = key_index(s_sel[warp - 8]);
        if (e < 0 || e >= E) e = 0;
        bulk_g2s_evict_first(dn_buf + static_cast<size_t>(warp - 8) * J * p.rbd,
                             Lp.wd + (static_cast<size_t>(e) * H + j0) * p.rbd,
                             static_cast<uint32_t>(nrows) * p.rbd, &bars[6], pol);
      }
    }
    SI_TRACE_MARK(0, 4);

    // [G] gate/up of this block's unit -> h line
    if (my_unit >= 0) {
      float acc = 0.f;
      const bool ok = mbar_wait_bounded(&bars[2 + (pr >> 3)], par, p.status);
      if (ok) {
        const uint8_t *row = gu_buf + (gm * 32 + pr) * p.rb;
        for (int sb = lane8; sb < nsb; sb += 8)
          acc += q4k_sb_dot(reinterpret_cast<const uint4 *>(row + sb * kQ4KBytes),
                            reinterpret_cast<const uint4 *>(xt.qs + sb * kActSbStride), xt.d + 8 * sb,
                            xt.s + 8 * sb);
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      const float other = __shfl_xor_sync(0xffffffffu, acc, 8);
      if ((threadIdx.x & 15) == 0) h_s[pr] = __fdiv_rn(acc, 1.f + expf(-acc)) * other;
      if (threadIdx.x == kArmT && shared_unit && it + 1 < n_iters)
#pragma unroll 1
        for (int g = 0; g < 4; ++g) arm(bars, 2 + g, 2 * gubytes, armed, used);
      if (__syncthreads_or(!ok)) goto fail;
      if (lane == 0 && warp >= 8 && warp < 8 + k && nrows > 0) {
        // the down rows, now that this block's gate/up rows are in: they are
        // needed only after the h exchange
        const StackLayerPtrs &Lp = s_layers[l];
        int e = key_index(s_sel[warp - 8]);
        if (e < 0 || e >= E) e = 0;
        bulk_g2s_evict_first(dn_buf + static_cast<size_t>(warp - 8) * J * p.rbd,
                             Lp.wd + (static_cast<size_t>(e) * H + j0) * p.rbd,
                             static_cast<uint32_t>(nrows) * p.rbd, &bars[6], pol);
      }
      if (lane == 0 && warp >= 8 && shared_unit && it + 1 < n_iters) {
        // the next iteration's shared gate/up unit (warps 8..15, one group each)
        const StackLayerPtrs &Ln = s_layers[l + 1 == p.n_layers ? 0 : l + 1];
        const int w = warp - 8;
        const size_t row0 = static_cast<size_t>(my_unit - units_r) * 32 + 8 * (w & 3);
        bulk_g2s_evict_first(gu_buf + w * gubytes, (w < 4 ? Ln.wsg : Ln.wsu) + row0 * p.rb, gubytes,
                             &bars[2 + (w & 3)], pol);
      }
      if (warp == 0) {
        uint16_t d16, s16;
        const uint32_t q = static_cast<uint32_t>(q8_1_encode_warp(h_s[lane], d16, s16)) & 0xFFu;
        const uint32_t w = q | (__shfl_down_sync(0xffffffffu, q, 1) << 8) |
                           (__shfl_down_sync(0xffffffffu, q, 2) << 16) |
                           (__shfl_down_sync(0xffffffffu, q, 3) << 24);   // lane 4j: code word j
        // lane j < 4: words 2j, 2j + 1; lane 4: scales; one coalesced store
        const uint32_t wa = __shfl_sync(0xffffffffu, w, (8 * lane) & 31);
        const uint32_t wb = __shfl_sync(0xffffffffu, w, (8 * lane + 4) & 31);
        uint64_t *line = p.hl + (static_cast<size_t>(par) * units + my_unit) * kSlot;
        if (lane < 4)
          st_tag2(line + 2 * lane, tagged(tag, wa), tagged(tag, wb));
        else if (lane == 4)
          st_tag2(line + 8, tagged(tag, static_cast<uint32_t>(d16) | (static_cast<uint32_t>(s16) << 16)),
                  tagged(tag, 0u));
      }
    }
    if (warp == 1) {   // softmax over the selected logits, summed in rank order
      const int r = lane < k ? lane : 0;
      const float ex = expf(key_value(s_sel[r]) - key_value(s_sel[0]));
      float sum = 0.f;
#pragma unroll 1
      for (int q = 0; q < k; ++q) sum += __shfl_sync(0xffffffffu, ex, q);
      if (lane < k) {
        s_wts[lane] = ex * __frcp_rn(sum);
        if (c == 0 && p.ids_out) {
          int e = key_index(s_sel[lane]);
          p.ids_out[static_cast<size_t>(it) * k + lane] = (e < 0 || e >= E) ? 0 : e;
        }
      }
    }
    SI_TRACE_MARK(0, 5);
    float sigma = 0.f;
    if (kShared && nrows > 0) {
      const __nv_bfloat16 *wsg = reinterpret_cast<const __nv_bfloat16 *>(pbuf + par * pstr + 4 * H);
      sigma = __fdiv_rn(1.f, 1.f + expf(-sigma_dot(wsg, y, H, red)));
    }

    // [D] gather h, down for this block's rows -> X3 line
    if (nrows > 0) {
      bool ok = true;
      {
        const uint64_t *hl = p.hl + static_cast<size_t>(par) * units * kSlot;
        uint64_t v[2][2];
#pragma unroll
        for (int s = 0; s < 2; ++s)
          if (g_q[s] >= 0) ld_tag2(hl + g_q[s], v[s][0], v[s][1]);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (g_q[s] < 0) continue;
          ok &= get_pair(hl + g_q[s], tag, v[s][0], v[s][1], p.status);
          SI_TRACE_LATEST(0, 14);
          if (g_dst[s] >= 0) {
            *reinterpret_cast<uint2 *>(smem + g_dst[s]) =
                make_uint2(static_cast<uint32_t>(v[s][0]), static_cast<uint32_t>(v[s][1]));
          } else {
            const uint32_t w = static_cast<uint32_t>(v[s][0]);
            ht.d[-g_dst[s] - 1] = half_bits_to_float(static_cast<uint16_t>(w & 0xFFFFu));
            ht.s[-g_dst[s] - 1] = half_bits_to_float(static_cast<uint16_t>(w >> 16));
          }
        }
      }
      if (__syncthreads_or(!ok)) goto fail;
      SI_TRACE_MARK(0, 6);
      bool okw = mbar_wait_bounded(&bars[6], par, p.status);
      if (kShared) okw &= mbar_wait_bounded(&bars[7], par, p.status);
#pragma unroll
      for (int s = 0; s < 2; ++s)
        if (okw && d_part[s] >= 0)
          part[d_part[s]] = q4k_half_dot(reinterpret_cast<const uint4 *>(smem + d_row[s]),
                                         reinterpret_cast<const uint4 *>(smem + d_act[s]), ht.d + d_blk[s],
                                         ht.s + d_blk[s], d_h[s]);
      if (__syncthreads_or(!okw)) goto fail;
      float ysum = 0.f;
      if (tlive) {
#pragma unroll 1
        for (int qq = 0; qq < tPP; ++qq) ysum += part[(tr * J + tj) * P_max + qq];
      }
      __syncthreads();
      if (tlive) part[tr * J + tj] = ysum;
      __syncthreads();
      if (warp == 0) {
        uint32_t tb = 0u;
        if (lane < nrows) {
          float acc = 0.f;
#pragma unroll 1
          for (int r = 0; r < k; ++r) acc = fmaf(s_wts[r], part[r * J + lane], acc);
          float tv = bf16_round(acc);
          if (kShared) tv = bf16_round(tv + bf16_round(sigma * part[k * J + lane]));
          tb = bf16_bits(tv);
        }
        // lane m < np3 writes rows 4m .. 4m + 3: one coalesced store
        const uint32_t r0 = __shfl_sync(0xffffffffu, tb, (4 * lane) & 31);
        const uint32_t r1 = __shfl_sync(0xffffffffu, tb, (4 * lane + 1) & 31);
        const uint32_t r2 = __shfl_sync(0xffffffffu, tb, (4 * lane + 2) & 31);
        const uint32_t r3 = __shfl_sync(0xffffffffu, tb, (4 * lane + 3) & 31);
        if (lane < p.np3)
          st_tag2(p.ol + (static_cast<size_t>(par) * G + c) * kSlot + 2 * lane, tagged(tag, r0 | (r1 << 16)),
                  tagged(tag, r2 | (r3 << 16)));
      }
    } else if (warp == 0 && lane < p.np3) {
      // no rows: the slot still says that this block is done with iteration it
      st_tag2(p.ol + (static_cast<size_t>(par) * G + c) * kSlot + 2 * lane, tagged(tag, 0u), tagged(tag, 0u));
    }
    SI_TRACE_MARK(0, 7);
    if (++l == p.n_layers) {
      l = 0;
      ++t;
    }
  }
  goto finish;
fail:
  if (threadIdx.x == kArmT)
#pragma unroll 1
    for (int b = 0; b < 8; ++b)
      if ((used >> b) & 1u) mbar_wait_bounded(&bars[b], ((armed >> b) & 1u) ^ 1u, p.status);
finish:
  // Tags of this launch are base + 1 .. base + n_iters; the next starts above.
  if (c == 0 && threadIdx.x == 0) *p.epoch = base + static_cast<uint32_t>(n_iters);
}

// ---------------------------------------------------------------------------
struct StackGeom {
  int G, J, np3, units;
  size_t off_epoch, off_layers, off_lg, off_hl, off_ol, bytes;
};

static int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

static StackGeom stack_geom(const si_moe_layer &L, int n_layers, int sms) {
  StackGeom g{};
  g.G = sms;
  g.J = sms > 0 ? (L.hidden + sms - 1) / sms : 0;
  g.J += g.J & 1;
  g.np3 = (g.J + 3) / 4;
  g.units = L.top_k * L.inter / 32 + L.shared_inter / 32;
  size_t off = sizeof(WsHeader);
  auto take = [&](size_t &field, size_t bytes) {
    field = off;
    off = round_up(off + bytes, 256);
  };
  take(g.off_epoch, 256);
  take(g.off_layers, sizeof(StackLayerPtrs) * n_layers);
  take(g.off_lg, 2 * 8u * kSlot * sms);
  take(g.off_hl, 2 * 8u * kSlot * g.units);
  take(g.off_ol, 2 * 8u * kSlot * sms);
  g.bytes = off;
  return g;
}

static StackSmem stack_smem(const si_moe_layer &L, int J, int n_layers) {
  StackSmem s{};
  const bool sh = L.shared_inter > 0;
  const int H = L.hidden, k = L.top_k, nsb = H / 256;
  const int nq = k * L.inter + L.shared_inter, n_slots = k + (sh ? 1 : 0);
  const int P_max = 2 * (L.inter > L.shared_inter ? L.inter : L.shared_inter) / 256;
  const int rb = H / 256 * kQ4KBytes, rbd = L.inter / 256 * kQ4KBytes,
            rbsd = sh ? L.shared_inter / 256 * kQ4KBytes : 0;
  size_t off = kStkFixedBytes;
  auto take = [&](uint32_t &field, size_t bytes, size_t align) {
    off = round_up(off, align);
    field = static_cast<uint32_t>(off);
    off += bytes;
  };
  take(s.layers, sizeof(StackLayerPtrs) * n_layers, 16);
  take(s.resid, 4u * H, 16);
  take(s.y, 4u * H, 16);
  take(s.tbuf, 4u * H, 16);
  take(s.part, 4u * n_slots * J * P_max, 16);
  take(s.xt_qs, static_cast<size_t>(nsb) * kActSbStride, 16);
  take(s.xt_d, 4u * nsb * 8, 16);
  take(s.xt_s, 4u * nsb * 8, 16);
  take(s.ht_qs, static_cast<size_t>(nq / 256) * kActSbStride, 16);
  take(s.ht_d, 4u * (nq / 32), 16);
  take(s.ht_s, 4u * (nq / 32), 16);
  s.pbuf_stride = static_cast<uint32_t>(round_up(8u * H, 128));
  take(s.pbuf, 2u * s.pbuf_stride, 128);
  take(s.gu, 64u * rb, 128);
  take(s.dn, static_cast<size_t>(J) * k * rbd, 128);
  take(s.sd, static_cast<size_t>(J) * rbsd, 128);
  s.bytes = static_cast<uint32_t>(off);
  return s;
}

// Whether the persistent kernel serves these layers: same shapes, Q4_K
// routed experts, Q4_K or no shared expert, bf16 router, and one resident
// block per SM covers every gate/up unit, down row and router row.
bool stack_supported(const si_moe_layer *layers, int n_layers) {
  const si_moe_layer &L = layers[0];
  for (int l = 0; l < n_layers; ++l) {
    const si_moe_layer &M = layers[l];
    if (M.hidden != L.hidden || M.n_experts != L.n_experts || M.top_k != L.top_k ||
        M.inter != L.inter || M.shared_inter != L.shared_inter || M.expert_type != SI_Q4_K ||
        down_type_of(M) != SI_Q4_K ||
        M.router_type != SI_BF16 || (M.shared_inter > 0 && M.shared_type != SI_Q4_K) ||
        M.eps != L.eps)
      return false;
  }
  if (L.hidden % 2048 != 0 || L.hidden > 4096 || L.n_experts > 256 || (L.n_experts & 1) ||
      L.inter % 256 || L.shared_inter % 256 || L.top_k > 8 || n_layers > 128)
    return false;
  const int sms = device_sms();
  if (sms <= 0) return false;
  const StackGeom g = stack_geom(L, n_layers, sms);
  const int n_slots = L.top_k + (L.shared_inter > 0 ? 1 : 0);
  const int P_max = 2 * (L.inter > L.shared_inter ? L.inter : L.shared_inter) / 256;
  if (sms < g.units || g.units * 5 > 2 * kStkThreads || g.J > 32 || sms * g.np3 > 2 * kStkThreads ||
      n_slots * g.J * P_max > 2 * kStkThreads || n_slots * g.J > kStkThreads)
    return false;
  if ((L.n_experts > 128 ? 2 * sms : sms) < L.n_experts) return false;
  if (sms > kStkThreads) return false;
  if (stack_smem(L, g.J, n_layers).bytes > 227 * 1024) return false;
  return true;
}

size_t stack_workspace_bytes(const si_moe_layer *layers, int n_layers) {
  return stack_geom(layers[0], n_layers, device_sms()).bytes;
}

cudaError_t preload_stack() {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, stack_kernel<0>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, stack_kernel<SI_Q4_K>);
  return e;
}

// Copies the per-layer pointer table into the workspace (synchronously, at
// set-up, outside any capture).
si_status stack_prepare(const si_moe_layer *layers, int n_layers, void *ws, cudaStream_t s) {
  const StackGeom g = stack_geom(layers[0], n_layers, device_sms());
  StackLayerPtrs *host = new StackLayerPtrs[n_layers];
  for (int l = 0; l < n_layers; ++l) {
    const si_moe_layer &L = layers[l];
    host[l] = StackLayerPtrs{static_cast<const __nv_bfloat16 *>(L.w_router),
                             static_cast<const __nv_bfloat16 *>(L.w_shared_sigmoid),
                             static_cast<const __nv_bfloat16 *>(L.w_norm),
                             static_cast<const uint8_t *>(L.w_gate),
                             static_cast<const uint8_t *>(L.w_up),
                             static_cast<const uint8_t *>(L.w_down),
                             static_cast<const uint8_t *>(L.ws_gate),
                             static_cast<const uint8_t *>(L.ws_up),
                             static_cast<const uint8_t *>(L.ws_down),
                             nullptr};
  }
  cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t *>(ws) + g.off_layers, host,
                                  sizeof(StackLayerPtrs) * n_layers, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  delete[] host;
  return cuda_status(e);
}

si_status stack_launch(const si_moe_layer *layers, int n_layers, int n_tokens, const void *x_in,
                       void *y_out, void *sum_out, int32_t *ids_out, void *ws, cudaStream_t s) {
  const si_moe_layer &L = layers[0];
  const int sms = device_sms();
  if (sms <= 0) return SI_ERR_CUDA;
  const StackGeom g = stack_geom(L, n_layers, sms);
  uint8_t *base = static_cast<uint8_t *>(ws);
  StackParams p{};
  p.layers = reinterpret_cast<const StackLayerPtrs *>(base + g.off_layers);
  p.n_layers = n_layers;
  p.n_tokens = n_tokens;
  p.H = L.hidden; p.E = L.n_experts; p.k = L.top_k; p.I = L.inter; p.Is = L.shared_inter;
  p.rb = L.hidden / 256 * kQ4KBytes;
  p.rbd = L.inter / 256 * kQ4KBytes;
  p.rbsd = L.shared_inter / 256 * kQ4KBytes;
  p.J = g.J;
  p.W = L.n_experts > 128 ? 4 : 8;      // as the router kernel's shape for these sizes
  p.nch = L.hidden / 8 / 32 / p.W;
  p.np3 = g.np3;
  p.eps = L.eps;
  p.sm = stack_smem(L, g.J, n_layers);
  p.x_in = static_cast<const __nv_bfloat16 *>(x_in);
  p.y_out = static_cast<__nv_bfloat16 *>(y_out);
  p.sum_out = static_cast<__nv_bfloat16 *>(sum_out);
  p.ids_out = ids_out;
  p.status = reinterpret_cast<uint32_t *>(base);
  p.epoch = reinterpret_cast<uint32_t *>(base + g.off_epoch);
  p.lg = reinterpret_cast<uint64_t *>(base + g.off_lg);
  p.hl = reinterpret_cast<uint64_t *>(base + g.off_hl);
  p.ol = reinterpret_cast<uint64_t *>(base + g.off_ol);
  const size_t smem = p.sm.bytes;
  if (smem > 227 * 1024) return SI_ERR_UNSUPPORTED;
  auto kern = L.shared_inter > 0 ? stack_kernel<SI_Q4_K> : stack_kernel<0>;
  cudaError_t e = allow_smem(kern, smem);
  if (e != cudaSuccess) return SI_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStkThreads, smem) != cudaSuccess ||
      per_sm < 1)
    return SI_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kStkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // every block resident: blocks wait on each other
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, p));
}

// Test only: one thread polls a pair that never carries the awaited tag.
__global__ void poll_timeout_kernel(const uint64_t *line, uint64_t budget_ns, uint32_t *status) {
  if (threadIdx.x == 0) {
    uint64_t a, b;
    ld_tag2(line, a, b);
    if (!pair_ok(a, b, 0xFFFFFFFFu)) poll_pair(line, 0xFFFFFFFFu, a, b, status, budget_ns);
  }
}

}  // namespace si

extern "C" si_status si_test_poll_timeout(uint64_t budget_ns, void *workspace, void *stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || budget_ns > 2000000000ull)
    return SI_ERR_INVALID_ARG;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  si::poll_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint64_t *>(ws + sizeof(si::WsHeader)), budget_ns,
      reinterpret_cast<uint32_t *>(ws));
  return si::cuda_status(cudaGetLastError());
}

#ifdef SI_TRACE
extern "C" int si_trace_dump_stack(void *dst) {
  return cudaMemcpyFromSymbol(dst, si::g_si_trace, sizeof(si::g_si_trace)) == cudaSuccess ? 0 : 4;
}
extern "C" int si_trace_reset_stack(void) {
  static uint64_t zeros[si::kTraceKernels * si::kTraceBlocks * si::kTracePhases];
  return cudaMemcpyToSymbol(si::g_si_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : 4;
}
#endif
