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
//   X2 h              - each gate/up unit writes its 32 Q8_1 codes + scales
//                       (quantised layers) or its 32 fp32 values (bf16
//                       layers); every block with down rows gathers them all;
//   X3 output rows    - each block writes bf16(routed + shared) of its rows;
//                       every block gathers all rows and folds the residual +
//                       RMSNorm of the next layer itself (Summary item 2 of
//                       the same page).
// A line element is 8 bytes, {payload word, tag}, written and read as single
// 64-bit accesses, so a reader that sees the tag of this iteration also sees
// its payload: one load both proves readiness and delivers the data (no
// counter, flag or fence round trip). Every writer owns whole 128-byte slots
// and fills its slot with one coalesced store (twice: each copy has half
// the readers): slots shared by several writers, polled by every block, made
// those writes wait behind the polls. Tags are epoch + iteration + 1, the
// epoch advancing by the iteration count at the end of every launch, so lines
// left by an earlier launch never match. Lines are double-buffered by
// iteration parity: a block writes buffer (i & 1) at iteration i only after it
// has gathered every block's X3 line of iteration i - 1, which each block
// writes after it has finished reading everything of iteration i - 2.
//
// Weights that do not depend on the routing are requested ahead, by warps
// that are idle at that moment: the next layer's router rows, shared-gate
// vector and norm weights and this layer's shared down rows while the logits
// are gathered; the next shared-expert gate/up unit (Q4_K, Q8_0) as soon as
// its buffer is free. Only the routed experts' bytes wait for the selection.
// Three layer kinds, one body (template arguments: routed and shared
// formats): Q4_K routed experts with a Q4_K, Q8_0 or no shared expert, whose
// 64-row gate/up unit fits shared memory whole, and bf16 layers, whose unit
// (256 KB) passes through a ring of bulk copies.
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
constexpr int kArmT = 480;          // the thread that arms the prefetch barriers (warp 15, lane 0)
// Every exchange slot is written kXRep times, and block b reads copy b % kXRep:
// a line polled by every block delays the store that the readers wait for
// (the polls queue ahead of it at the line's L2 slice), so each copy has only
// G / kXRep readers. The copies cost one warp-wide store instead of one.
constexpr int kXRep = 2;

// The 64 rows of a gate/up unit arrive in kGuGroups groups of 32 / kGuGroups
// gate rows and as many up rows, one bulk copy per matrix and group.
constexpr int kGuGroups = 4;
constexpr int kGuRows = 32 / kGuGroups;
// mbarriers of a stack block: 0, 1 the routing-independent prefetch (router
// rows, shared-gate vector, norm weights) by iteration parity; then one per
// gate/up group of the block's unit, and of its second unit (layers with
// more units than SMs); then the routed down rows; then the shared down rows.
enum {
  kBarPre = 0,
  kBarGu = 2,
  kBarGu2 = 2 + kGuGroups,
  kBarDn = 2 + 2 * kGuGroups,
  kBarSd = 3 + 2 * kGuGroups,
  kNumBars = 4 + 2 * kGuGroups
};

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
  int rb, rbs, rbd, rbsd;     // row bytes: routed / shared gate/up rows (H), routed / shared down rows
  int J;                      // down output rows per block (even)
  int np3;                    // X3: pairs of elements per block slot (ceil(J / 4))
  float eps;
  StackSmem sm;
  const __nv_bfloat16 *x_in;  // [T][H]
  __nv_bfloat16 *y_out, *sum_out;   // [T][H]
  int32_t *ids_out;           // [T][L][k] or null
  uint32_t *status;
  uint32_t *epoch;            // tag base
  uint64_t *lg;               // X1 [2][kXRep][G][kSlot]: {logit row c, logit row c + G}
  uint64_t *hl;               // X2 [2][kXRep][units][kSlot]: 8 code words, {d16 | s16 << 16}, pad
  uint64_t *ol;               // X3 [2][kXRep][G][kSlot]: bf16 pairs of this block's rows
};

// ---- tagged lines ----------------------------------------------------------
SI_DEV uint64_t tagged(uint32_t tag, uint32_t payload) {
  return (static_cast<uint64_t>(tag) << 32) | payload;
}
SI_DEV bool tag_ok(uint64_t v, uint32_t tag) { return static_cast<uint32_t>(v >> 32) == tag; }
SI_DEV void st_tag2(uint64_t *p, uint64_t a, uint64_t b) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
// Two elements (16-byte aligned); each 64-bit element is read atomically.
SI_DEV void ld_tag2(const uint64_t *p, uint64_t &a, uint64_t &b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p)
               : "memory");
}
SI_DEV bool pair_ok(uint64_t a, uint64_t b, uint32_t tag) { return tag_ok(a, tag) && tag_ok(b, tag); }

// Re-read the pair at p until both elements carry `tag`, for at most about
// budget_ns after an initial run of kSpinBeforeClock reads (no clock read on
// the fast path: it would stall the poller longer than a round trip);
// records SI_ERR_TIMEOUT and returns false if they never do.
SI_DEV bool poll_pair(const uint64_t *p, uint32_t tag, uint64_t &a, uint64_t &b, uint32_t *status,
                     uint64_t budget_ns = kWaitBudgetNs) {
#pragma unroll 1
  for (int i = 0; i < kSpinBeforeClock; ++i) {
    ld_tag2(p, a, b);
    if (pair_ok(a, b, tag)) return true;
  }
  const uint64_t t0 = now_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i) {
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
    float wv[8], yv[8];
    Load8<__nv_bfloat16>::run(w + i0, wv);
    Load8<float>::run(y + i0, yv);   // two 16-byte reads (no 8-way bank conflict)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(wv[i], yv[i], acc);
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

// The same sum with y as packed bf16 (identical values and order).
SI_DEV float sigma_dot_bf(const __nv_bfloat16 *w, const uint4 *y_bf, int n, float *red) {
  float acc = 0.f;
#pragma unroll 1
  for (int i0 = 8 * threadIdx.x; i0 < n; i0 += 8 * blockDim.x) {
    float wv[8], yv[8];
    Load8<__nv_bfloat16>::run(w + i0, wv);
    Load8<__nv_bfloat16>::run(y_bf + i0 / 8, yv);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(wv[i], yv[i], acc);
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
// bf16 gate/up units: 8 groups of 4 gate + 4 up rows through a ring of
// kBfRing slots of 8 rows.
constexpr int kBfGroups = 8;
constexpr int kBfRing = 4;
// after this many rounds of two groups the block requests its routed down
// rows into L2 (earlier they would take DRAM time from the gate/up rows it
// waits for)
constexpr int kBfDownAt = 2;
static_assert(kBfRing <= kGuGroups, "the ring's slots use the gate/up barriers");
// Issuing one bulk copy occupies the issuing thread for a few hundred cycles
// whatever its size, and many small copies ramp up more slowly than a few
// large ones, so copies are few and large and issued one per warp (lane 0)
// by warps that have nothing else to do at that moment. A barrier is armed
// (arrive + expected bytes) before any copy completing on it is issued; every
// arming flips the barrier's bit in `s_arm` (parity of the phases armed so
// far) and sets its "used" bit, so that an error exit can wait for the last
// armed phase of each barrier and leave no copy in flight.
SI_DEV void arm(uint64_t *bars, uint32_t *s_arm, int b, uint32_t bytes) {
  mbar_arrive_expect_tx(&bars[b], bytes);
  atomicXor(s_arm, 1u << b);
  atomicOr(s_arm, 1u << (16 + b));
}

// bf16 ring: group g (rows 4g .. 4g + 3 of the unit's gate and of its up
// matrix) into slot g % kBfRing, armed and requested by the calling thread.
SI_DEV void issue_bf16_group(const StackParams &p, const StackLayerPtrs &Lp, const uint64_t *s_sel, int unit,
                             int units_r, bool shared_unit, int g, uint8_t *ring, uint64_t *bars,
                             uint32_t *s_arm, uint64_t pol) {
  const int sl = g % kBfRing;
  const uint8_t *gsrc, *usrc;
  size_t row0;
  if (shared_unit) {
    row0 = static_cast<size_t>(unit - units_r) * 32;
    gsrc = Lp.wsg;
    usrc = Lp.wsu;
  } else {
    const int nhb = p.I / 32, slot = unit / nhb, hb = unit - slot * nhb;
    int e = key_index(s_sel[slot]);
    if (e < 0 || e >= p.E) e = 0;
    row0 = static_cast<size_t>(e) * p.I + static_cast<size_t>(hb) * 32;
    gsrc = Lp.wg;
    usrc = Lp.wu;
  }
  row0 += 4 * g;
  const uint32_t bytes = 4u * p.rb;
  arm(bars, s_arm, kBarGu + sl, 2 * bytes);
  bulk_g2s_evict_first(ring + static_cast<size_t>(sl) * 8 * p.rb, gsrc + row0 * p.rb, bytes, &bars[kBarGu + sl],
                       pol);
  bulk_g2s_evict_first(ring + (static_cast<size_t>(sl) * 8 + 4) * p.rb, usrc + row0 * p.rb, bytes,
                       &bars[kBarGu + sl], pol);
}

// Gather X3 (t = bf16(routed + shared) per row) into `tbuf` and fold it into
// the residual: s = bf16(t + resid) with the sum of squares in the norm
// kernel's order (the first 256 threads own rows 8i..8i+7 of every
// 2048-row slice); returns r = rsqrt(mean(s^2) + eps) in `r` (every thread).
// Thread i reads pairs i and i + 512 of the slots: f_src = element offset,
// f_row = first row, f_n = rows of this block in the pair (0 for a pair that
// only proves presence). `resid` holds the residual on entry and s on exit.
// Returns false (in every thread) if a slot did not arrive in time.
SI_DEV bool fold_sum(const StackParams &p, const uint64_t *ol, uint32_t tag, float *resid,
                     float *tbuf, float *red, const int f_src[2], const int f_row[2], const int f_n[2],
                     float &r) {
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
      const float4 c0 = *reinterpret_cast<const float4 *>(resid + r0);
      const float4 c1 = *reinterpret_cast<const float4 *>(resid + r0 + 4);
      const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
      const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      float sv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sv[e] = bf16_round(tv[e] + cv[e]);
        ss = fmaf(sv[e], sv[e], ss);
      }
      *reinterpret_cast<float4 *>(resid + r0) = make_float4(sv[0], sv[1], sv[2], sv[3]);
      *reinterpret_cast<float4 *>(resid + r0 + 4) = make_float4(sv[4], sv[5], sv[6], sv[7]);
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  }
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += red[i];
  r = rsqrtf(__fdiv_rn(tot, static_cast<float>(H)) + p.eps);
  return true;
}

// Phase timing of profiling builds (-DSI_TRACE). A %globaltimer read stalls
// its thread for about half a microsecond, so a launch stamps only two points
// of its last iteration (thread 0 of every block): the iteration start
// (phase 0) and the phase selected with si_trace_stack_phase; phase 14 sits
// right after phase 0 and measures the stall of a stamp itself. A profiling
// run takes many launches per phase.
#ifdef SI_TRACE
static __device__ int g_stk_trace_phase;
#define STK_TRACE_START()   \
  do {                      \
    STK_TRACE(0);           \
    STK_TRACE(14);          \
  } while (0)
#define STK_TRACE(ph)                                                                     \
  do {                                                                                    \
    if (threadIdx.x == 0 && it + 1 == n_iters && ((ph) == 0 || (ph) == tr_sel) && c < kTraceBlocks) \
      g_si_trace[0][c][(ph)] = now_ns();                                                  \
  } while (0)
#else
#define STK_TRACE_START() \
  do {                    \
  } while (0)
#define STK_TRACE(ph) \
  do {                \
  } while (0)
#endif

template <int EFMT, int SFMT, int DFMT = SI_Q4_K>
__global__ void __launch_bounds__(kStkThreads, 1) stack_kernel(StackParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr bool kShared = SFMT != 0;
  // bf16 experts (and shared expert): a unit of 64 rows of H bf16 is larger
  // than shared memory, so its rows pass through a ring of kBfRing slots of 8
  // rows (bulk copies, refilled as the groups are consumed); h travels as
  // fp32 (two slots per unit); a unit block's routed down rows go to L2 half
  // way through its gate/up rows and into the ring's space after them.
  constexpr bool kBf = EFMT == SI_BF16;
  constexpr int kSu = kBf ? 2 : 1;           // X2 slots per gate/up unit
  constexpr int kGq = kBf ? 5 : 2;           // X2 pairs gathered per thread
  // A Q8_0 shared expert: its gate/up unit (64 rows of H / 32 blocks of 34
  // bytes) is about twice a Q4_K unit, so in the block that owns it the
  // unit's buffer also holds the routed down rows, which arrive only after
  // the unit's dot products are done; the next unit is requested once the
  // down rows are consumed.
  constexpr bool kShQ80 = SFMT == SI_Q8_0;
  // routed down rows in Q5_K (the shipped format: 176-byte super-blocks,
  // the same half-super-block pieces)
  constexpr bool kDnQ5 = DFMT == SI_Q5_K;
  const int G = gridDim.x, c = blockIdx.x;
  const int H = p.H, I = p.I, Is = kShared ? p.Is : 0, k = p.k, E = p.E;
  const int nsb = H / kQKK;
  const int units_r = k * I / 32, units = units_r + Is / 32;
  const int nsb_r = I / kQKK, nsb_s = Is / kQKK;
  // down pieces of a row: Q4_K halves of 128 weights, Q8_0 whole 256-weight
  // groups (a Q8_0 half would start off a 16-byte boundary)
  const int P_r = 2 * nsb_r, P_s = kShared ? (kShQ80 ? nsb_s : 2 * nsb_s) : 1;
  // the pieces of a row take a power-of-two group of lanes (6 pieces: 8
  // lanes, two of them idle), so a group never straddles two warps
  const int P_rp = P_r <= 2 ? P_r : (P_r <= 4 ? 4 : (P_r <= 8 ? 8 : (P_r <= 16 ? 16 : 32)));
  const int P_sp = P_s <= 2 ? P_s : (P_s <= 4 ? 4 : (P_s <= 8 ? 8 : (P_s <= 16 ? 16 : 32)));
  const int P_max = P_rp > P_sp ? P_rp : P_sp;
  const int n_iters = p.n_tokens * p.n_layers;
  const int J = p.J;
  const int nvec = H / 2048;   // router: 16-byte vectors of a row per thread of the first 256

#ifdef SI_TRACE
  const int tr_sel = g_stk_trace_phase;
#endif
  // ---- shared memory --------------------------------------------------------
  static_assert(kNumBars <= 16, "barrier area holds 16 barriers");
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);     // kNumBars
  uint32_t *s_arm = reinterpret_cast<uint32_t *>(smem + 128);
  uint32_t *s_base = reinterpret_cast<uint32_t *>(smem + 132);
  float *red = reinterpret_cast<float *>(smem + 192);      // [16]
  float *s_part = reinterpret_cast<float *>(smem + 256);   // [2][8] router partials per warp
  float *s_wts = reinterpret_cast<float *>(smem + 320);    // [8]
  uint64_t *s_sel = reinterpret_cast<uint64_t *>(smem + 384);
  uint64_t *s_cand = reinterpret_cast<uint64_t *>(smem + 448);   // [64]
  float *h_s = reinterpret_cast<float *>(smem + 960);      // [2][32] h of the block's units
  float *s_gu = reinterpret_cast<float *>(smem + 1216);    // [64] bf16 gate/up row dots
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
  uint8_t *sd_buf = smem + p.sm.sd;   // [J] shared down rows
  // bf16 layers: y as packed bf16 and h as fp32 in place of the Q8_1 tiles
  uint4 *y_bf = reinterpret_cast<uint4 *>(smem + p.sm.xt_qs);   // [H / 8]
  float *hf = reinterpret_cast<float *>(smem + p.sm.ht_qs);      // [k I + Is]

  // ---- static assignment ----------------------------------------------------
  const int my_unit = c < units ? c : -1;
  const bool shared_unit = kShared && my_unit >= units_r;
  // more units than blocks (quantised layers without a shared expert only):
  // block c also takes unit c + G; its routed down rows then arrive, after
  // its gate/up dot products, in the space of its units' rows
  const int my_unit2 = (!kShared && !kBf && c + G < units) ? c + G : -1;
  const int dn_off = static_cast<int>(((kShQ80 && shared_unit) || my_unit2 >= 0) ? p.sm.gu : p.sm.dn);
  uint8_t *gu_buf2 = gu_buf + 64 * p.rb;   // the second unit's gate [32] + up [32] rows
  uint8_t *dn_buf = smem + dn_off;    // [k][J] routed down rows
  const int rb_unit = shared_unit ? p.rbs : p.rb;   // row bytes of this block's gate/up unit
  const int j0 = c * J;
  const int nrows = j0 < H ? min(J, H - j0) : 0;
  const int row_a = c, row_b = c + G;   // router rows of this block
  const int rep = c % kXRep;            // the copy of every exchange slot this block reads
  const int nrr = (row_a < E ? 1 : 0) + (row_b < E ? 1 : 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pr = threadIdx.x >> 4, gm = (threadIdx.x >> 3) & 1, lane8 = threadIdx.x & 7;   // gate/up
  const uint64_t pol = policy_evict_first();
  // X2 gather: pair q (5 per unit slot: 4 code pairs, 1 scale pair) ->
  // element offset g_q and shared memory destination g_dst (byte offset of 8
  // codes, or -(unit + 1) for the scales)
  // (bf16: pair q = unit q / 16, values 2 (q % 16), + 1 of its h, g_dst the
  // index of the first in hf)
  int g_q[kGq], g_dst[kGq];
#pragma unroll
  for (int s = 0; s < kGq; ++s) {
    const int q = static_cast<int>(threadIdx.x) + s * kStkThreads;
    if constexpr (kBf) {
      const int u = q / 16, m = q % 16;
      g_q[s] = q < units * 16 ? u * 2 * kSlot + 2 * m : -1;
      g_dst[s] = 32 * u + 2 * m;
    } else {
      const int u = q / 5, sub = q - 5 * (q / 5);
      g_q[s] = q < units * 5 ? u * kSlot + 2 * sub : -1;   // element offset of the pair
      const int base_sb = u < units_r ? (u / (I / 32)) * nsb_r : k * nsb_r;
      const int hb = u < units_r ? u % (I / 32) : u - units_r;
      g_dst[s] = sub < 4 ? static_cast<int>(p.sm.ht_qs) + (base_sb + hb / 8) * kActSbStride + (hb % 8) * 32 +
                               8 * sub
                         : -(u + 1);
    }
  }
  // down: item (slot r, row jl, half-super-block qq) of this thread in pass s;
  // the P pieces of a (slot, row) lie in consecutive lanes of one warp, the
  // first of them (qq == 0) sums them in order
  int d_row[2], d_act[2], d_blk[2], d_h[2], d_dst[2], d_P[2];
  bool d_live[2], d_first[2], d_q80[2], d_q5[2];
  const int items_r = k * J * P_rp;
  const int items = items_r + (kShared ? J * P_sp : 0);
  if constexpr (!kBf) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int u = static_cast<int>(threadIdx.x) + s * kStkThreads;
      int r, jl, qq;
      if (u < items_r) {
        r = u / (J * P_rp);
        const int rem = u - r * (J * P_rp);
        jl = rem / P_rp;
        qq = rem - jl * P_rp;
      } else {
        r = k;
        jl = (u - items_r) / P_sp;
        qq = (u - items_r) - jl * P_sp;
      }
      const bool sh = kShared && r == k;
      d_q80[s] = kShQ80 && sh;
      d_q5[s] = kDnQ5 && !sh;
      const int sb = d_q80[s] ? qq : qq >> 1;
      d_live[s] = u < items && jl < nrows && qq < (sh ? P_s : P_r);
      d_first[s] = qq == 0;
      d_P[s] = sh ? P_s : P_r;
      d_dst[s] = r * J + jl;
      d_row[s] = (sh ? static_cast<int>(p.sm.sd) + jl * p.rbsd : dn_off + (r * J + jl) * p.rbd) +
                 sb * (d_q80[s] ? 8 * kQ80Bytes : (d_q5[s] ? kQ5KBytes : kQ4KBytes));
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

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    *s_base = __ldcg(p.epoch);
    *s_arm = 0u;
  }
  {
    const unsigned long long *src = reinterpret_cast<const unsigned long long *>(p.layers);
    unsigned long long *dst = reinterpret_cast<unsigned long long *>(s_layers);
#pragma unroll 1
    for (int i = threadIdx.x; i < p.n_layers * 10; i += blockDim.x) dst[i] = __ldg(src + i);
  }
  __syncthreads();
  const uint32_t base = *s_base;

  int t = 0, l = 0;   // token and layer of iteration it
  const uint32_t gbytes = static_cast<uint32_t>((nrr + (kShared ? 1 : 0) + 1) * H * 2);
  const uint32_t cbytes = static_cast<uint32_t>(kGuRows) * p.rb;   // one copy: a group's gate (or up) rows
  const uint32_t cbytes_s = static_cast<uint32_t>(kGuRows) * p.rbs;   // the same of a shared unit
  if (threadIdx.x == kArmT && n_iters > 0) {
    // iteration 0's routing-independent bytes and shared gate/up unit
    const StackLayerPtrs &L0 = s_layers[0];
    arm(bars, s_arm, kBarPre, gbytes);
    if (nrr > 0) bulk_g2s(pbuf, L0.w_router + static_cast<size_t>(row_a) * H, H * 2, &bars[kBarPre]);
    if (nrr > 1) bulk_g2s(pbuf + 2 * H, L0.w_router + static_cast<size_t>(row_b) * H, H * 2, &bars[kBarPre]);
    if (kShared) bulk_g2s(pbuf + 4 * H, L0.w_sg, H * 2, &bars[kBarPre]);
    bulk_g2s(pbuf + 6 * H, L0.w_norm, H * 2, &bars[kBarPre]);
    if (!kBf && shared_unit) {
      const size_t row0 = static_cast<size_t>(my_unit - units_r) * 32;
#pragma unroll 1
      for (int g = 0; g < kGuGroups; ++g) {
        arm(bars, s_arm, kBarGu + g, 2 * cbytes_s);
        bulk_g2s_evict_first(gu_buf + kGuRows * g * p.rbs, L0.wsg + (row0 + kGuRows * g) * p.rbs, cbytes_s,
                             &bars[kBarGu + g], pol);
        bulk_g2s_evict_first(gu_buf + (32 + kGuRows * g) * p.rbs, L0.wsu + (row0 + kGuRows * g) * p.rbs,
                             cbytes_s, &bars[kBarGu + g], pol);
      }
    }
  }

  float r_norm = 0.f;   // rsqrt(mean(s^2) + eps) of the latest fold
  uint32_t bf_ph = 0u;  // bf16 ring: bit s = parity of slot s's next phase
  for (int it = 0;; ++it) {
    const uint32_t tag = base + static_cast<uint32_t>(it) + 1u, par = it & 1u;
    STK_TRACE_START();
    if (threadIdx.x == kArmT && it < n_iters) {   // copies issued during this iteration's logit gather
      if (it + 1 < n_iters) arm(bars, s_arm, kBarPre + (par ^ 1u), gbytes);
      if (kShared && nrows > 0) arm(bars, s_arm, kBarSd, static_cast<uint32_t>(nrows) * p.rbsd);
    }
    // [N] the fold of the previous iteration's outputs (at a token's first
    // layer, those are the previous token's results): resid := s, r_norm
    if (it > 0) {
      if (!fold_sum(p, p.ol + (static_cast<size_t>((it - 1) & 1) * kXRep + rep) * G * kSlot, tag - 1u, resid, tbuf, red,
                    f_src, f_row, f_n, r_norm))
        goto fail;
      if (l == 0) {   // token t - 1 is done: its last norm output and residual
        const __nv_bfloat16 *wn =
            reinterpret_cast<const __nv_bfloat16 *>(pbuf + ((it - 1) & 1) * pstr + 6 * H);
#pragma unroll 1
        for (int i = threadIdx.x; i < nrows; i += blockDim.x) {
          const float yv = bf16_round(__fmul_rn(__fmul_rn(resid[j0 + i], r_norm), __bfloat162float(wn[j0 + i])));
          p.y_out[static_cast<size_t>(t - 1) * H + j0 + i] = __float2bfloat16_rn(yv);
          if (p.sum_out)
            p.sum_out[static_cast<size_t>(t - 1) * H + j0 + i] = __float2bfloat16_rn(resid[j0 + i]);
        }
        __syncthreads();   // resid is overwritten below
      }
    }
#ifdef SI_TRACE
    if (it == n_iters && threadIdx.x == 0 && tr_sel == 13 && c < kTraceBlocks) g_si_trace[0][c][13] = now_ns();
#endif
    if (it == n_iters) break;
    STK_TRACE(1);

    // [R] y = this iteration's FFN input (x_in at a token's first layer, else
    // bf16(s * r * w_norm) with the previous layer's norm weights) and the
    // router rows' dot products in the same pass: thread i < 256 owns 16-byte
    // vectors i, i + 256, ... of a row (8 values each)
    {
      bool ok = true;
      if (threadIdx.x < 256) {
        ok = mbar_wait_bounded(&bars[kBarPre + par], (it >> 1) & 1, p.status);
        const uint8_t *pb = pbuf + par * pstr;
        const __nv_bfloat16 *wn =
            reinterpret_cast<const __nv_bfloat16 *>(pbuf + (par ^ 1u) * pstr + 6 * H);
        float acc_a = 0.f, acc_b = 0.f;
#pragma unroll 1
        for (int i = 0; i < nvec; ++i) {
          const int v = static_cast<int>(threadIdx.x) + 256 * i;
          float yv[8];
          if (l == 0) {
            Load8<__nv_bfloat16>::run(p.x_in + static_cast<size_t>(t) * H + 8 * v, yv);
            *reinterpret_cast<float4 *>(resid + 8 * v) = make_float4(yv[0], yv[1], yv[2], yv[3]);
            *reinterpret_cast<float4 *>(resid + 8 * v + 4) = make_float4(yv[4], yv[5], yv[6], yv[7]);
          } else {
            float wv[8];
            Load8<__nv_bfloat16>::run(wn + 8 * v, wv);
            const float4 s0 = *reinterpret_cast<const float4 *>(resid + 8 * v);
            const float4 s1 = *reinterpret_cast<const float4 *>(resid + 8 * v + 4);
            const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) yv[e] = bf16_round(__fmul_rn(__fmul_rn(sv[e], r_norm), wv[e]));
          }
          if constexpr (!kBf) {
            *reinterpret_cast<float4 *>(y + 8 * v) = make_float4(yv[0], yv[1], yv[2], yv[3]);
            *reinterpret_cast<float4 *>(y + 8 * v + 4) = make_float4(yv[4], yv[5], yv[6], yv[7]);
          } else
            y_bf[v] = make_uint4(bf16_bits(yv[0]) | (static_cast<uint32_t>(bf16_bits(yv[1])) << 16),
                                 bf16_bits(yv[2]) | (static_cast<uint32_t>(bf16_bits(yv[3])) << 16),
                                 bf16_bits(yv[4]) | (static_cast<uint32_t>(bf16_bits(yv[5])) << 16),
                                 bf16_bits(yv[6]) | (static_cast<uint32_t>(bf16_bits(yv[7])) << 16));
          if (ok && nrr > 0) {
            float wa[8];
            Load8<__nv_bfloat16>::run(pb + 16 * v, wa);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc_a = fmaf(wa[e], yv[e], acc_a);
            if (nrr > 1) {
              float wb[8];
              Load8<__nv_bfloat16>::run(pb + 2 * H + 16 * v, wb);
#pragma unroll
              for (int e = 0; e < 8; ++e) acc_b = fmaf(wb[e], yv[e], acc_b);
            }
          }
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
          acc_a += __shfl_xor_sync(0xffffffffu, acc_a, m);
          acc_b += __shfl_xor_sync(0xffffffffu, acc_b, m);
        }
        if (lane == 0) {
          s_part[warp] = acc_a;
          s_part[8 + warp] = acc_b;
        }
      }
      if (__syncthreads_or(!ok)) goto fail;
      if (warp == 0) {
        float lg[2] = {0.f, 0.f};
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
          if (rr < nrr) {
            lg[rr] = s_part[8 * rr];
#pragma unroll
            for (int w = 1; w < 8; ++w) lg[rr] += s_part[8 * rr + w];
          }
        // lane r < kXRep writes copy r
        if (lane < kXRep)
          st_tag2(p.lg + ((static_cast<size_t>(par) * kXRep + lane) * G + c) * kSlot,
                  tagged(tag, __float_as_uint(lg[0])), tagged(tag, __float_as_uint(lg[1])));
      }
    }
    STK_TRACE(2);
    // the gate/up activations, while the logits travel
    if constexpr (!kBf) quantize_y(y, H, xt);   // ends with __syncthreads
    STK_TRACE(3);

    // [S] warps 0..7 gather the logits of experts 32w .. 32w + 31 (expert e
    // is row e of block e, or row e - G of block e - G) and sort them; the
    // first 8 of every warp are the candidates. Meanwhile the other warps
    // request the next iteration's router rows, shared-gate vector and norm
    // weights and this iteration's shared down rows.
    {
      bool ok = true;
      if (warp < 8) {
        const int ex = 32 * warp + lane;
        uint64_t key = 0ull;   // below every real key
        if (ex < E) {
          const int slot = ex < G ? ex : ex - G;
          const uint64_t *q = p.lg + ((static_cast<size_t>(par) * kXRep + rep) * G + slot) * kSlot;
          uint64_t a, b;
          ld_tag2(q, a, b);
          ok = get_pair(q, tag, a, b, p.status);
          key = make_key(__uint_as_float(static_cast<uint32_t>(ex < G ? a : b)), ex);
        }
        key = warp_sort32(key, lane);
        if (lane < 8) s_cand[warp * 8 + lane] = key;
      } else if (lane == 0) {
        if (threadIdx.x == kArmT) {
          if (!kBf && my_unit >= 0 && !shared_unit)
#pragma unroll 1
            for (int g = 0; g < kGuGroups; ++g) arm(bars, s_arm, kBarGu + g, 2 * cbytes);
          if (my_unit2 >= 0)
#pragma unroll 1
            for (int g = 0; g < kGuGroups; ++g) arm(bars, s_arm, kBarGu2 + g, 2 * cbytes);
          if (nrows > 0) arm(bars, s_arm, kBarDn, static_cast<uint32_t>(k * nrows * p.rbd));
        }
        const StackLayerPtrs &Ln = s_layers[l + 1 == p.n_layers ? 0 : l + 1];
        uint8_t *dst = pbuf + (par ^ 1u) * pstr;
        uint64_t *bar = &bars[kBarPre + (par ^ 1u)];
        const bool next = it + 1 < n_iters;
        if (warp == 12 && next && nrr > 0)
          bulk_g2s(dst, Ln.w_router + static_cast<size_t>(row_a) * H, H * 2, bar);
        if (warp == 13 && next && nrr > 1)
          bulk_g2s(dst + 2 * H, Ln.w_router + static_cast<size_t>(row_b) * H, H * 2, bar);
        if (warp == 14 && next && kShared) bulk_g2s(dst + 4 * H, Ln.w_sg, H * 2, bar);
        if (warp == 15 && next) bulk_g2s(dst + 6 * H, Ln.w_norm, H * 2, bar);
        if (warp == 11 && kShared && nrows > 0)
          bulk_g2s_evict_first(sd_buf, s_layers[l].wsd + static_cast<size_t>(j0) * p.rbsd,
                               static_cast<uint32_t>(nrows) * p.rbsd, &bars[kBarSd], pol);
      }
      if (__syncthreads_or(!ok)) goto fail;
    }
    STK_TRACE(4);
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
    STK_TRACE(5);
    // routed bytes, one copy per warp: warps 0 .. 2 kGuGroups - 1 this block's
    // gate/up unit (warp w: group w % kGuGroups of the gate (w < kGuGroups) or
    // up rows), warps 8 .. 8 + k - 1
    // its down rows of each selected expert if it has no gate/up unit (a block
    // with a unit requests them once its gate/up rows have landed)
    if (lane == 0) {
      const StackLayerPtrs &Lp = s_layers[l];
      if (kBf && warp < kBfRing && my_unit >= 0)
        issue_bf16_group(p, Lp, s_sel, my_unit, units_r, shared_unit, warp, gu_buf, bars, s_arm, pol);
      if (!kBf && warp < 2 * kGuGroups && my_unit >= 0 && !shared_unit) {
        const int slot = my_unit / (I / 32), hb = my_unit - slot * (I / 32);
        int e = key_index(s_sel[slot]);
        if (e < 0 || e >= E) e = 0;
        const int g = warp % kGuGroups;
        const bool up = warp >= kGuGroups;
        const size_t row0 = static_cast<size_t>(e) * I + static_cast<size_t>(hb) * 32 + kGuRows * g;
        bulk_g2s_evict_first(gu_buf + ((up ? 32 : 0) + kGuRows * g) * p.rb, (up ? Lp.wu : Lp.wg) + row0 * p.rb,
                             cbytes, &bars[kBarGu + g], pol);
      }
      if (warp >= 8 && warp < 8 + 2 * kGuGroups && my_unit2 >= 0) {   // the second unit, warps 8..15
        const int slot = my_unit2 / (I / 32), hb = my_unit2 - slot * (I / 32);
        int e = key_index(s_sel[slot]);
        if (e < 0 || e >= E) e = 0;
        const int g = (warp - 8) % kGuGroups;
        const bool up = warp - 8 >= kGuGroups;
        const size_t row0 = static_cast<size_t>(e) * I + static_cast<size_t>(hb) * 32 + kGuRows * g;
        bulk_g2s_evict_first(gu_buf2 + ((up ? 32 : 0) + kGuRows * g) * p.rb, (up ? Lp.wu : Lp.wg) + row0 * p.rb,
                             cbytes, &bars[kBarGu2 + g], pol);
      }
      if (warp >= 8 && warp < 8 + k && nrows > 0 && (kBf || my_unit < 0)) {
        int e = key_index(s_sel[warp - 8]);
        if (e < 0 || e >= E) e = 0;
        const uint8_t *src = Lp.wd + (static_cast<size_t>(e) * H + j0) * p.rbd;
        if (my_unit < 0)   // (a bf16 unit block's ring holds its gate/up rows until [G] ends)
          bulk_g2s_evict_first(dn_buf + static_cast<size_t>(warp - 8) * J * p.rbd, src,
                               static_cast<uint32_t>(nrows) * p.rbd, &bars[kBarDn], pol);
      }
    }
    // while the routed bytes travel: softmax over the selected logits (rank
    // order) and the ids
    if (warp == 4) {
      const int r = lane < k ? lane : 0;
      const float ex = expf(key_value(s_sel[r]) - key_value(s_sel[0]));
      float sum = 0.f;
#pragma unroll 1
      for (int q = 0; q < k; ++q) sum += __shfl_sync(0xffffffffu, ex, q);
      if (lane < k) {
        s_wts[lane] = ex * __frcp_rn(sum);
        if (c == 0 && p.ids_out) {
          const int e = key_index(s_sel[lane]);
          p.ids_out[static_cast<size_t>(it) * k + lane] = (e < 0 || e >= E) ? 0 : e;
        }
      }
    }
    STK_TRACE(6);

    // [G] gate/up of this block's unit -> h line
    if constexpr (kBf) {
      if (my_unit >= 0) {
        // the unit's 8 groups of 4 gate + 4 up rows pass through the ring two
        // at a time: warps 0..7 take row w of group 2j, warps 8..15 row w - 8
        // of group 2j + 1, each row dotted by one warp in the four-kernel
        // path's lane order and reduction; after a round's barrier its two
        // slots are refilled with the groups 4 ahead; h is formed at the end
        bool ok = true;
        const int half = warp >> 3, wr = warp & 7;
#pragma unroll 1
        for (int j = 0; j < kBfGroups / 2; ++j) {
          const int g = 2 * j + half, sl = g % kBfRing;
          ok = mbar_wait_bounded(&bars[kBarGu + sl], (bf_ph >> sl) & 1u, p.status);
          bf_ph ^= 1u << sl;
          if (ok) {
            const uint4 *row = reinterpret_cast<const uint4 *>(gu_buf + (sl * 8 + wr) * p.rb);
            float acc = 0.f;
#pragma unroll 1
            for (int c0 = 0; c0 < H; c0 += 2048) {
              uint4 w[8];
#pragma unroll
              for (int cc = 0; cc < 8; ++cc) {
                const int k0 = c0 + (cc * 32 + lane) * 8;
                if (k0 < H) w[cc] = row[k0 / 8];
              }
              dot_row8(w, y_bf, c0, H, lane, acc);
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
            if (lane == 0) s_gu[8 * g + wr] = acc;
          }
          if (__syncthreads_or(!ok)) goto fail;
          if ((threadIdx.x == 256 || threadIdx.x == 288) && 2 * j + kBfRing < kBfGroups)
            issue_bf16_group(p, s_layers[l], s_sel, my_unit, units_r, shared_unit,
                             2 * j + kBfRing + (threadIdx.x == 288 ? 1 : 0), gu_buf, bars, s_arm, pol);
          if (j + 1 == kBfDownAt && lane == 4 && warp >= 8 && warp < 8 + k && nrows > 0) {
            int e = key_index(s_sel[warp - 8]);
            if (e < 0 || e >= E) e = 0;
            bulk_prefetch_l2(s_layers[l].wd + (static_cast<size_t>(e) * H + j0) * p.rbd,
                             static_cast<uint32_t>(nrows) * p.rbd);
          }
        }
        if (warp == 0) {   // pair q: gate row 8 (q / 4) + q % 4, up row + 4
          const int gi = 8 * (lane >> 2) + (lane & 3);
          const float ag = s_gu[gi], au = s_gu[gi + 4];
          h_s[lane] = __fdiv_rn(ag, 1.f + expf(-ag)) * au;
        }
        // the routed down rows (in L2 since the selection) into the ring's
        // space, which no copy of this iteration targets any more
        if (lane == 0 && warp >= 8 && warp < 8 + k && nrows > 0) {
          int e = key_index(s_sel[warp - 8]);
          if (e < 0 || e >= E) e = 0;
          bulk_g2s_evict_first(dn_buf + static_cast<size_t>(warp - 8) * J * p.rbd,
                               s_layers[l].wd + (static_cast<size_t>(e) * H + j0) * p.rbd,
                               static_cast<uint32_t>(nrows) * p.rbd, &bars[kBarDn], pol);
        }
        // the next layer's shared unit into L2 while DRAM is quiet (it does
        // not depend on the routing): lane 1 of warps 8..15, an eighth each
        if (shared_unit && it + 1 < n_iters && lane == 1 && warp >= 8) {
          const StackLayerPtrs &Ln = s_layers[l + 1 == p.n_layers ? 0 : l + 1];
          const int q = warp - 8;   // 0..3 gate rows, 4..7 up rows, 8 rows each
          const size_t row0 = static_cast<size_t>(my_unit - units_r) * 32 + 8 * (q & 3);
          bulk_prefetch_l2((q < 4 ? Ln.wsg : Ln.wsu) + row0 * p.rb, 8u * p.rb);
        }
        __syncwarp();
        STK_TRACE(7);
        if (warp == 0) {
          // item i = 16 r + m of copy r: values 2m, 2m + 1; lane L writes
          // items L, L + 32, ...
          const uint32_t hv = __float_as_uint(h_s[lane]);
#pragma unroll
          for (int i0 = 0; i0 < 16 * kXRep; i0 += 32) {
            const int i = i0 + lane, r = i / 16, m = i - 16 * r;
            const uint32_t wa2 = __shfl_sync(0xffffffffu, hv, (2 * m) & 31);
            const uint32_t wb2 = __shfl_sync(0xffffffffu, hv, (2 * m + 1) & 31);
            if (i < 16 * kXRep)
              st_tag2(p.hl + ((static_cast<size_t>(par) * kXRep + r) * units + my_unit) * kSu * kSlot + 2 * m,
                      tagged(tag, wa2), tagged(tag, wb2));
          }
        }
      }
    } else if (my_unit >= 0) {
      float acc = 0.f;
      const bool ok = mbar_wait_bounded(&bars[kBarGu + pr / kGuRows], par, p.status);
      if (ok) {
        const uint8_t *row = gu_buf + (gm * 32 + pr) * rb_unit;
        if (kShQ80 && shared_unit) {
          for (int sb = lane8; sb < nsb; sb += 8)
            acc += q80_sb_dot(reinterpret_cast<const uint4 *>(row + sb * 8 * kQ80Bytes),
                              reinterpret_cast<const uint4 *>(xt.qs + sb * kActSbStride), xt.d + 8 * sb);
        } else {
          for (int sb = lane8; sb < nsb; sb += 8)
            acc += q4k_sb_dot(reinterpret_cast<const uint4 *>(row + sb * kQ4KBytes),
                              reinterpret_cast<const uint4 *>(xt.qs + sb * kActSbStride), xt.d + 8 * sb,
                              xt.s + 8 * sb);
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      const float other = __shfl_xor_sync(0xffffffffu, acc, 8);
      if ((threadIdx.x & 15) == 0) h_s[pr] = __fdiv_rn(acc, 1.f + expf(-acc)) * other;
      bool ok2 = true;
      if (my_unit2 >= 0) {   // block-uniform: the second unit, the same rows of it
        float acc2 = 0.f;
        ok2 = mbar_wait_bounded(&bars[kBarGu2 + pr / kGuRows], par, p.status);
        if (ok2) {
          const uint8_t *row = gu_buf2 + (gm * 32 + pr) * p.rb;
          for (int sb = lane8; sb < nsb; sb += 8)
            acc2 += q4k_sb_dot(reinterpret_cast<const uint4 *>(row + sb * kQ4KBytes),
                               reinterpret_cast<const uint4 *>(xt.qs + sb * kActSbStride), xt.d + 8 * sb,
                               xt.s + 8 * sb);
        }
        acc2 += __shfl_xor_sync(0xffffffffu, acc2, 1);
        acc2 += __shfl_xor_sync(0xffffffffu, acc2, 2);
        acc2 += __shfl_xor_sync(0xffffffffu, acc2, 4);
        const float other2 = __shfl_xor_sync(0xffffffffu, acc2, 8);
        if ((threadIdx.x & 15) == 0) h_s[32 + pr] = __fdiv_rn(acc2, 1.f + expf(-acc2)) * other2;
      }
      if (__syncthreads_or(!(ok && ok2))) goto fail;
      STK_TRACE(7);
      // every wait on this iteration's gate/up phases is over
      if (lane == 0 && warp >= 8 && warp < 8 + k && nrows > 0) {
        // the down rows, now that this block's gate/up rows are in: they are
        // needed only after the h exchange
        const StackLayerPtrs &Lp = s_layers[l];
        int e = key_index(s_sel[warp - 8]);
        if (e < 0 || e >= E) e = 0;
        bulk_g2s_evict_first(dn_buf + static_cast<size_t>(warp - 8) * J * p.rbd,
                             Lp.wd + (static_cast<size_t>(e) * H + j0) * p.rbd,
                             static_cast<uint32_t>(nrows) * p.rbd, &bars[kBarDn], pol);
      }
      if (!kShQ80 && lane == 0 && warp >= 2 && warp < 2 + kGuGroups && shared_unit && it + 1 < n_iters) {
        // the next iteration's shared gate/up group warp - 2, armed and
        // requested by one thread
        const StackLayerPtrs &Ln = s_layers[l + 1 == p.n_layers ? 0 : l + 1];
        const int g = warp - 2;
        const size_t row0 = static_cast<size_t>(my_unit - units_r) * 32 + kGuRows * g;
        arm(bars, s_arm, kBarGu + g, 2 * cbytes_s);
        bulk_g2s_evict_first(gu_buf + kGuRows * g * p.rbs, Ln.wsg + row0 * p.rbs, cbytes_s, &bars[kBarGu + g],
                             pol);
        bulk_g2s_evict_first(gu_buf + (32 + kGuRows * g) * p.rbs, Ln.wsu + row0 * p.rbs, cbytes_s,
                             &bars[kBarGu + g], pol);
      }
      if (warp == 0 || (warp == 1 && my_unit2 >= 0)) {   // warp u: unit u's h
        const int un = warp == 0 ? my_unit : my_unit2;
        uint16_t d16, s16;
        const uint32_t q = static_cast<uint32_t>(q8_1_encode_warp(h_s[32 * warp + lane], d16, s16)) & 0xFFu;
        const uint32_t w = q | (__shfl_down_sync(0xffffffffu, q, 1) << 8) |
                           (__shfl_down_sync(0xffffffffu, q, 2) << 16) |
                           (__shfl_down_sync(0xffffffffu, q, 3) << 24);   // lane 4j: code word j
        // item i = 5 r + j of copy r: pair j < 4 = code words 2j, 2j + 1,
        // pair 4 = the scales; lane L writes items L, L + 32, ...
#pragma unroll
        for (int i0 = 0; i0 < 5 * kXRep; i0 += 32) {
          const int i = i0 + lane, r = i / 5, j = i - 5 * r;
          const uint32_t wa = __shfl_sync(0xffffffffu, w, (8 * j) & 31);
          const uint32_t wb = __shfl_sync(0xffffffffu, w, (8 * j + 4) & 31);
          uint64_t *line = p.hl + ((static_cast<size_t>(par) * kXRep + r) * units + un) * kSlot;
          if (i < 5 * kXRep) {
            if (j < 4)
              st_tag2(line + 2 * j, tagged(tag, wa), tagged(tag, wb));
            else
              st_tag2(line + 8, tagged(tag, static_cast<uint32_t>(d16) | (static_cast<uint32_t>(s16) << 16)),
                      tagged(tag, 0u));
          }
        }
      }
    }
    STK_TRACE(8);
    // the shared expert's gate sigma(w_sg . y), while the h lines travel
    float sigma = 0.f;
    if (kShared && nrows > 0) {
      const __nv_bfloat16 *wsg = reinterpret_cast<const __nv_bfloat16 *>(pbuf + par * pstr + 4 * H);
      const float z = kBf ? sigma_dot_bf(wsg, y_bf, H, red) : sigma_dot(wsg, y, H, red);
      sigma = __fdiv_rn(1.f, 1.f + expf(-z));
    }

    // [D] gather h, down for this block's rows -> X3 line. The first reads of
    // the h lines go out, then the down rows of this pass are taken apart
    // into registers (they usually land before the last h line), then the h
    // lines are polled.
    if (nrows > 0) {
      bool ok = true;
      const uint64_t *hl = p.hl + (static_cast<size_t>(par) * kXRep + rep) * units * kSu * kSlot;
      uint64_t v[kGq][2];
#pragma unroll
      for (int s = 0; s < kGq; ++s)
        if (g_q[s] >= 0) ld_tag2(hl + g_q[s], v[s][0], v[s][1]);
      bool okw = mbar_wait_bounded(&bars[kBarDn], par, p.status);
      if (kShared) okw &= mbar_wait_bounded(&bars[kBarSd], par, p.status);
      Q4KHalf wq;
      if constexpr (!kBf)
        if (okw && d_live[0] && !d_q80[0] && !d_q5[0])
          q4k_half_load(reinterpret_cast<const uint4 *>(smem + d_row[0]), d_h[0], wq);
#pragma unroll
      for (int s = 0; s < kGq; ++s) {
        if (g_q[s] < 0) continue;
        ok &= get_pair(hl + g_q[s], tag, v[s][0], v[s][1], p.status);
        if constexpr (kBf) {
          *reinterpret_cast<float2 *>(hf + g_dst[s]) =
              make_float2(__uint_as_float(static_cast<uint32_t>(v[s][0])),
                          __uint_as_float(static_cast<uint32_t>(v[s][1])));
        } else if (g_dst[s] >= 0) {
          *reinterpret_cast<uint2 *>(smem + g_dst[s]) =
              make_uint2(static_cast<uint32_t>(v[s][0]), static_cast<uint32_t>(v[s][1]));
        } else {
          const uint32_t w = static_cast<uint32_t>(v[s][0]);
          ht.d[-g_dst[s] - 1] = half_bits_to_float(static_cast<uint16_t>(w & 0xFFFFu));
          ht.s[-g_dst[s] - 1] = half_bits_to_float(static_cast<uint16_t>(w >> 16));
        }
      }
      if (__syncthreads_or(!(ok && okw))) goto fail;
      STK_TRACE(9);
      STK_TRACE(10);
      if constexpr (kBf) {
        // tasks (slot, row) of 8 lanes each, the four-kernel path's order:
        // lane l8 holds columns cc + 8 l8 + 64 i (i < 8) of each 512-wide
        // chunk, then the 8 lanes are summed
        const int sub = lane >> 3, l8 = lane & 7;
        const int ntask = (k + (kShared ? 1 : 0)) * J;
        // two tasks per 8 lanes at a time (tasks t and t + 64), their
        // products interleaved: two independent fma chains, each in the
        // order of its own task
#pragma unroll 1
        for (int t0 = 0; t0 < ntask; t0 += 8 * (kStkThreads / 32)) {
          int tr[2], tj[2], tw[2];
          bool live[2];
          const uint8_t *row[2];
          const float *hv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int task = t0 + 4 * (kStkThreads / 32) * u + 4 * warp + sub;
            tr[u] = task / J;
            tj[u] = task - tr[u] * J;
            live[u] = task < ntask && tj[u] < nrows;
            const bool sh = kShared && tr[u] == k;
            tw[u] = live[u] ? (sh ? Is : I) : 0;
            row[u] = sh ? sd_buf + static_cast<size_t>(tj[u]) * p.rbsd
                        : dn_buf + static_cast<size_t>(tr[u] * J + tj[u]) * p.rbd;
            hv[u] = hf + tr[u] * I;
          }
          float acc[2] = {0.f, 0.f};
          const int wmax = tw[0] > tw[1] ? tw[0] : tw[1];
#pragma unroll 1
          for (int cc = 0; cc < wmax; cc += 512) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int col = cc + l8 * 8 + 64 * i;
                if (col < tw[u]) {
                  // dot_down8's products and order; h read as two float4
                  float wv[8];
                  Load8<__nv_bfloat16>::run(row[u] + 2 * col, wv);
                  const float4 h0 = *reinterpret_cast<const float4 *>(hv[u] + col);
                  const float4 h1 = *reinterpret_cast<const float4 *>(hv[u] + col + 4);
                  const float hh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                  for (int q = 0; q < 8; ++q) acc[u] = fmaf(wv[q], hh[q], acc[u]);
                }
              }
            }
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            float v = acc[u];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            if (live[u] && l8 == 0) part[tr[u] * J + tj[u]] = v;
          }
        }
      } else {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (s * kStkThreads < items) {   // block-uniform
          float v = 0.f;
          if (d_live[s]) {
            const uint4 *a = reinterpret_cast<const uint4 *>(smem + d_act[s]);
            if (kShQ80 && d_q80[s])
              v = q80_sb_dot(reinterpret_cast<const uint4 *>(smem + d_row[s]), a, ht.d + d_blk[s]);
            else if (kDnQ5 && d_q5[s])
              v = q5k_half_dot(smem + d_row[s], a, ht.d + d_blk[s], ht.s + d_blk[s], d_h[s]);
            else
              v = s == 0 ? q4k_half_dot_loaded(wq, a, ht.d + d_blk[s], ht.s + d_blk[s], d_h[s])
                         : q4k_half_dot(reinterpret_cast<const uint4 *>(smem + d_row[s]), a, ht.d + d_blk[s],
                                        ht.s + d_blk[s], d_h[s]);
          }
          // the pieces of a (slot, row), summed in order by its first lane
          float ysum = 0.f;
          ysum += v;
#pragma unroll 1
          for (int q = 1; q < P_max; ++q) {
            const float o = __shfl_down_sync(0xffffffffu, v, q);
            if (q < d_P[s]) ysum += o;
          }
          if (d_live[s] && d_first[s]) part[d_dst[s]] = ysum;
        }
      }
      }
      __syncthreads();
      STK_TRACE(11);
      if (warp == 0) {
        uint32_t tb = 0u;
        if (lane < nrows) {
          // the 8 partial rows first, then the rank-order fma chain
          float pv[8], wv[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            pv[r] = r < k ? part[r * J + lane] : 0.f;
            wv[r] = r < k ? s_wts[r] : 0.f;
          }
          float acc = 0.f;
#pragma unroll
          for (int r = 0; r < 8; ++r)
            if (r < k) acc = fmaf(wv[r], pv[r], acc);
          float tv = bf16_round(acc);
          if (kShared) tv = bf16_round(tv + bf16_round(sigma * part[k * J + lane]));
          tb = bf16_bits(tv);
        }
        // item i = np3 r + m of copy r: rows 4m .. 4m + 3; lane L writes
        // items L, L + 32, ...
#pragma unroll 1
        for (int i0 = 0; i0 < p.np3 * kXRep; i0 += 32) {
          const int i = i0 + lane, r = i / p.np3, m = i - r * p.np3;
          const uint32_t r0 = __shfl_sync(0xffffffffu, tb, (4 * m) & 31);
          const uint32_t r1 = __shfl_sync(0xffffffffu, tb, (4 * m + 1) & 31);
          const uint32_t r2 = __shfl_sync(0xffffffffu, tb, (4 * m + 2) & 31);
          const uint32_t r3 = __shfl_sync(0xffffffffu, tb, (4 * m + 3) & 31);
          if (i < p.np3 * kXRep)
            st_tag2(p.ol + ((static_cast<size_t>(par) * kXRep + r) * G + c) * kSlot + 2 * m,
                    tagged(tag, r0 | (r1 << 16)), tagged(tag, r2 | (r3 << 16)));
        }
      }
    } else if (warp == 0) {
      // no rows: the slot still says that this block is done with iteration it
#pragma unroll 1
      for (int i = lane; i < p.np3 * kXRep; i += 32) {
        const int r = i / p.np3, m = i - r * p.np3;
        st_tag2(p.ol + ((static_cast<size_t>(par) * kXRep + r) * G + c) * kSlot + 2 * m, tagged(tag, 0u),
                tagged(tag, 0u));
      }
    }
    if (kShQ80 && lane == 0 && warp >= 2 && warp < 2 + kGuGroups && shared_unit && it + 1 < n_iters) {
      // the next iteration's shared gate/up group warp - 2: this block's
      // down rows, which share its buffer, have been consumed (the barrier
      // after the down dot products; a block without rows never used them)
      const StackLayerPtrs &Ln = s_layers[l + 1 == p.n_layers ? 0 : l + 1];
      const int g = warp - 2;
      const size_t row0 = static_cast<size_t>(my_unit - units_r) * 32 + kGuRows * g;
      arm(bars, s_arm, kBarGu + g, 2 * cbytes_s);
      bulk_g2s_evict_first(gu_buf + kGuRows * g * p.rbs, Ln.wsg + row0 * p.rbs, cbytes_s, &bars[kBarGu + g],
                           pol);
      bulk_g2s_evict_first(gu_buf + (32 + kGuRows * g) * p.rbs, Ln.wsu + row0 * p.rbs, cbytes_s,
                           &bars[kBarGu + g], pol);
    }
    STK_TRACE(12);
    if (++l == p.n_layers) {
      l = 0;
      ++t;
    }
  }
  goto finish;
fail:
  // every thread arrives here together (each jump follows a block-wide
  // vote); wait for the last armed phase of each barrier
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t a = *s_arm;
#pragma unroll 1
    for (int b = 0; b < kNumBars; ++b)
      if ((a >> (16 + b)) & 1u) mbar_wait_bounded(&bars[b], ((a >> b) & 1u) ^ 1u, p.status);
  }
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
  take(g.off_lg, 2 * 8u * kSlot * kXRep * sms);
  const size_t su = L.expert_type == SI_BF16 ? 2 : 1;   // X2 slots per unit
  take(g.off_hl, 2 * 8u * kSlot * kXRep * g.units * su);
  take(g.off_ol, 2 * 8u * kSlot * kXRep * sms);
  g.bytes = off;
  return g;
}

// Row bytes of a shared-expert matrix row of `width` weights.
static int shared_row_bytes(const si_moe_layer &L, int width) {
  return L.shared_type == SI_Q8_0 ? width / 32 * kQ80Bytes : width / 256 * kQ4KBytes;
}

// Pieces of one routed / shared down row (the down step's work items), and
// the power-of-two lane groups they take.
static int down_pieces_routed(const si_moe_layer &L) { return 2 * L.inter / 256; }
static int down_pieces_shared(const si_moe_layer &L) {
  return L.shared_type == SI_Q8_0 ? L.shared_inter / 256 : 2 * L.shared_inter / 256;
}
static int lane_group(int pieces) {
  int g = 1;
  while (g < pieces) g *= 2;
  return g;
}

// bf16 layers: no Q8_1 tiles; y as packed bf16 (in the place of the x
// tile), h as fp32 (in the place of the h tile); the gate/up ring and the
// routed down rows share one region.
static StackSmem stack_smem_bf16(const si_moe_layer &L, int J, int n_layers) {
  StackSmem s{};
  const bool sh = L.shared_inter > 0;
  const int H = L.hidden, k = L.top_k;
  const int nq = k * L.inter + L.shared_inter, n_slots = k + (sh ? 1 : 0);
  size_t off = kStkFixedBytes;
  auto take = [&](uint32_t &field, size_t bytes, size_t align) {
    off = round_up(off, align);
    field = static_cast<uint32_t>(off);
    off += bytes;
  };
  take(s.layers, sizeof(StackLayerPtrs) * n_layers, 16);
  take(s.resid, 4u * H, 16);
  take(s.tbuf, 4u * H, 16);
  s.y = s.tbuf;   // unused: y lives as packed bf16 only
  take(s.part, 4u * n_slots * J, 16);
  take(s.xt_qs, 2u * H, 16);
  s.xt_d = s.xt_s = s.xt_qs;
  take(s.ht_qs, 4u * nq, 16);
  s.ht_d = s.ht_s = s.ht_qs;
  s.pbuf_stride = static_cast<uint32_t>(round_up(8u * H, 128));
  take(s.pbuf, 2u * s.pbuf_stride, 128);
  // the gate/up ring (kBfRing slots of 8 rows of H) and, once the ring is
  // drained, the routed down rows: one region
  const size_t ring = static_cast<size_t>(kBfRing) * 8 * H * 2;
  const size_t down = static_cast<size_t>(J) * k * L.inter * 2;
  take(s.gu, ring > down ? ring : down, 128);
  s.dn = s.gu;
  take(s.sd, static_cast<size_t>(J) * L.shared_inter * 2, 128);
  s.bytes = static_cast<uint32_t>(off);
  return s;
}

static StackSmem stack_smem(const si_moe_layer &L, int J, int n_layers) {
  if (L.expert_type == SI_BF16) return stack_smem_bf16(L, J, n_layers);
  StackSmem s{};
  const bool sh = L.shared_inter > 0;
  const bool q80 = sh && L.shared_type == SI_Q8_0;
  const int H = L.hidden, k = L.top_k, nsb = H / 256;
  const int nq = k * L.inter + L.shared_inter, n_slots = k + (sh ? 1 : 0);
  const int P_r = lane_group(down_pieces_routed(L)), P_s = sh ? lane_group(down_pieces_shared(L)) : 0;
  const int P_max = P_r > P_s ? P_r : P_s;
  const int rb = H / 256 * kQ4KBytes, rbd = L.inter / 256 * (down_type_of(L) == SI_Q5_K ? kQ5KBytes : kQ4KBytes),
            rbsd = sh ? shared_row_bytes(L, L.shared_inter) : 0;
  const int sms = device_sms();
  const bool two_units = !sh && sms > 0 && k * L.inter / 32 > sms;
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
  if (q80) {
    // one region: a routed unit followed by the routed down rows, or the
    // shared unit (the routed down rows of its block overlap it)
    const size_t routed = 64u * rb + static_cast<size_t>(J) * k * rbd;
    const size_t shared = 64u * static_cast<size_t>(shared_row_bytes(L, H));
    take(s.gu, routed > shared ? routed : shared, 128);
    s.dn = s.gu + 64u * rb;
  } else if (two_units) {
    // one region: two units (a block with a second unit takes its routed
    // down rows into this space after its dot products), or one unit and
    // the routed down rows
    const size_t one = 64u * rb + static_cast<size_t>(J) * k * rbd, two = 128u * rb;
    take(s.gu, one > two ? one : two, 128);
    s.dn = s.gu + 64u * rb;
  } else {
    take(s.gu, 64u * rb, 128);
    take(s.dn, static_cast<size_t>(J) * k * rbd, 128);
  }
  take(s.sd, static_cast<size_t>(J) * rbsd, 128);
  s.bytes = static_cast<uint32_t>(off);
  return s;
}

// Whether the persistent kernel serves these layers: same shapes, Q4_K
// routed experts, a Q4_K, Q8_0 or no shared expert, bf16 router, and one
// resident block per SM covers every gate/up unit, down row and router row.
// bf16 layers: bf16 routed and shared experts and router, the same shapes,
// H a multiple of 2048 (<= 4096), I and Is multiples of 32, and every task of
// the down step (slot, row) and every h pair within the block's threads.
static bool stack_supported_bf16(const si_moe_layer *layers, int n_layers) {
  const si_moe_layer &L = layers[0];
  for (int l = 0; l < n_layers; ++l) {
    const si_moe_layer &M = layers[l];
    if (M.hidden != L.hidden || M.n_experts != L.n_experts || M.top_k != L.top_k ||
        M.inter != L.inter || M.shared_inter != L.shared_inter || M.expert_type != SI_BF16 ||
        down_type_of(M) != SI_BF16 || M.router_type != SI_BF16 ||
        (M.shared_inter > 0 && M.shared_type != SI_BF16) || M.eps != L.eps)
      return false;
  }
  if (L.hidden % 2048 != 0 || L.hidden > 4096 || L.n_experts > 256 || (L.n_experts & 1) ||
      L.inter % 32 || L.shared_inter % 32 || L.inter <= 0 || L.top_k > 8 || L.top_k < 1 || n_layers > 128)
    return false;
  const int sms = device_sms();
  if (sms <= 0 || sms > kStkThreads) return false;
  const StackGeom g = stack_geom(L, n_layers, sms);
  const int n_slots = L.top_k + (L.shared_inter > 0 ? 1 : 0);
  if (sms < g.units || g.units * 16 > 5 * kStkThreads || g.J > 32 || sms * g.np3 > 2 * kStkThreads ||
      n_slots * g.J > kStkThreads)
    return false;
  if ((L.n_experts > 128 ? 2 * sms : sms) < L.n_experts) return false;
  return stack_smem(L, g.J, n_layers).bytes <= 227 * 1024;
}

bool stack_supported(const si_moe_layer *layers, int n_layers) {
  const si_moe_layer &L = layers[0];
  if (L.expert_type == SI_BF16) return stack_supported_bf16(layers, n_layers);
  for (int l = 0; l < n_layers; ++l) {
    const si_moe_layer &M = layers[l];
    if (M.hidden != L.hidden || M.n_experts != L.n_experts || M.top_k != L.top_k ||
        M.inter != L.inter || M.shared_inter != L.shared_inter || M.expert_type != SI_Q4_K ||
        (down_type_of(M) != SI_Q4_K && down_type_of(M) != SI_Q5_K) || down_type_of(M) != down_type_of(L) ||
        M.router_type != SI_BF16 ||
        (M.shared_inter > 0 && M.shared_type != SI_Q4_K && M.shared_type != SI_Q8_0) ||
        (M.shared_inter > 0 && M.shared_type != L.shared_type) || M.eps != L.eps)
      return false;
  }
  if (L.hidden % 2048 != 0 || L.hidden > 4096 || L.n_experts > 256 || (L.n_experts & 1) ||
      L.inter % 256 || L.shared_inter % 256 || L.top_k > 8 || n_layers > 128)
    return false;
  const int sms = device_sms();
  if (sms <= 0) return false;
  const StackGeom g = stack_geom(L, n_layers, sms);
  const int n_slots = L.top_k + (L.shared_inter > 0 ? 1 : 0);
  const int P_r = lane_group(down_pieces_routed(L));
  const int P_s = L.shared_inter > 0 ? lane_group(down_pieces_shared(L)) : 0;
  const int P_max = P_r > P_s ? P_r : P_s;
  // a second gate/up unit per block only without a shared expert
  if ((L.shared_inter > 0 ? sms : 2 * sms) < g.units || g.units * 5 > 2 * kStkThreads || g.J > 32 || sms * g.np3 > 2 * kStkThreads ||
      n_slots * g.J * P_max > 2 * kStkThreads || n_slots * g.J > kStkThreads)
    return false;
  // the pieces of a (slot, row) of the down step are summed across a
  // power-of-two group of lanes of one warp: the groups must divide 32, and
  // the shared slot's groups must start on a multiple of their size
  if (32 % P_r || (L.shared_inter > 0 && (32 % P_s || (L.top_k * g.J * P_r) % P_s))) return false;
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
  cudaError_t e = cudaFuncGetAttributes(&a, stack_kernel<SI_Q4_K, 0>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, stack_kernel<SI_Q4_K, SI_Q4_K>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, stack_kernel<SI_Q4_K, SI_Q8_0>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, stack_kernel<SI_Q4_K, 0, SI_Q5_K>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, stack_kernel<SI_Q4_K, SI_Q4_K, SI_Q5_K>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, stack_kernel<SI_Q4_K, SI_Q8_0, SI_Q5_K>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, stack_kernel<SI_BF16, 0>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, stack_kernel<SI_BF16, SI_BF16>);
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
  const bool bf = L.expert_type == SI_BF16;
  p.rb = bf ? L.hidden * 2 : L.hidden / 256 * kQ4KBytes;
  p.rbs = L.shared_inter > 0 && !bf ? shared_row_bytes(L, L.hidden) : p.rb;
  const bool q5 = !bf && down_type_of(L) == SI_Q5_K;
  p.rbd = bf ? L.inter * 2 : L.inter / 256 * (q5 ? kQ5KBytes : kQ4KBytes);
  p.rbsd = L.shared_inter > 0 ? (bf ? L.shared_inter * 2 : shared_row_bytes(L, L.shared_inter)) : 0;
  p.J = g.J;
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
  auto kern = bf ? (L.shared_inter == 0 ? stack_kernel<SI_BF16, 0> : stack_kernel<SI_BF16, SI_BF16>)
              : q5 ? (L.shared_inter == 0      ? stack_kernel<SI_Q4_K, 0, SI_Q5_K>
                      : L.shared_type == SI_Q8_0 ? stack_kernel<SI_Q4_K, SI_Q8_0, SI_Q5_K>
                                                 : stack_kernel<SI_Q4_K, SI_Q4_K, SI_Q5_K>)
              : L.shared_inter == 0      ? stack_kernel<SI_Q4_K, 0>
              : L.shared_type == SI_Q8_0 ? stack_kernel<SI_Q4_K, SI_Q8_0>
                                         : stack_kernel<SI_Q4_K, SI_Q4_K>;
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
extern "C" int si_trace_stack_phase(int phase) {
  return cudaMemcpyToSymbol(si::g_stk_trace_phase, &phase, sizeof(phase)) == cudaSuccess ? 0 : 4;
}
extern "C" int si_trace_dump_stack(void *dst) {
  return cudaMemcpyFromSymbol(dst, si::g_si_trace, sizeof(si::g_si_trace)) == cudaSuccess ? 0 : 4;
}
extern "C" int si_trace_reset_stack(void) {
  static uint64_t zeros[si::kTraceKernels * si::kTraceBlocks * si::kTracePhases];
  return cudaMemcpyToSymbol(si::g_si_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : 4;
}
#endif
