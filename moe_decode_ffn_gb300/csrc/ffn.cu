// Routed experts + shared expert for one decode token.
//
// "perf(qwen3.6): fuse decode kernel launches - shared-expert + GDN
// conv/L2-norm" (sparkinfer PR #239), Summary item 1: gate and up GEMVs and
// the SwiGLU h = silu(g) * u in one pass over a staged input, the down GEMV
// separate. "Q4_K shared-expert FFN kernels + Q8_0/Q5_K->Q4_K requant of the
// MoE FFN stage" (sparkinfer PR #359), Summary: activations as Q8_1, Q4_K and
// Q8_0 weights dotted with int8 dp4a, h re-quantised to Q8_1 before down.
// "perf(qwen3.6): fused router GEMV+top-k + folded residual-norm (decode)"
// (sparkinfer PR #273), "Relation to open PRs": the shared expert's output is
// gated by sigmoid of a GEMV.
//
// GB300 design. The shared expert is treated as one more "slot" next to the k
// routed experts, so one gate/up launch and one down launch cover all of them.
//  * gate/up: one thread block per 32-row unit of h (one Q8_1 block of h):
//    the unit's 32 gate rows and 32 up rows arrive by 1-D TMA bulk copies
//    (cp.async.bulk) into shared memory in four mbarrier groups, so all of a
//    block's bytes are requested at once and compute on the first group
//    overlaps the arrival of the rest. One thread per (row, 256-weight
//    super-block); 8 lanes reduce a row; the block quantises its 32 h values
//    to Q8_1 itself. Shared-expert units depend only on x, so their copies
//    are issued before the kernel waits on the router.
//  * down: one thread block per tile of output rows, all slots; the weight
//    rows depend only on the expert ids (written by the router, two kernels
//    back), so they are requested before waiting on gate/up; only the h tile
//    (a few KB) is read after the wait. The rank-order combination and the
//    sigmoid gate are applied in the same block.
//  * bf16 weights (four times the bytes, no dequantisation): a warp per two
//    row pairs, x staged once as packed bf16; each gate/up unit also issues L2 bulk
//    prefetches for its share of its slot's down rows, so the down kernel
//    reads L2 while DRAM streams without a gap between the two launches.
#include "common.cuh"
#include "host.hpp"

namespace si {

enum SharedFmt { kNoShared = 0, kSharedQ4K = SI_Q4_K, kSharedQ80 = SI_Q8_0 };

SI_TRACE_BUFFER

constexpr int kGuThreads = 512;   // 32 row pairs x (2 matrices x 8 lanes)
constexpr int kDownThreads = 512;    // bf16 down
constexpr int kDownQThreads = 512;   // quantised down

struct GateUpParams {
  const __nv_bfloat16 *x;
  const uint8_t *x_q8;      // nullable: Q8_1 blocks of x
  const int32_t *ids;
  int H, E, k, I, Is;
  const uint8_t *wg, *wu;   // routed [E][I] rows
  const uint8_t *wsg, *wsu; // shared [Is] rows
  int rb_r, rb_s;           // gate/up row bytes, routed / shared
  int units_routed;         // k * I / 32
  const uint8_t *wd, *wsd;  // down rows (bf16 weights: staged into L2 by the gate/up units)
  int rbd_r, rbd_s;
  int8_t *hq;               // [k*I + Is] codes
  float *hd, *hs;           // [(k*I + Is)/32] block scale / sum (fp16 values)
  float *hf;                // [k*I + Is] h in fp32
  int e0, e1;               // routed experts computed: [e0, e1) (all of them: [0, E))
  uint32_t *status;
};

struct DownParams {
  const __nv_bfloat16 *x;
  const __nv_bfloat16 *w_sg;  // nullable when no shared expert
  const int32_t *ids;
  const float *wts;
  int H, E, k, I, Is, J;
  const uint8_t *wd, *wsd;    // routed [E][H] rows of I, shared [H] rows of Is
  int rbd_r, rbd_s;
  int down_q5;                // routed down rows are Q5_K (else Q4_K)
  const int8_t *hq;
  const float *hd, *hs, *hf;
  __nv_bfloat16 *routed, *shared;
  int e0, e1;                 // routed experts computed: [e0, e1)
  float *slot_y;              // nullable: [k][H] fp32 slot outputs instead of `routed`
  uint32_t *status;
};

// Expert id of routed slot r, validated (an out-of-range id is recorded and
// replaced by 0 so that no access leaves the weight arrays).
SI_DEV int load_expert(const int32_t *ids, int r, int E, uint32_t *status) {
  int e = __ldcg(ids + r);
  if (e < 0 || e >= E) {
    record_status(status, SI_ERR_INVALID_ARG);
    e = 0;
  }
  return e;
}

template <int SFMT>
SI_DEV float row_dot_q(const uint8_t *row, bool shared, int nsb, int lane8, const ActTile &a) {
  float acc = 0.f;
  for (int sb = lane8; sb < nsb; sb += 8) {
    const uint4 *av = reinterpret_cast<const uint4 *>(a.qs + sb * kActSbStride);
    if (SFMT == kSharedQ80 && shared)
      acc += q80_sb_dot(reinterpret_cast<const uint4 *>(row + sb * 272), av, a.d + 8 * sb);
    else
      acc += q4k_sb_dot(reinterpret_cast<const uint4 *>(row + sb * kQ4KBytes), av, a.d + 8 * sb,
                        a.s + 8 * sb);
  }
  return acc;
}

// ---------------------------------------------------------------------------
// gate/up + SiLU gating + Q8_1 of h, quantised weights.
// ---------------------------------------------------------------------------
template <int SFMT>
__global__ void __launch_bounds__(kGuThreads, 2) gateup_q_kernel(GateUpParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int nsb = p.H / kQKK;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);                 // 4 groups
  ActTile act;
  act.qs = smem + 64;
  act.d = reinterpret_cast<float *>(act.qs + nsb * kActSbStride);
  act.s = act.d + nsb * 8;
  float *h_s = act.s + nsb * 8;                                        // [32]
  const int rb_max = (SFMT == kNoShared) ? p.rb_r : max(p.rb_r, p.rb_s);
  uint8_t *wbuf = reinterpret_cast<uint8_t *>(h_s + 32);               // [2][32][rb_max]
  wbuf = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(wbuf) + 127) & ~uintptr_t(127));

  SI_TRACE_MARK(1, 0);
  const int unit = blockIdx.x;
  const bool shared = (SFMT != kNoShared) && unit >= p.units_routed;
  const int nhb_r = p.I / 32;
  const int slot = shared ? p.k : unit / nhb_r;
  const int hb = shared ? unit - p.units_routed : unit % nhb_r;
  const int rb = shared ? p.rb_s : p.rb_r;

  if (threadIdx.x == 0) {
    for (int g = 0; g < 4; ++g) mbar_init(&bars[g], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Gate rows of the unit go to wbuf, up rows to wbuf + 32 * rb_max, each at
  // the unit's own row stride rb; group g (rows 8g..8g+7 of both) completes
  // on bars[g].
  uint8_t *gate_buf = wbuf, *up_buf = wbuf + 32 * rb_max;
  auto issue = [&](const uint8_t *g_rows, const uint8_t *u_rows) {
    const uint64_t pol = policy_evict_first();
    const uint32_t bytes = 8u * rb;
    for (int g = 0; g < 4; ++g) {
      mbar_arrive_expect_tx(&bars[g], 2 * bytes);
      bulk_g2s_evict_first(gate_buf + 8 * g * rb, g_rows + static_cast<size_t>(8 * g) * rb, bytes,
                           &bars[g], pol);
      bulk_g2s_evict_first(up_buf + 8 * g * rb, u_rows + static_cast<size_t>(8 * g) * rb, bytes,
                           &bars[g], pol);
    }
  };
  if (shared && threadIdx.x == 0)
    issue(p.wsg + static_cast<size_t>(hb) * 32 * rb, p.wsu + static_cast<size_t>(hb) * 32 * rb);

  // x -> Q8_1 tile (x comes from work before the predecessor kernel).
  if (p.x_q8) tile_from_q8_1(p.x_q8, p.H, act);
  else quantize_to_tile<__nv_bfloat16>(p.x, p.H, act);
  SI_TRACE_MARK(1, 1);

  grid_dep_wait();
  grid_dep_launch();
  SI_TRACE_MARK(1, 2);

  __shared__ int s_owned;
  if (!shared && threadIdx.x == 0) {
    const int e = load_expert(p.ids, slot, p.E, p.status);
    s_owned = e >= p.e0 && e < p.e1;
    const size_t row0 = static_cast<size_t>(e) * p.I + static_cast<size_t>(hb) * 32;
    if (s_owned) issue(p.wg + row0 * rb, p.wu + row0 * rb);
  }
  if (!shared) {
    __syncthreads();
    if (!s_owned) return;   // an expert another partition computes: nothing requested, nothing to wait for
  }
  SI_TRACE_MARK(1, 3);

  const int pr = threadIdx.x >> 4, m = (threadIdx.x >> 3) & 1, lane8 = threadIdx.x & 7;
  const int grp = pr >> 3;
  float acc = 0.f;
  if (mbar_wait_bounded(&bars[grp], 0, p.status))
    acc = row_dot_q<SFMT>((m ? up_buf : gate_buf) + pr * rb, shared, nsb, lane8, act);
  SI_TRACE_MARK(1, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  const float other = __shfl_xor_sync(0xffffffffu, acc, 8);
  const int slot_off = slot * p.I;   // shared slot: k * I
  if ((threadIdx.x & 15) == 0) {
    const float g = acc, u = other;
    const float h = __fdiv_rn(g, 1.f + expf(-g)) * u;
    h_s[pr] = h;
    p.hf[slot_off + hb * 32 + pr] = h;
  }
  __syncthreads();
  SI_TRACE_MARK(1, 5);
  if (threadIdx.x < 32) {
    uint16_t d16, s16;
    const int q = q8_1_encode_warp(h_s[threadIdx.x], d16, s16);
    p.hq[slot_off + hb * 32 + threadIdx.x] = static_cast<int8_t>(q);
    if (threadIdx.x == 0) {
      const int bidx = (slot_off + hb * 32) / 32;
      p.hd[bidx] = half_bits_to_float(d16);
      p.hs[bidx] = half_bits_to_float(s16);
    }
  }
  SI_TRACE_MARK(1, 6);
}

// ---------------------------------------------------------------------------
// down + rank-order combination + sigmoid-gated shared output, quantised.
// ---------------------------------------------------------------------------
SI_DEV float block_dot_bf16(const __nv_bfloat16 *a, const __nv_bfloat16 *b, int n, float *red) {
  float acc = 0.f;
  for (int i0 = 8 * threadIdx.x; i0 < n; i0 += 8 * blockDim.x) {
    float va[8], vb[8];
    Load8<__nv_bfloat16>::run(a + i0, va);
    Load8<__nv_bfloat16>::run(b + i0, vb);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(va[i], vb[i], acc);
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  float tot = 0.f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) tot += red[i];
  return tot;
}

// Work items of one output row: Q4_K rows split into half super-blocks
// (128 weights), Q8_0 rows into whole 256-weight units (a Q8_0 half would
// start off a 16-byte boundary).
template <int SFMT>
SI_DEV int down_pieces(bool shared_slot, int width) {
  return (SFMT == kSharedQ80 && shared_slot) ? width / kQKK : 2 * (width / kQKK);
}

template <int SFMT>
__global__ void __launch_bounds__(kDownQThreads, 2) down_q_kernel(DownParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr bool kShared = SFMT != kNoShared;
  const int n_slots = p.k + (kShared ? 1 : 0);
  const int nsb_r = p.I / kQKK, nsb_s = kShared ? p.Is / kQKK : 0;
  const int P_r = down_pieces<SFMT>(false, p.I);
  const int P_s = kShared ? down_pieces<SFMT>(true, p.Is) : 1;   // 1: never divides (no shared items)
  const int P_max = max(P_r, P_s);
  const int nq = p.k * p.I + (kShared ? p.Is : 0);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
  float *wts = reinterpret_cast<float *>(smem + 16);           // [8]
  float *red = wts + 8;                                        // [16]
  float *part = red + 16;                                      // [n_slots][J][P_max]
  ActTile act;
  act.qs = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(part + n_slots * p.J * P_max) + 15) & ~uintptr_t(15));
  act.d = reinterpret_cast<float *>(act.qs + (p.k * nsb_r + nsb_s) * kActSbStride);
  act.s = act.d + nq / 32;
  uint8_t *wbuf = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(act.s + nq / 32) + 127) & ~uintptr_t(127));

  SI_TRACE_MARK(2, 0);
  const int j0 = blockIdx.x * p.J;
  const int nrows = min(p.J, p.H - j0);
  __shared__ int s_own[8];   // slot r's expert lies in [e0, e1)
  if (threadIdx.x == 0) {
    mbar_init(bar, n_slots);
    fence_mbar_init();
  }
  __syncthreads();
  // Expert ids and weights come from the router (two kernels back): one
  // thread per slot reads its id and requests that expert's rows at once
  // (a slot of an expert outside [e0, e1) only arrives).
  if (threadIdx.x < n_slots) {
    const uint64_t pol = policy_evict_first();
    const int r = threadIdx.x;
    if (r < p.k) {
      const int e = load_expert(p.ids, r, p.E, p.status);
      const bool own = e >= p.e0 && e < p.e1;
      s_own[r] = own;
      wts[r] = p.wts ? __ldcg(p.wts + r) : 0.f;
      const uint32_t br = own ? static_cast<uint32_t>(nrows) * p.rbd_r : 0u;
      mbar_arrive_expect_tx(bar, br);
      if (own)
        bulk_g2s_evict_first(wbuf + static_cast<size_t>(r) * p.J * p.rbd_r,
                             p.wd + (static_cast<size_t>(e) * p.H + j0) * p.rbd_r, br, bar, pol);
    } else {
      const uint32_t bs = static_cast<uint32_t>(nrows) * p.rbd_s;
      mbar_arrive_expect_tx(bar, bs);
      bulk_g2s_evict_first(wbuf + static_cast<size_t>(p.k) * p.J * p.rbd_r,
                           p.wsd + static_cast<size_t>(j0) * p.rbd_s, bs, bar, pol);
    }
  }
  SI_TRACE_MARK(2, 1);
  float sigma = 0.f;
  if (kShared) {
    const float z = block_dot_bf16(p.w_sg, p.x, p.H, red);
    sigma = __fdiv_rn(1.f, 1.f + expf(-z));
  }
  SI_TRACE_MARK(2, 2);

  grid_dep_wait();
  grid_dep_launch();
  SI_TRACE_MARK(2, 3);

  // h codes of every slot -> tile (super-blocks at the padded stride).
  for (int c = threadIdx.x; c < nq / 16; c += blockDim.x) {
    const int o = 16 * c;
    int base_sb, w;
    if (o < p.k * p.I) {
      base_sb = (o / p.I) * nsb_r;
      w = o % p.I;
    } else {
      base_sb = p.k * nsb_r;
      w = o - p.k * p.I;
    }
    *reinterpret_cast<uint4 *>(act.qs + (base_sb + w / kQKK) * kActSbStride + w % kQKK) =
        __ldcg(reinterpret_cast<const uint4 *>(p.hq + o));
  }
  for (int b = threadIdx.x; b < nq / 32; b += blockDim.x) {
    act.d[b] = __ldcg(p.hd + b);
    act.s[b] = __ldcg(p.hs + b);
  }
  __syncthreads();
  SI_TRACE_MARK(2, 4);
  mbar_wait_bounded(bar, 0, p.status);
  SI_TRACE_MARK(2, 5);

  const int items_r = p.k * p.J * P_r;
  const int items = items_r + (kShared ? p.J * P_s : 0);
  for (int u = threadIdx.x; u < items; u += blockDim.x) {
    int r, jl, q;
    if (u < items_r) {
      r = u / (p.J * P_r);
      const int rem = u % (p.J * P_r);
      jl = rem / P_r;
      q = rem % P_r;
    } else {
      r = p.k;
      jl = (u - items_r) / P_s;
      q = (u - items_r) % P_s;
    }
    if (jl >= nrows) continue;
    if (r < p.k && !s_own[r]) {   // computed by another partition
      part[(r * p.J + jl) * P_max + q] = 0.f;
      continue;
    }
    const bool sh = kShared && r == p.k;
    const uint8_t *row = wbuf + static_cast<size_t>(r) * p.J * p.rbd_r +
                         static_cast<size_t>(jl) * (sh ? p.rbd_s : p.rbd_r);
    const int sb0 = r * nsb_r;           // shared slot: k * nsb_r
    const int blk0 = (r * p.I) / 32;     // shared slot: k * I / 32
    float v;
    if (SFMT == kSharedQ80 && sh) {
      v = q80_sb_dot(reinterpret_cast<const uint4 *>(row + q * 272),
                     reinterpret_cast<const uint4 *>(act.qs + (sb0 + q) * kActSbStride),
                     act.d + blk0 + 8 * q);
    } else if (p.down_q5 && !sh) {
      const int sb = q >> 1;
      v = q5k_half_dot(row + sb * kQ5KBytes,
                       reinterpret_cast<const uint4 *>(act.qs + (sb0 + sb) * kActSbStride),
                       act.d + blk0 + 8 * sb, act.s + blk0 + 8 * sb, q & 1);
    } else {
      const int sb = q >> 1;
      v = q4k_half_dot(reinterpret_cast<const uint4 *>(row + sb * kQ4KBytes),
                       reinterpret_cast<const uint4 *>(act.qs + (sb0 + sb) * kActSbStride),
                       act.d + blk0 + 8 * sb, act.s + blk0 + 8 * sb, q & 1);
    }
    part[(r * p.J + jl) * P_max + q] = v;
  }
  __syncthreads();
  SI_TRACE_MARK(2, 6);
  // Combine in two short parallel phases: per (slot, row) the pieces in
  // order, then per row the slots in rank order, then the shared slot.
  float *ys = part;   // reuse: [n_slots][J] after the pieces are summed
  float ysum = 0.f;
  const int tr = threadIdx.x / p.J, tj = threadIdx.x % p.J;
  const bool tlive = threadIdx.x < n_slots * p.J && tj < nrows;
  if (tlive) {
    const int P = (kShared && tr == p.k) ? P_s : P_r;
    for (int q = 0; q < P; ++q) ysum += part[(tr * p.J + tj) * P_max + q];
  }
  __syncthreads();
  if (tlive) ys[tr * p.J + tj] = ysum;
  __syncthreads();
  if (threadIdx.x < nrows) {
    const int jl = threadIdx.x;
    if (p.slot_y) {
      // expert-parallel form: every slot's output (0 bits for the slots of
      // other partitions), combined after the partitions' outputs are summed
      for (int r = 0; r < p.k; ++r)
        p.slot_y[static_cast<size_t>(r) * p.H + j0 + jl] = s_own[r] ? ys[r * p.J + jl] : 0.f;
    } else {
      float acc = 0.f;
      for (int r = 0; r < p.k; ++r) acc = fmaf(wts[r], ys[r * p.J + jl], acc);
      p.routed[j0 + jl] = __float2bfloat16_rn(acc);
    }
    if (kShared) p.shared[j0 + jl] = __float2bfloat16_rn(sigma * ys[p.k * p.J + jl]);
  }
  SI_TRACE_MARK(2, 7);
}

// ---------------------------------------------------------------------------
// bf16 weights: fp32 activations, warp-level dot products.
// ---------------------------------------------------------------------------

// Gate/up, bf16: warp w owns row pairs 2w and 2w + 1 of the unit. Its rows
// are taken as a sequence of items (pair, 2048-wide chunk, gate or up) with
// two register buffers: the next item's eight 16-byte loads per lane are in
// flight while the current one is dotted.
__global__ void __launch_bounds__(kGuThreads, 1) gateup_bf16_kernel(GateUpParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint4 *xs = reinterpret_cast<uint4 *>(smem);   // [H / 8]
  const int unit = blockIdx.x;
  const bool shared = p.Is > 0 && unit >= p.units_routed;
  const int nhb_r = p.I / 32;
  const int slot = shared ? p.k : unit / nhb_r;
  const int hb = shared ? unit - p.units_routed : unit % nhb_r;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < p.H / 8; i += blockDim.x)   // x is final before the router ran
    xs[i] = __ldcg(reinterpret_cast<const uint4 *>(p.x) + i);
  __syncthreads();
  grid_dep_wait();
  grid_dep_launch();
  const __nv_bfloat16 *g_rows, *u_rows;
  const uint8_t *down;
  size_t rbd;
  if (shared) {
    g_rows = reinterpret_cast<const __nv_bfloat16 *>(p.wsg) + static_cast<size_t>(hb) * 32 * p.H;
    u_rows = reinterpret_cast<const __nv_bfloat16 *>(p.wsu) + static_cast<size_t>(hb) * 32 * p.H;
    down = p.wsd;
    rbd = static_cast<size_t>(p.rbd_s);
  } else {
    const int e = load_expert(p.ids, slot, p.E, p.status);
    const size_t row0 = static_cast<size_t>(e) * p.I + static_cast<size_t>(hb) * 32;
    g_rows = reinterpret_cast<const __nv_bfloat16 *>(p.wg) + row0 * p.H;
    u_rows = reinterpret_cast<const __nv_bfloat16 *>(p.wu) + row0 * p.H;
    down = p.wd ? p.wd + static_cast<size_t>(e) * p.H * p.rbd_r : nullptr;
    rbd = static_cast<size_t>(p.rbd_r);
  }
  const int per_pair = 2 * ((p.H + 2047) / 2048), n_items = 2 * per_pair;
  // item it: pair it / per_pair, chunk (it % per_pair) / 2, gate (even) or up (odd)
  auto item_row = [&](int it, int &c0) {
    const int q = it / per_pair, rem = it - q * per_pair;
    c0 = (rem >> 1) * 2048;
    return ((rem & 1) ? u_rows : g_rows) + static_cast<size_t>(2 * warp + q) * p.H;
  };
  uint4 wa[8], wb[8];
  int ca, cb;
  load_row8(item_row(0, ca), ca, p.H, lane, wa);
  float ag = 0.f, au = 0.f;
#pragma unroll 1
  for (int it = 0; it < n_items; it += 2) {
    load_row8(item_row(it + 1, cb), cb, p.H, lane, wb);
    if (it == 0 && lane == 0 && warp < 4 && down) {
      // this unit's share of its slot's down rows, staged into L2 for the
      // down kernel while the gate/up rows stream (same bytes, no gap between
      // the two kernels' reads): rows [hb * per, ...) in four pieces
      const int n_hb = shared ? p.Is / 32 : nhb_r;
      const int per = (p.H + n_hb - 1) / n_hb;
      const int r0 = min(p.H, hb * per), r1 = min(p.H, r0 + per);
      const int n4 = (r1 - r0 + 3) / 4;
      const int a = min(r1, r0 + warp * n4), b = min(r1, a + n4);
      if (b > a)
        bulk_prefetch_l2(down + static_cast<size_t>(a) * rbd, static_cast<uint32_t>((b - a) * rbd));
    }
    dot_row8(wa, xs, ca, p.H, lane, ag);
    if (it + 2 < n_items) load_row8(item_row(it + 2, ca), ca, p.H, lane, wa);
    dot_row8(wb, xs, cb, p.H, lane, au);
    if ((it + 2) % per_pair == 0) {   // pair complete
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) {
        ag += __shfl_xor_sync(0xffffffffu, ag, m);
        au += __shfl_xor_sync(0xffffffffu, au, m);
      }
      if (lane == 0)
        p.hf[slot * p.I + hb * 32 + 2 * warp + it / per_pair] = __fdiv_rn(ag, 1.f + expf(-ag)) * au;
      ag = 0.f;
      au = 0.f;
    }
  }
}

// Down task `task` of this block (slot r, local row jl): its weight row, or
// null past the block's rows. The ids are final before the gate/up kernel
// starts, so this may run before the wait on gate/up.
SI_DEV const __nv_bfloat16 *down_row(const DownParams &p, int task, int n_slots, int nrows, int j0,
                                     int &r, int &jl, int &width) {
  r = task / p.J;
  jl = task - r * p.J;
  width = 0;
  if (task >= n_slots * p.J || jl >= nrows) return nullptr;
  if (p.Is > 0 && r == p.k) {
    width = p.Is;
    return reinterpret_cast<const __nv_bfloat16 *>(p.wsd) + static_cast<size_t>(j0 + jl) * p.Is;
  }
  width = p.I;
  const int e = load_expert(p.ids, r, p.E, p.status);
  return reinterpret_cast<const __nv_bfloat16 *>(p.wd) + (static_cast<size_t>(e) * p.H + j0 + jl) * p.I;
}

// Whole-row dot of one task whose first chunk is already in `u0`, reduced
// over its 8 lanes.
SI_DEV float down_task_dot(const __nv_bfloat16 *row, const uint4 u0[8], const float *hv, int width,
                           int l8) {
  float acc = 0.f;
  if (row) {
    dot_down8(u0, hv, 0, width, l8, acc);
#pragma unroll 1
    for (int cc = 512; cc < width; cc += 512) {
      uint4 u[8];
      load_down8(row, cc, width, l8, u);
      dot_down8(u, hv, cc, width, l8, acc);
    }
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  return acc;
}

// Down, bf16: one block per tile of J output rows, tasks (slot, row) of 8
// lanes; the first round's rows are requested before the wait on gate/up
// (they depend only on the expert ids).
__global__ void __launch_bounds__(kDownThreads, 1) down_bf16_kernel(DownParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const bool has_shared = p.Is > 0;
  const int n_slots = p.k + (has_shared ? 1 : 0);
  const int nq = p.k * p.I + p.Is;
  float *wts = reinterpret_cast<float *>(smem);   // [8]
  float *red = wts + 8;                           // [kDownThreads / 32]
  float *y = red + kDownThreads / 32;             // [n_slots][J]
  float *hs = reinterpret_cast<float *>(            // [nq], 16-byte aligned
      (reinterpret_cast<uintptr_t>(y + n_slots * p.J) + 15) & ~uintptr_t(15));
  const int j0 = blockIdx.x * p.J;
  const int nrows = min(p.J, p.H - j0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane >> 3, l8 = lane & 7;   // 4 tasks per warp, 8 lanes each
  const int ntask = n_slots * p.J, step = 4 * (kDownThreads / 32);
  if (threadIdx.x < p.k) wts[threadIdx.x] = __ldcg(p.wts + threadIdx.x);
  int t0 = 4 * warp;
  int r, jl, wd;
  const __nv_bfloat16 *row = down_row(p, t0 + sub, n_slots, nrows, j0, r, jl, wd);
  uint4 u[8];
  load_down8(row, 0, wd, l8, u);
  float sigma = 0.f;
  if (has_shared) {
    const float z = block_dot_bf16(p.w_sg, p.x, p.H, red);
    sigma = __fdiv_rn(1.f, 1.f + expf(-z));
  }
  grid_dep_wait();
  grid_dep_launch();
  for (int i = threadIdx.x; i < nq / 4; i += blockDim.x)
    reinterpret_cast<float4 *>(hs)[i] = __ldcg(reinterpret_cast<const float4 *>(p.hf) + i);
  __syncthreads();
#pragma unroll 1
  for (;;) {
    const float acc = down_task_dot(row, u, hs + r * p.I, wd, l8);
    if (row && l8 == 0) y[r * p.J + jl] = acc;
    t0 += step;
    if (t0 >= ntask) break;
    row = down_row(p, t0 + sub, n_slots, nrows, j0, r, jl, wd);
    load_down8(row, 0, wd, l8, u);
  }
  __syncthreads();
  if (threadIdx.x < nrows) {
    const int jl = threadIdx.x;
    float acc = 0.f;
    for (int r = 0; r < p.k; ++r) acc = fmaf(wts[r], y[r * p.J + jl], acc);
    p.routed[j0 + jl] = __float2bfloat16_rn(acc);
    if (has_shared) p.shared[j0 + jl] = __float2bfloat16_rn(sigma * y[p.k * p.J + jl]);
  }
}

// ---------------------------------------------------------------------------
// Test export: exact per-(row, 32-block) integer dots of Q4_K x Q8_1.
// ---------------------------------------------------------------------------
__global__ void q4k_block_dots_kernel(const uint8_t *w, int rows, int k, const uint8_t *a,
                                      int32_t *out) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int nsb = k / kQKK;
  ActTile t;
  t.qs = smem;
  t.d = reinterpret_cast<float *>(smem + nsb * kActSbStride);
  t.s = t.d + nsb * 8;
  tile_from_q8_1(a, k, t);
  const int r = blockIdx.x;
  for (int sb = threadIdx.x; sb < nsb; sb += blockDim.x) {
    int isum[8];
    uint32_t dd, sw[3];
    q4k_isums(reinterpret_cast<const uint4 *>(w + (static_cast<size_t>(r) * nsb + sb) * kQ4KBytes),
              reinterpret_cast<const uint4 *>(t.qs + sb * kActSbStride), isum, dd, sw);
    for (int j = 0; j < 8; ++j) out[static_cast<size_t>(r) * (k / 32) + 8 * sb + j] = isum[j];
  }
}

// routed[j] = bf16(sum_r w[r] * y[r][j]): the fp32 fma chain over the slots
// in rank order, the down kernel's combine, on slot outputs gathered from
// expert partitions.
__global__ void __launch_bounds__(256) combine_slots_kernel(const float *y, const float *w, int k,
                                                            int H, __nv_bfloat16 *routed) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= H) return;
  float acc = 0.f;
  for (int r = 0; r < k; ++r) acc = fmaf(__ldg(w + r), __ldg(y + static_cast<size_t>(r) * H + j), acc);
  routed[j] = __float2bfloat16_rn(acc);
}

// Test export: exact per-(vector, row, 32-block) integer sums of the
// single-token helpers: whole Q4_K super-blocks (gate/up), Q4_K halves
// (routed and shared down) or Q5_K halves (the Q5_K routed down).
__global__ void block_dots_kernel(int kind, const uint8_t *w, int rows, int k, const uint8_t *a,
                                  int32_t *out) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int nsb = k / kQKK, nb = k / 32;
  ActTile t;
  t.qs = smem;
  t.d = reinterpret_cast<float *>(smem + nsb * kActSbStride);
  t.s = t.d + nb;
  tile_from_q8_1(a + static_cast<size_t>(blockIdx.y) * nb * kQ81Bytes, k, t);
  const int r = blockIdx.x;
  const int sbb = kind == SI_TEST_DOTS_Q5K_HALF ? kQ5KBytes : kQ4KBytes;
  int32_t *o = out + (static_cast<size_t>(blockIdx.y) * rows + r) * nb;
  for (int sb = threadIdx.x; sb < nsb; sb += blockDim.x) {
    const uint8_t *wb = w + (static_cast<size_t>(r) * nsb + sb) * sbb;
    const uint4 *av = reinterpret_cast<const uint4 *>(t.qs + sb * kActSbStride);
    if (kind == SI_TEST_DOTS_Q4K_SB) {
      int isum[8];
      uint32_t dd, sw[3];
      q4k_isums(reinterpret_cast<const uint4 *>(wb), av, isum, dd, sw);
      for (int j = 0; j < 8; ++j) o[8 * sb + j] = isum[j];
    } else {
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        int isum[4];
        if (kind == SI_TEST_DOTS_Q4K_HALF)
          q4k_half_isums(reinterpret_cast<const uint4 *>(wb), av, h, isum);
        else
          q5k_half_isums(wb, av, h, isum);
        for (int j = 0; j < 4; ++j) o[8 * sb + 4 * h + j] = isum[j];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int row_bytes_of(si_dtype t, int k) {
  switch (t) {
    case SI_Q4_K: return k / 256 * kQ4KBytes;
    case SI_Q5_K: return k / 256 * kQ5KBytes;
    case SI_Q8_0: return k / 32 * kQ80Bytes;
    case SI_BF16: return 2 * k;
    default: return 0;
  }
}

FfnGeom ffn_geom(const si_moe_layer &L) {
  FfnGeom g{};
  const bool sh = L.shared_inter > 0;
  g.n_slots = L.top_k + (sh ? 1 : 0);
  g.n_units = L.top_k * L.inter / 32 + (sh ? L.shared_inter / 32 : 0);
  const size_t nq = static_cast<size_t>(L.top_k) * L.inter + (sh ? L.shared_inter : 0);
  size_t off = sizeof(WsHeader);
  g.off_hq = off;
  off = round_up(off + nq, 256);
  g.off_hd = off;
  off = round_up(off + nq / 32 * sizeof(float), 256);
  g.off_hs = off;
  off = round_up(off + nq / 32 * sizeof(float), 256);
  g.off_hf = off;
  off = round_up(off + nq * sizeof(float), 256);
  g.bytes = off;
  return g;
}

si_status ffn_check(const si_moe_layer &L) {
  const bool sh = L.shared_inter > 0;
  if (L.hidden < 256 || L.hidden % 256 || L.hidden > 16384) return SI_ERR_INVALID_ARG;
  if (L.n_experts < 1 || L.n_experts > 256 || L.top_k < 1 || L.top_k > 8 || L.top_k > L.n_experts)
    return SI_ERR_INVALID_ARG;
  if (L.inter < 256 || L.inter % 256 || L.inter > 4096) return SI_ERR_INVALID_ARG;
  if (L.shared_inter < 0 || (sh && (L.shared_inter % 256 || L.shared_inter > 4096)))
    return SI_ERR_INVALID_ARG;
  if (!L.w_gate || !L.w_up || !L.w_down) return SI_ERR_INVALID_ARG;
  if (!aligned16(L.w_gate) || !aligned16(L.w_up) || !aligned16(L.w_down)) return SI_ERR_INVALID_ARG;
  if (sh) {
    if (!L.ws_gate || !L.ws_up || !L.ws_down || !L.w_shared_sigmoid) return SI_ERR_INVALID_ARG;
    if (!aligned16(L.ws_gate) || !aligned16(L.ws_up) || !aligned16(L.ws_down) ||
        !aligned16(L.w_shared_sigmoid))
      return SI_ERR_INVALID_ARG;
  }
  if (L.expert_type == SI_Q4_K) {
    if (sh && L.shared_type != SI_Q4_K && L.shared_type != SI_Q8_0) return SI_ERR_UNSUPPORTED;
    if (down_type_of(L) != SI_Q4_K && down_type_of(L) != SI_Q5_K) return SI_ERR_UNSUPPORTED;
    // the gate/up shared-memory buffer holds 64 rows of the widest format
    const int rb = sh ? max(row_bytes_of(SI_Q4_K, L.hidden), row_bytes_of(L.shared_type, L.hidden))
                      : row_bytes_of(SI_Q4_K, L.hidden);
    if (64u * rb + 4096u + L.hidden / 256 * 400u > 227u * 1024u) return SI_ERR_UNSUPPORTED;
  } else if (L.expert_type == SI_BF16) {
    if (sh && L.shared_type != SI_BF16) return SI_ERR_UNSUPPORTED;
    if (down_type_of(L) != SI_BF16) return SI_ERR_UNSUPPORTED;
  } else {
    return SI_ERR_UNSUPPORTED;
  }
  return SI_OK;
}

static size_t gateup_q_smem(const si_moe_layer &L, int rb_max) {
  const int nsb = L.hidden / 256;
  size_t off = 64 + nsb * kActSbStride + 2 * nsb * 8 * sizeof(float) + 32 * sizeof(float);
  off = round_up(off, 128);
  return off + 64u * rb_max + 128;
}

static size_t down_q_smem(const si_moe_layer &L, int J, int rbd_r, int rbd_s) {
  const bool sh = L.shared_inter > 0;
  const int n_slots = L.top_k + (sh ? 1 : 0);
  const int nq = L.top_k * L.inter + (sh ? L.shared_inter : 0);
  const int p_max = 2 * max(L.inter, sh ? L.shared_inter : 0) / 256;
  size_t off = 16 + 24 * sizeof(float) + static_cast<size_t>(n_slots) * J * p_max * sizeof(float);
  off = round_up(off, 16) + (nq / 256) * kActSbStride + 2 * (nq / 32) * sizeof(float);
  off = round_up(off, 128);
  return off + static_cast<size_t>(J) * (L.top_k * rbd_r + (sh ? rbd_s : 0)) + 128;
}

template <int SFMT>
static cudaError_t launch_q(const GateUpParams &gp, const DownParams &dp, size_t gsm, size_t dsm,
                            int down_ctas, int units, cudaStream_t s, bool gateup_only) {
  cudaError_t e = allow_smem(gateup_q_kernel<SFMT>, gsm);
  if (e != cudaSuccess) return e;
  e = allow_smem(down_q_kernel<SFMT>, dsm);
  if (e != cudaSuccess) return e;
  e = launch_pdl(gateup_q_kernel<SFMT>, dim3(units), dim3(kGuThreads), gsm, s, gp);
  if (e != cudaSuccess || gateup_only) return e;
  return launch_pdl(down_q_kernel<SFMT>, dim3(down_ctas), dim3(kDownQThreads), dsm, s, dp);
}

cudaError_t preload_ffn() {
  cudaFuncAttributes a;
  const void *ks[] = {
      reinterpret_cast<const void *>(gateup_q_kernel<kNoShared>),
      reinterpret_cast<const void *>(gateup_q_kernel<kSharedQ4K>),
      reinterpret_cast<const void *>(gateup_q_kernel<kSharedQ80>),
      reinterpret_cast<const void *>(down_q_kernel<kNoShared>),
      reinterpret_cast<const void *>(down_q_kernel<kSharedQ4K>),
      reinterpret_cast<const void *>(down_q_kernel<kSharedQ80>),
      reinterpret_cast<const void *>(gateup_bf16_kernel),
      reinterpret_cast<const void *>(down_bf16_kernel),
      reinterpret_cast<const void *>(q4k_block_dots_kernel)};
  for (const void *k : ks) {
    const cudaError_t e = cudaFuncGetAttributes(&a, k);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

si_status ffn_launch(const si_moe_layer &L, const void *x, const void *x_q8_1, const int32_t *ids,
                     const float *wts, void *routed, void *shared, void *ws, uint32_t *status,
                     cudaStream_t s, bool gateup_only, int e0, int e1, float *slot_y) {
  const FfnGeom g = ffn_geom(L);
  const bool sh = L.shared_inter > 0;
  uint8_t *base = static_cast<uint8_t *>(ws);
  GateUpParams gp{};
  gp.x = static_cast<const __nv_bfloat16 *>(x);
  gp.x_q8 = static_cast<const uint8_t *>(x_q8_1);
  gp.ids = ids;
  gp.H = L.hidden; gp.E = L.n_experts; gp.k = L.top_k; gp.I = L.inter;
  gp.Is = sh ? L.shared_inter : 0;
  gp.wg = static_cast<const uint8_t *>(L.w_gate);
  gp.wu = static_cast<const uint8_t *>(L.w_up);
  gp.wsg = static_cast<const uint8_t *>(L.ws_gate);
  gp.wsu = static_cast<const uint8_t *>(L.ws_up);
  gp.rb_r = row_bytes_of(L.expert_type, L.hidden);
  gp.rb_s = sh ? row_bytes_of(L.shared_type, L.hidden) : 0;
  gp.units_routed = L.top_k * L.inter / 32;
  gp.hq = reinterpret_cast<int8_t *>(base + g.off_hq);
  gp.hd = reinterpret_cast<float *>(base + g.off_hd);
  gp.hs = reinterpret_cast<float *>(base + g.off_hs);
  gp.hf = reinterpret_cast<float *>(base + g.off_hf);
  gp.e0 = e0;
  gp.e1 = e1 < 0 ? L.n_experts : e1;
  gp.status = status;

  const int sms = sm_count();
  DownParams dp{};
  dp.x = gp.x;
  dp.w_sg = static_cast<const __nv_bfloat16 *>(L.w_shared_sigmoid);
  dp.ids = ids; dp.wts = wts;
  dp.H = L.hidden; dp.E = L.n_experts; dp.k = L.top_k; dp.I = L.inter; dp.Is = gp.Is;
  dp.J = (L.hidden + sms - 1) / sms;
  dp.wd = static_cast<const uint8_t *>(L.w_down);
  dp.wsd = static_cast<const uint8_t *>(L.ws_down);
  dp.rbd_r = row_bytes_of(down_type_of(L), L.inter);
  dp.down_q5 = down_type_of(L) == SI_Q5_K ? 1 : 0;
  dp.rbd_s = sh ? row_bytes_of(L.shared_type, L.shared_inter) : 0;
  dp.hq = gp.hq; dp.hd = gp.hd; dp.hs = gp.hs; dp.hf = gp.hf;
  dp.routed = static_cast<__nv_bfloat16 *>(routed);
  dp.shared = static_cast<__nv_bfloat16 *>(shared);
  dp.e0 = gp.e0;
  dp.e1 = gp.e1;
  dp.slot_y = slot_y;
  dp.status = gp.status;
  const int down_ctas = (L.hidden + dp.J - 1) / dp.J;
  if (L.expert_type == SI_BF16 && !gateup_only) {
    gp.wd = dp.wd;
    gp.wsd = dp.wsd;
    gp.rbd_r = dp.rbd_r;
    gp.rbd_s = dp.rbd_s;
  }

  cudaError_t e;
  if (L.expert_type == SI_Q4_K) {
    const int rb_max = sh ? max(gp.rb_r, gp.rb_s) : gp.rb_r;
    const size_t gsm = gateup_q_smem(L, rb_max);
    const size_t dsm = down_q_smem(L, dp.J, dp.rbd_r, dp.rbd_s);
    if (!sh) e = launch_q<kNoShared>(gp, dp, gsm, dsm, down_ctas, g.n_units, s, gateup_only);
    else if (L.shared_type == SI_Q4_K)
      e = launch_q<kSharedQ4K>(gp, dp, gsm, dsm, down_ctas, g.n_units, s, gateup_only);
    else e = launch_q<kSharedQ80>(gp, dp, gsm, dsm, down_ctas, g.n_units, s, gateup_only);
  } else {
    const size_t gsm = static_cast<size_t>(L.hidden) * 2;
    const int nq = L.top_k * L.inter + gp.Is;
    const size_t dsm = (8 + kDownThreads / 32) * sizeof(float) + (g.n_slots * dp.J + nq) * sizeof(float) + 16;
    e = allow_smem(gateup_bf16_kernel, gsm);
    if (e == cudaSuccess) e = allow_smem(down_bf16_kernel, dsm);
    if (e == cudaSuccess)
      e = launch_pdl(gateup_bf16_kernel, dim3(g.n_units), dim3(kGuThreads), gsm, s, gp);
    if (e == cudaSuccess && !gateup_only)
      e = launch_pdl(down_bf16_kernel, dim3(down_ctas), dim3(kDownThreads), dsm, s, dp);
  }
  return cuda_status(e);
}

}  // namespace si

using namespace si;

extern "C" size_t si_moe_ffn_workspace_bytes(const si_moe_layer *L, int n_tokens) {
  if (!L || n_tokens != 1) return 0;
  return ffn_geom(*L).bytes;
}

extern "C" si_status si_moe_ffn_decode(const si_moe_layer *L, int n_tokens, const void *x,
                                       const void *x_q8_1, const int32_t *topk_ids,
                                       const float *topk_w, void *routed_out, void *shared_out,
                                       void *workspace, size_t workspace_bytes, void *stream) {
  if (!L || !x || !topk_ids || !topk_w || !routed_out) return SI_ERR_INVALID_ARG;
  if (n_tokens != 1) return SI_ERR_UNSUPPORTED;
  const si_status st = ffn_check(*L);
  if (st != SI_OK) return st;
  if (L->shared_inter > 0 && !shared_out) return SI_ERR_INVALID_ARG;
  if (!aligned16(x) || (x_q8_1 && (reinterpret_cast<uintptr_t>(x_q8_1) & 3u)) ||
      (reinterpret_cast<uintptr_t>(topk_ids) & 3u) || (reinterpret_cast<uintptr_t>(topk_w) & 3u) ||
      (reinterpret_cast<uintptr_t>(routed_out) & 1u) ||
      (shared_out && (reinterpret_cast<uintptr_t>(shared_out) & 1u)))
    return SI_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < ffn_geom(*L).bytes)
    return SI_ERR_WORKSPACE;
  return ffn_launch(*L, x, x_q8_1, topk_ids, topk_w, routed_out, shared_out, workspace,
                    static_cast<uint32_t *>(workspace), static_cast<cudaStream_t>(stream), false);
}

extern "C" si_status si_moe_ffn_decode_ep(const si_moe_layer *L, int e0, int e1, const void *x,
                                          const void *x_q8_1, const int32_t *topk_ids, float *slot_y,
                                          void *shared_out, void *workspace, size_t workspace_bytes,
                                          void *stream) {
  if (!L || !x || !topk_ids || !slot_y) return SI_ERR_INVALID_ARG;
  const si_status st = ffn_check(*L);
  if (st != SI_OK) return st;
  if (L->expert_type != SI_Q4_K) return SI_ERR_UNSUPPORTED;
  if (e0 < 0 || e1 < e0 || e1 > L->n_experts) return SI_ERR_INVALID_ARG;
  if (L->shared_inter > 0 && !shared_out) return SI_ERR_INVALID_ARG;
  if (!aligned16(x) || (x_q8_1 && (reinterpret_cast<uintptr_t>(x_q8_1) & 3u)) ||
      (reinterpret_cast<uintptr_t>(topk_ids) & 3u) || (reinterpret_cast<uintptr_t>(slot_y) & 3u) ||
      (shared_out && (reinterpret_cast<uintptr_t>(shared_out) & 1u)))
    return SI_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < ffn_geom(*L).bytes)
    return SI_ERR_WORKSPACE;
  return ffn_launch(*L, x, x_q8_1, topk_ids, nullptr, nullptr, shared_out, workspace,
                    static_cast<uint32_t *>(workspace), static_cast<cudaStream_t>(stream), false, e0, e1,
                    slot_y);
}

extern "C" si_status si_moe_combine_slots(const float *slot_y, const float *topk_w, int k, int hidden,
                                          void *routed_out, void *stream) {
  if (!slot_y || !topk_w || !routed_out || k < 1 || k > 8 || hidden < 1) return SI_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(slot_y) & 3u) || (reinterpret_cast<uintptr_t>(topk_w) & 3u) ||
      (reinterpret_cast<uintptr_t>(routed_out) & 1u))
    return SI_ERR_INVALID_ARG;
  return cuda_status(launch_pdl(combine_slots_kernel, dim3((hidden + 255) / 256), dim3(256), 0,
                                static_cast<cudaStream_t>(stream), slot_y, topk_w, k, hidden,
                                static_cast<__nv_bfloat16 *>(routed_out)));
}

extern "C" si_status si_moe_ffn_gateup(const si_moe_layer *L, int n_tokens, const void *x,
                                       const void *x_q8_1, const int32_t *topk_ids,
                                       void *workspace, size_t workspace_bytes, void *stream) {
  if (!L || !x || !topk_ids) return SI_ERR_INVALID_ARG;
  if (n_tokens != 1) return SI_ERR_UNSUPPORTED;
  const si_status st = ffn_check(*L);
  if (st != SI_OK) return st;
  if (!aligned16(x) || (x_q8_1 && (reinterpret_cast<uintptr_t>(x_q8_1) & 3u)) ||
      (reinterpret_cast<uintptr_t>(topk_ids) & 3u))
    return SI_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < ffn_geom(*L).bytes)
    return SI_ERR_WORKSPACE;
  return ffn_launch(*L, x, x_q8_1, topk_ids, nullptr, nullptr, nullptr, workspace,
                    static_cast<uint32_t *>(workspace), static_cast<cudaStream_t>(stream), true);
}

extern "C" si_status si_test_q4k_block_dots(const void *w, int rows, int k, const void *a_q8_1,
                                            int32_t *out, void *stream) {
  if (!w || !a_q8_1 || !out || rows < 1 || k < 256 || k % 256 || k > 16384) return SI_ERR_INVALID_ARG;
  if (!aligned16(w) || (reinterpret_cast<uintptr_t>(a_q8_1) & 3u)) return SI_ERR_INVALID_ARG;
  const size_t smem = (k / 256) * (kActSbStride + 64);
  cudaError_t e = allow_smem(q4k_block_dots_kernel, smem);
  if (e == cudaSuccess)
    e = launch_pdl(q4k_block_dots_kernel, dim3(rows), dim3(128), smem,
                   static_cast<cudaStream_t>(stream), static_cast<const uint8_t *>(w), rows, k,
                   static_cast<const uint8_t *>(a_q8_1), out);
  return cuda_status(e);
}

extern "C" si_status si_test_block_dots(int kind, const void *w, int rows, int k, const void *a_q8_1,
                                        int n_vec, int32_t *out, void *stream) {
  if (kind < SI_TEST_DOTS_Q4K_SB || kind > SI_TEST_DOTS_Q4K_HALF_TOKENS) return SI_ERR_INVALID_ARG;
  if (!w || !a_q8_1 || !out || rows < 1 || rows > 65535 || k < 256 || k % 256 || k > 16384 ||
      n_vec < 1)
    return SI_ERR_INVALID_ARG;
  if (!aligned16(w) || (reinterpret_cast<uintptr_t>(a_q8_1) & 3u) ||
      (reinterpret_cast<uintptr_t>(out) & 3u))
    return SI_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kind >= SI_TEST_DOTS_Q4K_SB_TOKENS) {
    if (n_vec > 8) return SI_ERR_INVALID_ARG;
    return batched_test_dots(w, rows, k, a_q8_1, n_vec, kind == SI_TEST_DOTS_Q4K_HALF_TOKENS, out, s);
  }
  if (n_vec > 65535) return SI_ERR_INVALID_ARG;
  const size_t smem = (k / 256) * (kActSbStride + 64);
  cudaError_t e = allow_smem(block_dots_kernel, smem);
  if (e == cudaSuccess)
    e = launch_pdl(block_dots_kernel, dim3(rows, n_vec), dim3(128), smem, s, kind,
                   static_cast<const uint8_t *>(w), rows, k, static_cast<const uint8_t *>(a_q8_1), out);
  return cuda_status(e);
}

#ifdef SI_TRACE
extern "C" int si_trace_dump_ffn(void *dst) {
  return cudaMemcpyFromSymbol(dst, si::g_si_trace, sizeof(si::g_si_trace)) == cudaSuccess ? 0 : 4;
}
extern "C" int si_trace_reset_ffn(void) {
  static uint64_t zeros[si::kTraceKernels * si::kTraceBlocks * si::kTracePhases];
  return cudaMemcpyToSymbol(si::g_si_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : 4;
}
#endif
