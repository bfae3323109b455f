// Shared device helpers for the decode MoE FFN kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/si_moe.h"

#define SI_DEV __device__ __forceinline__

namespace si {

constexpr int kQK = 32;          // values per Q8_0 / Q8_1 block
constexpr int kQKK = 256;        // weights per Q4_K super-block
constexpr int kQ4KBytes = 144;
constexpr int kQ80Bytes = 34;
constexpr int kQ81Bytes = 36;

// Bounded waits: a kernel that has waited this long on an mbarrier (its
// bulk copies never landed) gives up and records SI_ERR_TIMEOUT.
constexpr uint64_t kWaitBudgetNs = 1000000000ull;   // 1 s

// Device status word: first 4 bytes of every workspace.
struct WsHeader {
  uint32_t status;
  uint32_t pad[63];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

SI_DEV void record_status(uint32_t *status, uint32_t code) {
  if (status) atomicCAS(status, 0u, code);
}

// ---------------------------------------------------------------------------
// Phase tracing (profiling builds only: compiled with -DSI_TRACE). Thread 0 of
// each block stamps %globaltimer (ns) at numbered phases into a per-file
// device buffer [kernel][block][phase]; si_trace_dump copies it out.
// ---------------------------------------------------------------------------
constexpr int kTraceKernels = 4, kTraceBlocks = 1024, kTracePhases = 16;
#ifdef SI_TRACE
SI_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define SI_TRACE_BUFFER static __device__ uint64_t g_si_trace[kTraceKernels][kTraceBlocks][kTracePhases];
#define SI_TRACE_MARK(kernel, phase)                                                         \
  do {                                                                                       \
    if (threadIdx.x == 0 && blockIdx.x < kTraceBlocks && blockIdx.y == 0)                    \
      g_si_trace[(kernel)][blockIdx.x][(phase)] = globaltimer_ns();                          \
  } while (0)
// Latest %globaltimer over the block's threads (any thread may call it).
#define SI_TRACE_LATEST(kernel, phase)                                                       \
  do {                                                                                       \
    if (blockIdx.x < kTraceBlocks && blockIdx.y == 0)                                        \
      atomicMax(reinterpret_cast<unsigned long long *>(&g_si_trace[(kernel)][blockIdx.x][(phase)]), \
                static_cast<unsigned long long>(globaltimer_ns()));                          \
  } while (0)
#else
#define SI_TRACE_BUFFER
#define SI_TRACE_MARK(kernel, phase) \
  do {                               \
  } while (0)
#define SI_TRACE_LATEST(kernel, phase) \
  do {                                 \
  } while (0)
#endif

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------
SI_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
SI_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// mbarrier + bulk async copy (TMA, 1-D)
// ---------------------------------------------------------------------------
SI_DEV uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SI_DEV void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

SI_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

SI_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

SI_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

SI_DEV uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Reading %globaltimer stalls the reading thread for about half a
// microsecond on GB300, longer than most of the waits below: every bounded
// wait therefore spins a fixed number of times before it first reads the
// clock, and then reads it only between long runs of attempts.
constexpr int kSpinBeforeClock = 4096;

// Wait for phase `parity` of `bar` for at most about `budget_ns` (plus the
// initial spin). Returns false on timeout (after recording SI_ERR_TIMEOUT).
// The spin loop is out of line so that every call site stays one try_wait
// long.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t *bar, uint32_t parity,
                                                   uint32_t *status, uint64_t budget_ns) {
#pragma unroll 1
  for (int i = 0; i < kSpinBeforeClock; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (now_ns() - t0 > budget_ns) break;
  }
  record_status(status, SI_ERR_TIMEOUT);
  return false;
}
SI_DEV bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t *status,
                              uint64_t budget_ns = kWaitBudgetNs) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, status, budget_ns);
}

// Global -> shared bulk copy completing on `bar` (bytes and both addresses
// must be multiples of 16).
SI_DEV void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Same, with an L2 eviction hint: weights streamed once per token.
SI_DEV void bulk_g2s_evict_first(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                 uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

SI_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------
SI_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
SI_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
SI_DEV float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }
SI_DEV uint16_t bf16_bits(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t *>(&b);
}
SI_DEV float half_bits_to_float(uint16_t h) {
  __half_raw r;
  r.x = h;
  return __half2float(__half(r));
}
SI_DEV uint16_t float_to_half_bits(float v) {
  __half h = __float2half_rn(v);
  return reinterpret_cast<__half_raw &>(h).x;
}

// Load 8 consecutive values of type T as fp32 (16-byte aligned for bf16).
template <typename T> struct Load8;
template <> struct Load8<__nv_bfloat16> {
  static SI_DEV void run(const void *p, float v[8]) {
    uint4 u = *reinterpret_cast<const uint4 *>(p);
    v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
    v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
  }
};
template <> struct Load8<float> {
  static SI_DEV void run(const void *p, float v[8]) {
    float4 a = reinterpret_cast<const float4 *>(p)[0];
    float4 b = reinterpret_cast<const float4 *>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

// ---------------------------------------------------------------------------
// Q8_1 block encoder, cooperative over 4 lanes of one warp (lanes 4g..4g+3
// hold values 8*(lane&3) .. +7 of one 32-value block).
//   d32 = amax / 127 (IEEE), q = round-half-away(x / d32) clamped to +-127,
//   d16 = fp16(d32), s16 = fp16(d32 * sum q).
// Outputs: this lane's 8 codes packed in two words (little-endian bytes) and,
// identical on the 4 lanes, d16 and s16 bits.
// ---------------------------------------------------------------------------
SI_DEV void q8_1_encode_4lanes(const float v[8], uint32_t &q_lo, uint32_t &q_hi, uint16_t &d16,
                               uint16_t &s16) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const float d = __fdiv_rn(amax, 127.0f);
  const bool live = d > 0.f;          // d == 0: every code is 0
  const float dd = live ? d : 1.0f;
  int qi[8];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float r = fminf(fmaxf(roundf(__fdiv_rn(v[i], dd)), -127.f), 127.f);
    qi[i] = live ? static_cast<int>(r) : 0;
    sum += qi[i];
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  q_lo = (qi[0] & 0xFF) | ((qi[1] & 0xFF) << 8) | ((qi[2] & 0xFF) << 16) |
         (static_cast<uint32_t>(qi[3] & 0xFF) << 24);
  q_hi = (qi[4] & 0xFF) | ((qi[5] & 0xFF) << 8) | ((qi[6] & 0xFF) << 16) |
         (static_cast<uint32_t>(qi[7] & 0xFF) << 24);
  d16 = float_to_half_bits(d);
  s16 = float_to_half_bits(__fmul_rn(d, static_cast<float>(sum)));
}

// Same encoding with one value per lane: the 32 lanes of a warp hold one
// block (lane i = value i). One division per lane keeps the dependent chain
// short. Returns this lane's code; d16 / s16 identical on every lane.
SI_DEV int q8_1_encode_warp(float v, uint16_t &d16, uint16_t &s16) {
  // |v| as bits orders like the values (non-negative floats), so one warp
  // reduction gives amax; a second gives the exact integer sum of the codes
  const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
  const float d = __fdiv_rn(amax, 127.0f);
  const bool live = d > 0.f;
  const float r = fminf(fmaxf(roundf(__fdiv_rn(v, live ? d : 1.0f)), -127.f), 127.f);
  const int q = live ? static_cast<int>(r) : 0;
  const int sum = __reduce_add_sync(0xffffffffu, q);
  d16 = float_to_half_bits(d);
  s16 = float_to_half_bits(__fmul_rn(d, static_cast<float>(sum)));
  return q;
}

// ---------------------------------------------------------------------------
// Activation tile in shared memory, the form every quantised GEMV reads.
// Codes of 256-value super-block b live at qs + b * kActSbStride (256 bytes of
// codes + 16 bytes of padding, which keeps the 8 lanes that read 8
// consecutive super-blocks on distinct banks). d and s are the fp16 block
// scale and sum widened to fp32, per 32-block.
// ---------------------------------------------------------------------------
constexpr int kActSbStride = 272;

struct ActTile {
  uint8_t *qs;  // [nsb][272]
  float *d;     // [nsb * 8]
  float *s;     // [nsb * 8]
};

// Quantise n (multiple of 256) values of `x` (row of T) into an ActTile, all
// threads of the block cooperating (blockDim multiple of 32). Ends with
// __syncthreads().
template <typename T>
SI_DEV void quantize_to_tile(const T *x, int n, ActTile t) {
  const int groups = n / 8;  // 8 values per lane, 4 lanes per 32-block
  for (int g0 = 0; g0 < groups; g0 += blockDim.x) {
    const int g = g0 + threadIdx.x;
    const bool live = g < groups;   // warp-uniform when groups % 32 == 0
    float v[8];
    if (live) {
      Load8<T>::run(x + 8 * g, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    uint32_t lo, hi;
    uint16_t d16, s16;
    q8_1_encode_4lanes(v, lo, hi, d16, s16);
    if (live) {
      const int blk = g >> 2, part = g & 3;
      uint8_t *dst = t.qs + (blk >> 3) * kActSbStride + (blk & 7) * 32 + part * 8;
      *reinterpret_cast<uint2 *>(dst) = make_uint2(lo, hi);
      if (part == 0) {
        t.d[blk] = half_bits_to_float(d16);
        t.s[blk] = half_bits_to_float(s16);
      }
    }
  }
  __syncthreads();
}

// Fill an ActTile from Q8_1 blocks in global memory (36-byte blocks), all
// threads of the block cooperating. Ends with __syncthreads().
SI_DEV void tile_from_q8_1(const uint8_t *src, int n, ActTile t) {
  const int words = n / 32 * 9;
  for (int i = threadIdx.x; i < words; i += blockDim.x) {
    const int blk = i / 9, w = i % 9;
    const uint32_t v = __ldcg(reinterpret_cast<const uint32_t *>(src + blk * kQ81Bytes) + w);
    if (w == 0) {
      t.d[blk] = half_bits_to_float(static_cast<uint16_t>(v & 0xFFFF));
      t.s[blk] = half_bits_to_float(static_cast<uint16_t>(v >> 16));
    } else {
      *reinterpret_cast<uint32_t *>(t.qs + (blk >> 3) * kActSbStride + (blk & 7) * 32 + 4 * (w - 1)) = v;
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Q4_K super-block x Q8_1 activations.
// w: the 144-byte super-block (16-byte aligned, shared memory);
// a: the 256 activation codes of the matching super-block (16-byte aligned);
// isum[j] = exact sum over sub-block j of q_w * q_a.
// ---------------------------------------------------------------------------
SI_DEV void q4k_unpack_scales(const uint32_t sw[3], int sc[8], int mn[8]) {
  // sw = the 12 scale bytes as 3 little-endian words.
  const uint8_t *b = reinterpret_cast<const uint8_t *>(sw);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    sc[j] = b[j] & 63;
    mn[j] = b[j + 4] & 63;
    sc[j + 4] = (b[j + 8] & 0x0F) | ((b[j] >> 6) << 4);
    mn[j + 4] = (b[j + 8] >> 4) | ((b[j + 4] >> 6) << 4);
  }
}

// Exact int32 sums of one pair of Q4_K sub-blocks with their activation
// codes: sub-block 2p is the low nibbles, 2p + 1 the high nibbles of the
// pair's 32 code bytes (qw, 8 little-endian words); a points at the pair's 64
// activation codes (sub-block 2p, then 2p + 1). Every Q4_K dot of the library
// reduces its codes through this one function.
SI_DEV void q4k_pair_isums(const uint32_t *qw, const uint4 *a, int &lo, int &hi) {
  const uint4 al0 = a[0], al1 = a[1], ah0 = a[2], ah1 = a[3];
  const uint32_t aw_lo[8] = {al0.x, al0.y, al0.z, al0.w, al1.x, al1.y, al1.z, al1.w};
  const uint32_t aw_hi[8] = {ah0.x, ah0.y, ah0.z, ah0.w, ah1.x, ah1.y, ah1.z, ah1.w};
  lo = 0;
  hi = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    lo = __dp4a(static_cast<int>(qw[i] & 0x0F0F0F0Fu), static_cast<int>(aw_lo[i]), lo);
    hi = __dp4a(static_cast<int>((qw[i] >> 4) & 0x0F0F0F0Fu), static_cast<int>(aw_hi[i]), hi);
  }
}

// The 8 code words of pair p of a Q4_K super-block w (16-byte aligned).
SI_DEV void q4k_pair_words(const uint4 *w, int p, uint32_t qw[8]) {
  const uint4 q0 = w[1 + 2 * p], q1 = w[2 + 2 * p];
  qw[0] = q0.x; qw[1] = q0.y; qw[2] = q0.z; qw[3] = q0.w;
  qw[4] = q1.x; qw[5] = q1.y; qw[6] = q1.z; qw[7] = q1.w;
}

SI_DEV void q4k_isums(const uint4 *w, const uint4 *a, int isum[8], uint32_t &dd,
                      uint32_t sw[3]) {
  uint4 h = w[0];  // d, dmin, scale bytes 0..11
  dd = h.x;
  sw[0] = h.y; sw[1] = h.z; sw[2] = h.w;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint32_t qw[8];
    q4k_pair_words(w, p, qw);
    q4k_pair_isums(qw, a + 4 * p, isum[2 * p], isum[2 * p + 1]);
  }
}

// Exact float of an integer |v| < 2^22 (the exponent-bias conversion): v is
// added to the bit pattern of 1.5 * 2^23, whose unit in the last place is 1,
// and the bias is taken off again by one exact fp32 subtraction. It serves
// the scaled Q4_K sub-block sums (|sc * isum| <= 63 * 32 * 15 * 128 < 2^22)
// and the Q8_0 block sums (<= 32 * 128 * 128); Q5_K's scaled sums can pass
// 2^22 and keep the plain conversion.
SI_DEV float isum_to_float(int v) { return __fsub_rn(__int_as_float(0x4B400000 + v), 12582912.f); }

// Half h of a Q4_K super-block (sub-blocks 4h .. 4h + 3, 128 weights):
// isum[i] = exact sum over sub-block 4h + i of q_w * q_a.
SI_DEV void q4k_half_isums(const uint4 *w, const uint4 *a, int h, int isum[4]) {
#pragma unroll
  for (int pp = 0; pp < 2; ++pp) {
    const int p = 2 * h + pp;
    uint32_t qw[8];
    q4k_pair_words(w, p, qw);
    q4k_pair_isums(qw, a + 4 * p, isum[2 * pp], isum[2 * pp + 1]);
  }
}

// Pairs [p0, p0 + np) of one Q4_K super-block (pair p = sub-blocks 2p and
// 2p + 1, 64 weights): d * sum_j sc_j*d_a(j)*isum_j - dmin * sum_j m_j*s_a(j)
// over those j, the two sums accumulated in sub-block order, then one
// rounding per product and one for the difference. w: the 144-byte
// super-block, a: its 256 activation codes (both 16-byte aligned, shared
// memory); da, sa: the activation scales and sums of its 8 blocks. A rolled
// loop kept out of line: one copy of the code serves every caller.
static __device__ __noinline__ float q4k_dot_pairs(const uint8_t *w, const uint8_t *a,
                                                   const float *da, const float *sa, int p0,
                                                   int np) {
  float acc_d = 0.f, acc_m = 0.f;
  const uint8_t *sb = w + 4;   // the 12 scale bytes
#pragma unroll 1
  for (int p = p0; p < p0 + np; ++p) {
    uint32_t qw[8];
    q4k_pair_words(reinterpret_cast<const uint4 *>(w), p, qw);
    int lo, hi;
    q4k_pair_isums(qw, reinterpret_cast<const uint4 *>(a) + 4 * p, lo, hi);
    // 6-bit scale and min of sub-blocks j = 2p, 2p + 1 (j < 4: low 6 bits of
    // bytes j, j + 4; j >= 4: nibbles of byte j + 4 plus the top 2 bits of
    // bytes j - 4, j)
    int sc[2], mn[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int j = 2 * p + e;
      if (j < 4) {
        sc[e] = sb[j] & 63;
        mn[e] = sb[j + 4] & 63;
      } else {
        sc[e] = (sb[j + 4] & 0x0F) | ((sb[j - 4] >> 6) << 4);
        mn[e] = (sb[j + 4] >> 4) | ((sb[j] >> 6) << 4);
      }
    }
    acc_d = fmaf(isum_to_float(sc[0] * lo), da[2 * p], acc_d);
    acc_d = fmaf(isum_to_float(sc[1] * hi), da[2 * p + 1], acc_d);
    acc_m = fmaf(static_cast<float>(mn[0]), sa[2 * p], acc_m);
    acc_m = fmaf(static_cast<float>(mn[1]), sa[2 * p + 1], acc_m);
  }
  const uint32_t dd = *reinterpret_cast<const uint32_t *>(w);
  const float d = half_bits_to_float(static_cast<uint16_t>(dd & 0xFFFF));
  const float dmin = half_bits_to_float(static_cast<uint16_t>(dd >> 16));
  return __fsub_rn(__fmul_rn(d, acc_d), __fmul_rn(dmin, acc_m));
}

// The same two functions fully unrolled and inline, for kernels that run
// once per launch (their code is fetched once): half of a super-block
// (sub-blocks 4h..4h+3, 128 weights) and the whole super-block. Same order of
// accumulation and rounding as q4k_dot_pairs, so the same bits.
//
// A half taken apart ahead of its dot product: the 16 code words of its two
// pairs, the 6-bit scales and mins of its four sub-blocks (packed one per
// byte), d and dmin. The scales of sub-blocks 4..7 are their low nibble in
// bytes 8..11 plus the top two bits of bytes 0..3 (mins: high nibble, bytes
// 4..7), so all four come out of three words with a few masks.
struct Q4KHalf {
  uint32_t qw[16];
  uint32_t scw, mnw;
  float d, dmin;
};
SI_DEV void q4k_half_load(const uint4 *w, int h, Q4KHalf &q) {
  const uint4 hd = w[0];
  if (h) {
    q.scw = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
    q.mnw = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
  } else {
    q.scw = hd.y & 0x3F3F3F3Fu;
    q.mnw = hd.z & 0x3F3F3F3Fu;
  }
  q4k_pair_words(w, 2 * h, q.qw);
  q4k_pair_words(w, 2 * h + 1, q.qw + 8);
  q.d = half_bits_to_float(static_cast<uint16_t>(hd.x & 0xFFFF));
  q.dmin = half_bits_to_float(static_cast<uint16_t>(hd.x >> 16));
}
SI_DEV float q4k_half_dot_loaded(const Q4KHalf &q, const uint4 *a, const float *da, const float *sa,
                                 int h) {
  int isum[4];
  q4k_pair_isums(q.qw, a + 4 * (2 * h), isum[0], isum[1]);
  q4k_pair_isums(q.qw + 8, a + 4 * (2 * h + 1), isum[2], isum[3]);
  float acc_d = 0.f, acc_m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int sc = static_cast<int>((q.scw >> (8 * i)) & 0xFFu);
    const int mn = static_cast<int>((q.mnw >> (8 * i)) & 0xFFu);
    acc_d = fmaf(isum_to_float(sc * isum[i]), da[4 * h + i], acc_d);
    acc_m = fmaf(static_cast<float>(mn), sa[4 * h + i], acc_m);
  }
  return __fsub_rn(__fmul_rn(q.d, acc_d), __fmul_rn(q.dmin, acc_m));
}
SI_DEV float q4k_half_dot(const uint4 *w, const uint4 *a, const float *da, const float *sa,
                          int h) {
  Q4KHalf q;
  q4k_half_load(w, h, q);
  return q4k_half_dot_loaded(q, a, da, sa, h);
}

SI_DEV float q4k_sb_dot(const uint4 *w, const uint4 *a, const float *da, const float *sa) {
  int isum[8];
  uint32_t dd, sw[3];
  q4k_isums(w, a, isum, dd, sw);
  // scales / mins of sub-blocks 0..3 and 4..7, one per byte
  const uint32_t sc0 = sw[0] & 0x3F3F3F3Fu, mn0 = sw[1] & 0x3F3F3F3Fu;
  const uint32_t sc1 = (sw[2] & 0x0F0F0F0Fu) | ((sw[0] >> 2) & 0x30303030u);
  const uint32_t mn1 = ((sw[2] >> 4) & 0x0F0F0F0Fu) | ((sw[1] >> 2) & 0x30303030u);
  float acc_d = 0.f, acc_m = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int sc = static_cast<int>(((j < 4 ? sc0 : sc1) >> (8 * (j & 3))) & 0xFFu);
    const int mn = static_cast<int>(((j < 4 ? mn0 : mn1) >> (8 * (j & 3))) & 0xFFu);
    acc_d = fmaf(isum_to_float(sc * isum[j]), da[j], acc_d);
    acc_m = fmaf(static_cast<float>(mn), sa[j], acc_m);
  }
  const float d = half_bits_to_float(static_cast<uint16_t>(dd & 0xFFFF));
  const float dmin = half_bits_to_float(static_cast<uint16_t>(dd >> 16));
  return __fsub_rn(__fmul_rn(d, acc_d), __fmul_rn(dmin, acc_m));
}

// Q5_K super-block (176 bytes: fp16 d, fp16 dmin, 12 scale bytes as Q4_K,
// qh[32] fifth bits, 128 code bytes as Q4_K's codes) x Q8_1, half h
// (sub-blocks 4h..4h+3): the Q4_K half dot with each code's fifth bit (bit j
// of qh[i] for element i of sub-block j) OR-ed in as 16 before the dp4a.
constexpr int kQ5KBytes = 176;
// isum[i] = exact sum over sub-block 4h + i of q_w * q_a (q_w in 0..31).
SI_DEV void q5k_half_isums(const uint8_t *w, const uint4 *a, int h, int isum[4]) {
  const uint4 qh0 = *reinterpret_cast<const uint4 *>(w + 16);
  const uint4 qh1 = *reinterpret_cast<const uint4 *>(w + 32);
  const uint32_t qhw[8] = {qh0.x, qh0.y, qh0.z, qh0.w, qh1.x, qh1.y, qh1.z, qh1.w};
#pragma unroll
  for (int pp = 0; pp < 2; ++pp) {
    const int p = 2 * h + pp;
    const uint4 q0 = *reinterpret_cast<const uint4 *>(w + 48 + 32 * p);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(w + 64 + 32 * p);
    const uint4 al0 = a[4 * p + 0], al1 = a[4 * p + 1];
    const uint4 ah0 = a[4 * p + 2], ah1 = a[4 * p + 3];
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t aw_lo[8] = {al0.x, al0.y, al0.z, al0.w, al1.x, al1.y, al1.z, al1.w};
    const uint32_t aw_hi[8] = {ah0.x, ah0.y, ah0.z, ah0.w, ah1.x, ah1.y, ah1.z, ah1.w};
    int lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t b_lo = ((qhw[i] >> (2 * p)) & 0x01010101u) << 4;
      const uint32_t b_hi = ((qhw[i] >> (2 * p + 1)) & 0x01010101u) << 4;
      lo = __dp4a(static_cast<int>((qw[i] & 0x0F0F0F0Fu) | b_lo), static_cast<int>(aw_lo[i]), lo);
      hi = __dp4a(static_cast<int>(((qw[i] >> 4) & 0x0F0F0F0Fu) | b_hi), static_cast<int>(aw_hi[i]), hi);
    }
    isum[2 * pp] = lo;
    isum[2 * pp + 1] = hi;
  }
}

SI_DEV float q5k_half_dot(const uint8_t *w, const uint4 *a, const float *da, const float *sa, int h) {
  const uint4 hd = *reinterpret_cast<const uint4 *>(w);
  int sc8[8], mn8[8];
  const uint32_t sw[3] = {hd.y, hd.z, hd.w};
  q4k_unpack_scales(sw, sc8, mn8);
  int sc[4], mn[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    sc[i] = h ? sc8[4 + i] : sc8[i];
    mn[i] = h ? mn8[4 + i] : mn8[i];
  }
  int isum[4];
  q5k_half_isums(w, a, h, isum);
  float acc_d = 0.f, acc_m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc_d = fmaf(static_cast<float>(sc[i] * isum[i]), da[4 * h + i], acc_d);
    acc_m = fmaf(static_cast<float>(mn[i]), sa[4 * h + i], acc_m);
  }
  const float d = half_bits_to_float(static_cast<uint16_t>(hd.x & 0xFFFF));
  const float dmin = half_bits_to_float(static_cast<uint16_t>(hd.x >> 16));
  return __fsub_rn(__fmul_rn(d, acc_d), __fmul_rn(dmin, acc_m));
}

// Q8_0 x Q8_1 over 256 weights = 8 Q8_0 blocks (272 bytes, 16-byte aligned).
SI_DEV float q80_sb_dot(const uint4 *w, const uint4 *a, const float *da) {
  uint32_t ww[68];
#pragma unroll
  for (int i = 0; i < 17; ++i) {
    const uint4 u = w[i];
    ww[4 * i] = u.x; ww[4 * i + 1] = u.y; ww[4 * i + 2] = u.z; ww[4 * i + 3] = u.w;
  }
  float acc = 0.f;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    // block b starts at byte 34*b: fp16 d, then 32 code bytes.
    const int off = 34 * b;
    const int wi = off >> 2;
    uint32_t dword = ww[wi];
    const uint16_t dbits = (off & 2) ? static_cast<uint16_t>(dword >> 16)
                                     : static_cast<uint16_t>(dword & 0xFFFF);
    const int cstart = off + 2;  // byte offset of codes, 4-aligned when (off & 2)
    int s = 0;
    const uint4 a0 = a[2 * b], a1 = a[2 * b + 1];
    const uint32_t aw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t q;
      if (cstart & 2)
        q = __byte_perm(ww[(cstart >> 2) + i], ww[(cstart >> 2) + i + 1], 0x5432);
      else
        q = ww[(cstart >> 2) + i];
      s = __dp4a(static_cast<int>(q), static_cast<int>(aw[i]), s);
    }
    acc = fmaf(half_bits_to_float(dbits) * da[b], isum_to_float(s), acc);
  }
  return acc;
}

// Global -> L2 bulk prefetch (no destination, no completion; address and
// bytes multiples of 16). A later read of the range hits L2.
SI_DEV void bulk_prefetch_l2(const void *src_gmem, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// bf16 weight rows against fp32 activations (the bf16 gate/up and down dot
// products; every path that computes them uses these, in this order).
// ---------------------------------------------------------------------------
// Lane `lane` of every warp owns columns c0 + 256 c + 8 lane .. + 7 (c < 8)
// of each 2048-wide chunk of a row; x sits in shared memory as packed bf16
// (exact), so a lane's 16-byte reads of it are consecutive across the warp
// (no bank conflicts).
SI_DEV void load_row8(const __nv_bfloat16 *row, int c0, int H, int lane, uint4 w[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int k0 = c0 + (c * 32 + lane) * 8;
    if (k0 < H) w[c] = __ldcs(reinterpret_cast<const uint4 *>(row + k0));
  }
}

SI_DEV void dot_row8(const uint4 w[8], const uint4 *xs, int c0, int H, int lane, float &acc) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int k0 = c0 + (c * 32 + lane) * 8;
    if (k0 < H) {
      float wv[8], xv[8];
      Load8<__nv_bfloat16>::run(&w[c], wv);
      Load8<__nv_bfloat16>::run(&xs[k0 / 8], xv);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(wv[i], xv[i], acc);
    }
  }
}

// A 512-wide chunk of a down row: lane l8 of the task's 8 lanes holds
// columns cc + 8 l8 + 64 it .. + 7 (it < 8).
SI_DEV void load_down8(const __nv_bfloat16 *row, int cc, int width, int l8, uint4 u[8]) {
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int c = cc + l8 * 8 + 64 * it;
    if (row && c < width) u[it] = __ldcs(reinterpret_cast<const uint4 *>(row + c));
  }
}

SI_DEV void dot_down8(const uint4 u[8], const float *hv, int cc, int width, int l8, float &acc) {
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int c = cc + l8 * 8 + 64 * it;
    if (c < width) {
      float wv[8];
      Load8<__nv_bfloat16>::run(&u[it], wv);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(wv[i], hv[c + i], acc);
    }
  }
}

}  // namespace si
