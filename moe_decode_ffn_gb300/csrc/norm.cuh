// The residual RMSNorm of one row, shared by the norm kernel (quant_norm.cu)
// and the batched layer's combine + norm kernel (batched.cu), so that both
// give the same bits.
//
// "perf(qwen3.6): fused router GEMV+top-k + folded residual-norm (decode)"
// (sparkinfer PR #273), Summary item 2: routed + shared + residual folded into
// one add+RMSNorm, bit-identical to the residual add followed by the 2-input
// norm.
//
// One block of kNormThreads threads per row; thread i owns the 8 consecutive
// values 8i .. 8i + 7 of every 2048-value slice:
//   t = bf16(a + b); s = c ? bf16(t + c) : t; r = rsqrt(mean(s^2) + eps);
//   y = bf16((s * r) * w); optional Q8_1 of y.
// With b == nullptr: t = a. Sums of squares: each thread's fma chain in value
// order, a warp butterfly, then the warps' sums in warp order.
#pragma once

#include "common.cuh"

namespace si {

constexpr int kNormThreads = 256;

// load_a(i0, va) gives the 8 values a[i0 .. i0 + 7] of this row as fp32.
// s_sum: n floats of shared memory; s_red: kNormThreads / 32 floats.
template <class LoadA>
SI_DEV void add_rmsnorm_row(LoadA load_a, const __nv_bfloat16 *__restrict__ b,
                            const __nv_bfloat16 *__restrict__ c, const __nv_bfloat16 *__restrict__ w,
                            int n, float eps, int row, __nv_bfloat16 *__restrict__ sum_out,
                            __nv_bfloat16 *__restrict__ norm_out, uint8_t *__restrict__ q8_out,
                            float *s_sum, float *s_red) {
  const size_t base = static_cast<size_t>(row) * n;
  float ss = 0.f;
  for (int i0 = 8 * threadIdx.x; i0 < n; i0 += 8 * kNormThreads) {
    float va[8], vb[8], vc[8], s[8];
    load_a(i0, va);
    if (b) Load8<__nv_bfloat16>::run(b + base + i0, vb);
    if (c) Load8<__nv_bfloat16>::run(c + base + i0, vc);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float t = b ? bf16_round(va[i] + vb[i]) : va[i];
      s[i] = c ? bf16_round(t + vc[i]) : t;
      ss = fmaf(s[i], s[i], ss);
      s_sum[i0 + i] = s[i];
    }
    uint4 o;
    o.x = bf16_bits(s[0]) | (static_cast<uint32_t>(bf16_bits(s[1])) << 16);
    o.y = bf16_bits(s[2]) | (static_cast<uint32_t>(bf16_bits(s[3])) << 16);
    o.z = bf16_bits(s[4]) | (static_cast<uint32_t>(bf16_bits(s[5])) << 16);
    o.w = bf16_bits(s[6]) | (static_cast<uint32_t>(bf16_bits(s[7])) << 16);
    *reinterpret_cast<uint4 *>(sum_out + base + i0) = o;
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += s_red[i];
  const float r = rsqrtf(__fdiv_rn(tot, static_cast<float>(n)) + eps);
  for (int i0 = 8 * threadIdx.x; i0 < n; i0 += 8 * kNormThreads) {
    float vw[8], y[8];
    Load8<__nv_bfloat16>::run(w + i0, vw);
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = bf16_round(__fmul_rn(__fmul_rn(s_sum[i0 + i], r), vw[i]));
    uint4 o;
    o.x = bf16_bits(y[0]) | (static_cast<uint32_t>(bf16_bits(y[1])) << 16);
    o.y = bf16_bits(y[2]) | (static_cast<uint32_t>(bf16_bits(y[3])) << 16);
    o.z = bf16_bits(y[4]) | (static_cast<uint32_t>(bf16_bits(y[5])) << 16);
    o.w = bf16_bits(y[6]) | (static_cast<uint32_t>(bf16_bits(y[7])) << 16);
    *reinterpret_cast<uint4 *>(norm_out + base + i0) = o;
    if (q8_out) {  // n % 256 == 0, so whole warps take this branch together
      uint32_t lo, hi;
      uint16_t d16, s16;
      q8_1_encode_4lanes(y, lo, hi, d16, s16);
      const int g = i0 / 8;
      uint8_t *blk = q8_out + (static_cast<size_t>(row) * (n / 32) + (g >> 2)) * kQ81Bytes;
      uint32_t *q = reinterpret_cast<uint32_t *>(blk + 4 + 8 * (g & 3));
      q[0] = lo;
      q[1] = hi;
      if ((g & 3) == 0) *reinterpret_cast<uint32_t *>(blk) = d16 | (static_cast<uint32_t>(s16) << 16);
    }
  }
}

}  // namespace si
