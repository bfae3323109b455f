// Load-time requant of Q8_0 or Q5_K weight matrices to Q4_K.
//
// "perf(qwen36): Q4_K shared-expert FFN kernels + Q8_0/Q5_K->Q4_K requant of
// the MoE FFN stage" (PR #359), Summary bullets 1 and 2: the shared expert
// ships as Q8_0 and the routed down projection as Q5_K; both are requantised
// to Q4_K once, at model load, to cut the bytes every token reads. The page
// names the formats, not the procedure; here the source is dequantised to fp32
// and quantised with the library's min/max Q4_K quantiser, every step one IEEE
// fp32 operation:
//   per 32-wide sub-block j: lo = min w if negative else +0, hi = max w if
//   positive else +0, s_j = (hi - lo) / 15, m'_j = -lo;
//   d = fp16(max_j s_j / 63), dmin = fp16(max_j m'_j / 63);
//   sc_j = rint(s_j / d), m_j = rint(m'_j / dmin) in [0, 63] (0 if the divisor is 0);
//   q = rint((w + dmin * m_j) / (d * sc_j)) in [0, 15] (0 if the divisor is 0).
// One warp per super-block: lane i holds element i of each of the 8 sub-blocks.
#include "common.cuh"
#include "host.hpp"

namespace si {

constexpr int kRqThreads = 256;   // 8 super-blocks per block

SI_DEV float warp_min(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}
SI_DEV float warp_max(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}
SI_DEV float ld_half(const uint8_t *p) {   // fp16 at any 2-byte position, byte by byte
  return half_bits_to_float(static_cast<uint16_t>(p[0] | (p[1] << 8)));
}

__global__ void __launch_bounds__(kRqThreads) requant_q4k_kernel(const uint8_t *src, int src_q5,
                                                                 int64_t rows, int nsb,
                                                                 size_t src_row_bytes,
                                                                 uint8_t *dst) {
  const int lane = threadIdx.x & 31;
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * (kRqThreads / 32) + (threadIdx.x >> 5);
  if (blk >= rows * nsb) return;   // warp-uniform
  const int64_t r = blk / nsb;
  const int sb = static_cast<int>(blk - r * nsb);
  const uint8_t *row = src + static_cast<size_t>(r) * src_row_bytes;

  // ---- source weights, fp32 ----------------------------------------------------
  float x[8];
  if (src_q5) {
    // Q5_K: w = d * sc_j * q - dmin * m_j, each product exact, one rounding
    const uint8_t *b = row + static_cast<size_t>(sb) * kQ5KBytes;
    const float d = ld_half(b), dmin = ld_half(b + 2);
    const uint32_t sw[3] = {static_cast<uint32_t>(b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24)),
                            static_cast<uint32_t>(b[8] | (b[9] << 8) | (b[10] << 16) | (b[11] << 24)),
                            static_cast<uint32_t>(b[12] | (b[13] << 8) | (b[14] << 16) | (b[15] << 24))};
    int sc[8], mn[8];
    q4k_unpack_scales(sw, sc, mn);
    const int qh = b[16 + lane];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int byte = b[48 + 32 * (j >> 1) + lane];
      const int q = ((j & 1) ? (byte >> 4) : (byte & 15)) | (((qh >> j) & 1) << 4);
      x[j] = __fsub_rn(__fmul_rn(__fmul_rn(d, static_cast<float>(sc[j])), static_cast<float>(q)),
                       __fmul_rn(dmin, static_cast<float>(mn[j])));
    }
  } else {
    // Q8_0: super-block sb covers source blocks 8 sb .. 8 sb + 7 (34 bytes each)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint8_t *b = row + static_cast<size_t>(8 * sb + j) * kQ80Bytes;
      x[j] = __fmul_rn(ld_half(b), static_cast<float>(static_cast<int8_t>(b[2 + lane])));
    }
  }

  // ---- Q4_K of the 256 values ----------------------------------------------------
  float s[8], mneg[8];
  float smax = 0.f, mmax = -0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float mn = warp_min(x[j]), mx = warp_max(x[j]);
    const float lo = mn < 0.f ? mn : 0.f;
    const float hi = mx > 0.f ? mx : 0.f;
    s[j] = __fdiv_rn(__fsub_rn(hi, lo), 15.f);
    mneg[j] = -lo;
    smax = fmaxf(smax, s[j]);        // s >= +0: no signed-zero ambiguity
    mmax = j == 0 ? mneg[j] : fmaxf(mmax, mneg[j]);   // m' is -0 or positive
  }
  const uint16_t d16 = float_to_half_bits(__fdiv_rn(smax, 63.f));
  const uint16_t dm16 = float_to_half_bits(__fdiv_rn(mmax, 63.f));
  const float d = half_bits_to_float(d16), dm = half_bits_to_float(dm16);
  int sc[8], m[8], q[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sc[j] = d > 0.f ? static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(s[j], d)), 0.f), 63.f)) : 0;
    m[j] = dm > 0.f ? static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(mneg[j], dm)), 0.f), 63.f)) : 0;
    const float den = __fmul_rn(d, static_cast<float>(sc[j]));
    const float num = __fadd_rn(x[j], __fmul_rn(dm, static_cast<float>(m[j])));
    q[j] = den > 0.f ? static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(num, den)), 0.f), 15.f)) : 0;
  }

  // ---- pack (GGUF K-quant layout) -------------------------------------------------
  uint8_t *o = dst + (static_cast<size_t>(r) * nsb + sb) * kQ4KBytes;
#pragma unroll
  for (int p = 0; p < 4; ++p)
    o[16 + 32 * p + lane] = static_cast<uint8_t>(q[2 * p] | (q[2 * p + 1] << 4));
  if (lane == 0) {
    o[0] = static_cast<uint8_t>(d16 & 0xFF);
    o[1] = static_cast<uint8_t>(d16 >> 8);
    o[2] = static_cast<uint8_t>(dm16 & 0xFF);
    o[3] = static_cast<uint8_t>(dm16 >> 8);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      o[4 + j] = static_cast<uint8_t>((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
      o[8 + j] = static_cast<uint8_t>((m[j] & 63) | ((m[j + 4] >> 4) << 6));
      o[12 + j] = static_cast<uint8_t>((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
  }
}

}  // namespace si

using namespace si;

extern "C" si_status si_requant_q4_k(const void *src, si_dtype src_type, int64_t rows,
                                     int64_t cols, void *dst, void *stream) {
  if (!src || !dst || rows < 0 || cols <= 0 || cols % 256 || cols > (int64_t(1) << 30))
    return SI_ERR_INVALID_ARG;
  if (src_type != SI_Q8_0 && src_type != SI_Q5_K) return SI_ERR_UNSUPPORTED;
  if (rows == 0) return SI_OK;
  const int nsb = static_cast<int>(cols / 256);
  const size_t src_row_bytes = src_type == SI_Q5_K ? static_cast<size_t>(nsb) * kQ5KBytes
                                                   : static_cast<size_t>(cols / 32) * kQ80Bytes;
  const int64_t blocks = rows * nsb;
  const int64_t grid = (blocks + kRqThreads / 32 - 1) / (kRqThreads / 32);
  if (grid > 0x7FFFFFFF) return SI_ERR_INVALID_ARG;
  requant_q4k_kernel<<<static_cast<unsigned>(grid), kRqThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t *>(src), src_type == SI_Q5_K ? 1 : 0, rows, nsb, src_row_bytes,
      static_cast<uint8_t *>(dst));
  return cuda_status(cudaGetLastError());
}
