// Q8_1 activation quantisation and the 3-input residual RMSNorm.
//
// "Q4_K shared-expert FFN kernels + Q8_0/Q5_K->Q4_K requant of the MoE FFN
// stage" (sparkinfer PR #359), Summary: activations enter the expert GEMVs as
// Q8_1 blocks ("FNQ Q8_1", "quant_h Q8_1").
// "perf(qwen3.6): fused router GEMV+top-k + folded residual-norm (decode)"
// (sparkinfer PR #273), Summary item 2: routed + shared + residual folded into
// one add+RMSNorm, bit-identical to the residual add followed by the 2-input
// norm.
#include "common.cuh"
#include "host.hpp"
#include "norm.cuh"

namespace si {

// A block quantises a chunk of 64 U Q8_1 blocks (2048 U values): its loads
// are 16-byte, coalesced, U per thread issued before the first encode (U = 4
// for long vectors; 1 for short ones, where the chunk is the whole vector);
// the encoder takes 4 consecutive lanes per 32-value block (lane 4j + i holds
// values 8i .. 8i + 7 of one block); the 36-byte blocks are assembled in
// shared memory and leave as consecutive 16-byte stores (4-byte stores when
// y is not 16-byte aligned or for the last, partial chunk).
constexpr int kQuantThreads = 256;
template <typename T, int U>
__global__ void __launch_bounds__(kQuantThreads) quantize_q8_1_kernel(const T *__restrict__ x, int64_t n,
                                                                     uint8_t *__restrict__ y, int y_vec16) {
  constexpr int kChunkBlocks = kQuantThreads * U / 4;
  __shared__ __align__(16) uint32_t s_out[kChunkBlocks * kQ81Bytes / 4];
  grid_dep_wait();
  grid_dep_launch();
  const int64_t groups = n / 8;
  const int64_t g0 = static_cast<int64_t>(blockIdx.x) * kQuantThreads * U;
  float v[U][8];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t g = g0 + u * kQuantThreads + threadIdx.x;
    if (g < groups) {
      Load8<T>::run(x + 8 * g, v[u]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[u][i] = 0.f;
    }
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    uint32_t lo, hi;
    uint16_t d16, s16;
    q8_1_encode_4lanes(v[u], lo, hi, d16, s16);
    const int gl = u * kQuantThreads + threadIdx.x;   // group within the chunk
    uint32_t *blk = s_out + (gl >> 2) * (kQ81Bytes / 4);
    const int part = gl & 3;
    blk[1 + 2 * part] = lo;
    blk[2 + 2 * part] = hi;
    if (part == 0) blk[0] = d16 | (static_cast<uint32_t>(s16) << 16);
  }
  __syncthreads();
  const int64_t nblk_all = n / 32;
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * kChunkBlocks;
  const int nblk = nblk_all - b0 < kChunkBlocks ? static_cast<int>(nblk_all - b0) : kChunkBlocks;
  uint8_t *dst = y + b0 * kQ81Bytes;
  if (y_vec16 && nblk == kChunkBlocks) {
    const uint4 *src = reinterpret_cast<const uint4 *>(s_out);
#pragma unroll 1
    for (int i = threadIdx.x; i < kChunkBlocks * kQ81Bytes / 16; i += kQuantThreads)
      reinterpret_cast<uint4 *>(dst)[i] = src[i];
  } else {
#pragma unroll 1
    for (int i = threadIdx.x; i < nblk * (kQ81Bytes / 4); i += kQuantThreads)
      reinterpret_cast<uint32_t *>(dst)[i] = s_out[i];
  }
}

// ---------------------------------------------------------------------------
// add_rmsnorm: one block per row (the row function of norm.cuh).
// ---------------------------------------------------------------------------
SI_TRACE_BUFFER

__global__ void __launch_bounds__(kNormThreads)
    add_rmsnorm_kernel(const __nv_bfloat16 *__restrict__ a, const __nv_bfloat16 *__restrict__ b,
                       const __nv_bfloat16 *__restrict__ c, const __nv_bfloat16 *__restrict__ w,
                       int n, float eps, __nv_bfloat16 *__restrict__ sum_out,
                       __nv_bfloat16 *__restrict__ norm_out, uint8_t *__restrict__ q8_out) {
  extern __shared__ float s_sum[];  // [n]
  __shared__ float s_red[kNormThreads / 32];
  const int row = blockIdx.x;
  const __nv_bfloat16 *ar = a + static_cast<size_t>(row) * n;
  SI_TRACE_MARK(3, 0);
  grid_dep_wait();
  grid_dep_launch();
  SI_TRACE_MARK(3, 1);
  add_rmsnorm_row([&](int i0, float va[8]) { Load8<__nv_bfloat16>::run(ar + i0, va); }, b, c, w, n, eps, row,
                  sum_out, norm_out, q8_out, s_sum, s_red);
  SI_TRACE_MARK(3, 3);
}

// t = bf16(a + b), the separate residual-add kernel of the unfused chain.
__global__ void __launch_bounds__(256) residual_add_kernel(const __nv_bfloat16 *__restrict__ a,
                                                           const __nv_bfloat16 *__restrict__ b,
                                                           int64_t n, __nv_bfloat16 *__restrict__ t) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (8 * g >= n) return;
  float va[8], vb[8];
  Load8<__nv_bfloat16>::run(a + 8 * g, va);
  Load8<__nv_bfloat16>::run(b + 8 * g, vb);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = bf16_bits(va[2 * i] + vb[2 * i]) |
           (static_cast<uint32_t>(bf16_bits(va[2 * i + 1] + vb[2 * i + 1])) << 16);
  *reinterpret_cast<uint4 *>(t + 8 * g) = make_uint4(o[0], o[1], o[2], o[3]);
}

cudaError_t preload_norm() {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, add_rmsnorm_kernel);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, residual_add_kernel);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, quantize_q8_1_kernel<float, 1>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, quantize_q8_1_kernel<float, 4>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, quantize_q8_1_kernel<__nv_bfloat16, 1>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, quantize_q8_1_kernel<__nv_bfloat16, 4>);
  return e;
}

si_status norm_launch(const void *a, const void *b, const void *c, const void *w, int n, int rows,
                      float eps, void *sum_out, void *norm_out, void *q8_out, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(n) * sizeof(float);
  cudaError_t e = allow_smem(add_rmsnorm_kernel, smem);
  if (e != cudaSuccess) return SI_ERR_CUDA;
  e = launch_pdl(add_rmsnorm_kernel, dim3(rows), dim3(kNormThreads), smem, s,
                 static_cast<const __nv_bfloat16 *>(a), static_cast<const __nv_bfloat16 *>(b),
                 static_cast<const __nv_bfloat16 *>(c), static_cast<const __nv_bfloat16 *>(w), n,
                 eps, static_cast<__nv_bfloat16 *>(sum_out), static_cast<__nv_bfloat16 *>(norm_out),
                 static_cast<uint8_t *>(q8_out));
  return cuda_status(e);
}

}  // namespace si

using namespace si;

extern "C" si_status si_quantize_q8_1(const void *x, si_dtype x_type, int64_t n, void *y_q8_1,
                                      void *stream) {
  if (!x || !y_q8_1 || n <= 0 || n % 32 != 0) return SI_ERR_INVALID_ARG;
  if (x_type != SI_F32 && x_type != SI_BF16) return SI_ERR_UNSUPPORTED;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(y_q8_1) & 3u)) return SI_ERR_INVALID_ARG;
  // long vectors: four groups of 8 values per thread in flight; short ones
  // (up to 64 K values): one, so that a 2048-value vector is one block
  // without idle encodes
  const int U = n > 65536 ? 4 : 1;
  const int64_t chunk_blocks = kQuantThreads * U / 4;
  const int64_t chunks = (n / 32 + chunk_blocks - 1) / chunk_blocks;
  if (chunks > 0x7FFFFFFF) return SI_ERR_INVALID_ARG;
  const dim3 grid(static_cast<unsigned>(chunks));
  const int vec16 = (reinterpret_cast<uintptr_t>(y_q8_1) & 15u) == 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  uint8_t *yo = static_cast<uint8_t *>(y_q8_1);
  if (x_type == SI_F32) {
    const float *xf = static_cast<const float *>(x);
    e = U == 4 ? launch_pdl(quantize_q8_1_kernel<float, 4>, grid, dim3(kQuantThreads), 0, s, xf, n, yo, vec16)
               : launch_pdl(quantize_q8_1_kernel<float, 1>, grid, dim3(kQuantThreads), 0, s, xf, n, yo, vec16);
  } else {
    const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
    e = U == 4 ? launch_pdl(quantize_q8_1_kernel<__nv_bfloat16, 4>, grid, dim3(kQuantThreads), 0, s, xb, n, yo,
                            vec16)
               : launch_pdl(quantize_q8_1_kernel<__nv_bfloat16, 1>, grid, dim3(kQuantThreads), 0, s, xb, n, yo,
                            vec16);
  }
  return cuda_status(e);
}

extern "C" si_status si_add_rmsnorm3(const void *a, const void *b, const void *c,
                                     const void *w_norm, int n, int n_rows, float eps,
                                     void *sum_out, void *norm_out, void *norm_q8_1_out,
                                     void *stream) {
  if (!a || !b || !w_norm || !sum_out || !norm_out) return SI_ERR_INVALID_ARG;
  if (n <= 0 || n % 256 != 0 || n > 16384 || n_rows <= 0 || !(eps >= 0.f)) return SI_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || (c && !aligned16(c)) || !aligned16(w_norm) ||
      !aligned16(sum_out) || !aligned16(norm_out) ||
      (norm_q8_1_out && (reinterpret_cast<uintptr_t>(norm_q8_1_out) & 3u)))
    return SI_ERR_INVALID_ARG;
  return norm_launch(a, b, c, w_norm, n, n_rows, eps, sum_out, norm_out, norm_q8_1_out,
                     static_cast<cudaStream_t>(stream));
}

extern "C" si_status si_test_unfused_add_rmsnorm(const void *a, const void *b, const void *c,
                                                 const void *w_norm, int n, int n_rows, float eps,
                                                 void *t_scratch, void *sum_out, void *norm_out,
                                                 void *stream) {
  if (!a || !b || !c || !w_norm || !t_scratch || !sum_out || !norm_out) return SI_ERR_INVALID_ARG;
  if (n <= 0 || n % 256 != 0 || n > 16384 || n_rows <= 0) return SI_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(c) || !aligned16(w_norm) ||
      !aligned16(t_scratch) || !aligned16(sum_out) || !aligned16(norm_out))
    return SI_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t total = static_cast<int64_t>(n) * n_rows;
  cudaError_t e = launch_pdl(residual_add_kernel, dim3(static_cast<unsigned>((total / 8 + 255) / 256)),
                             dim3(256), 0, s, static_cast<const __nv_bfloat16 *>(a),
                             static_cast<const __nv_bfloat16 *>(b), total,
                             static_cast<__nv_bfloat16 *>(t_scratch));
  if (e != cudaSuccess) return SI_ERR_CUDA;
  // 2-input norm of (t, c): b == nullptr in the kernel means s = bf16(t + c).
  return norm_launch(t_scratch, nullptr, c, w_norm, n, n_rows, eps, sum_out, norm_out, nullptr, s);
}

#ifdef SI_TRACE
extern "C" int si_trace_dump_norm(void *dst) {
  return cudaMemcpyFromSymbol(dst, si::g_si_trace, sizeof(si::g_si_trace)) == cudaSuccess ? 0 : 4;
}
extern "C" int si_trace_reset_norm(void) {
  static uint64_t zeros[si::kTraceKernels * si::kTraceBlocks * si::kTracePhases];
  return cudaMemcpyToSymbol(si::g_si_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : 4;
}
#endif
