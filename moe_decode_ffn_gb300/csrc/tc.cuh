// tcgen05 (5th-generation tensor core) helpers for sm_103a: tensor-memory
// allocation, shared-memory matrix descriptors, kind::f16 MMA, commit to an
// mbarrier and tensor-memory loads. Inline PTX only.
#pragma once

#include "common.cuh"

namespace si {

// Shared-memory matrix descriptor, K-major, no swizzle. The operand is stored
// as 8-row x 16-byte "core matrices" of 128 contiguous bytes; `lbo` is the
// byte distance between core matrices adjacent along K, `sbo` between 8-row
// groups. Bits: [0,14) start >> 4, [16,30) lbo >> 4, [32,46) sbo >> 4,
// [46,48) descriptor version 1, [61,64) layout 0 (no swizzle).
SI_DEV uint64_t umma_desc_kmajor(uint32_t smem_byte_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_byte_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M x N.
// Bits: [4,6) D format (1 = f32), [7,10) A format (0 = f16), [10,13) B format
// (0 = f16), 15/16 A/B major (0 = K), [17,23) N >> 3, [24,29) M >> 4.
SI_DEV uint32_t umma_idesc_f16_f32(int m, int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Byte offset of element (row, k) of a K-major no-swizzle fp16 tile whose
// rows are `kdim` elements long (kdim a multiple of 8): core matrix
// (row / 8, k / 8) at ((row / 8) * (kdim / 8) + k / 8) * 128, then row % 8 at
// 16 bytes and k % 8 at 2 bytes. So lbo = 128 and sbo = kdim * 16.
SI_DEV uint32_t kmajor_offset(int row, int k, int kdim) {
  return static_cast<uint32_t>(((row >> 3) * (kdim >> 3) + (k >> 3)) * 128 + (row & 7) * 16 +
                               (k & 7) * 2);
}

SI_DEV void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
SI_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
SI_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
SI_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SI_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
SI_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, one thread.
SI_DEV void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                     uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every MMA issued so far by this thread has completed.
SI_DEV void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 8 consecutive fp32 columns of this warp's 32 TMEM lanes (one row per thread).
SI_DEV void tmem_ld8(uint32_t taddr, float v[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

SI_DEV uint32_t pack_half2(float a, float b) {
  return static_cast<uint32_t>(float_to_half_bits(a)) |
         (static_cast<uint32_t>(float_to_half_bits(b)) << 16);
}

}  // namespace si
