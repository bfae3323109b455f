// Expert selection helpers shared by the router and the persistent stack
// kernel: 64-bit keys whose unsigned order is the selection order (value
// descending, -0 == +0, then lower expert index first), branch-free
// max/min compare-exchange, a 32-lane shuffle bitonic sort, and the
// completion-count atomic.
#pragma once

#include "common.cuh"

namespace si {

SI_DEV uint64_t make_key(float v, int e) {
  uint32_t u = __float_as_uint(v + 0.0f);            // -0 -> +0
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);    // order-preserving map to unsigned
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(e));
}
SI_DEV float key_value(uint64_t k) {
  const uint32_t u = static_cast<uint32_t>(k >> 32);
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}
SI_DEV int key_index(uint64_t k) { return static_cast<int>(~static_cast<uint32_t>(k)); }

SI_DEV uint64_t kmax(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("max.u64 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
SI_DEV uint64_t kmin(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("min.u64 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Bitonic sort of the warp's 32 keys (one per lane) into selection order:
// lane 0 ends with the earliest key. 15 shuffle steps.
SI_DEV uint64_t warp_sort32(uint64_t key, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, key, stride);
      const bool lower = (lane & stride) == 0;
      const bool desc = (lane & size) == 0 || size == 32;
      key = (lower == desc) ? kmax(key, other) : kmin(key, other);
    }
  }
  return key;
}

SI_DEV uint32_t atom_inc_acq_rel(uint32_t *p, uint32_t bound) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(bound)
               : "memory");
  return old;
}

}  // namespace si
