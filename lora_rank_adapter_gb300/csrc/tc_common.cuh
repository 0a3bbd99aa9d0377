// tc_common.cuh -- pieces shared by the tensor-core (tcgen05) kernels: the
// stream-K split of work units over a persistent grid, warp-wide bounded
// waits, and the per-CTA slots of stream-K partial sums.
#pragma once

#include "common.cuh"

namespace lora {

// Units [0, U) are dealt to G CTAs in contiguous runs: CTA i takes [sk_begin(i), sk_begin(i + 1)).
__host__ __device__ __forceinline__ int64_t sk_begin(int64_t U, int G, int i) { return U * i / G; }
// The CTA whose run holds unit u.
__host__ __device__ __forceinline__ int sk_cta(int64_t U, int G, int64_t u) {
  int i = (int)(u * G / U);
  while (i + 1 < G && sk_begin(U, G, i + 1) <= u) ++i;
  while (i > 0 && sk_begin(U, G, i) > u) --i;
  return i;
}
// Partial sums live per CTA: a CTA's run meets a group of n units that it does
// not cover whole only as its first group (slot 0) or its last group (slot 1).
__host__ __device__ __forceinline__ int64_t part_slot(int64_t U, int G, int c, int64_t g, int64_t n) {
  return 2 * (int64_t)c + (sk_begin(U, G, c) / n == g ? 0 : 1);
}

__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// Every lane waits (bounded); true when all lanes saw the phase complete.
__device__ __forceinline__ bool wait_warp(uint64_t *bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

}  // namespace lora
