// multi.h -- argument struct and launchers of the multi-adapter (serving) ops.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/lora.h"

namespace lora {

struct MultiArgs {
  lora_addressing_t addr;
  const int32_t *ranks;
  const float *scalings;
  int32_t n;                             // num_slices
  int32_t out_slices[LORA_MAX_SLICES];   // host copy
  int64_t O;                             // sum of out_slices
  int64_t in;                            // contraction length (V for gather_shrink)
  const void *x; int64_t ldx;
  const void *a; int64_t sa_slot, sa_row, sa_col;
  const void *b; int64_t sb_slot, sb_row, sb_col;
  float *h; int64_t ldh;                 // shrink output, expand input
  void *y; int64_t ldy;
  const int64_t *ids;
};

size_t multi_ws_bytes(int op, int64_t T, int64_t in, int64_t O, int R, int S);
size_t schedule_bytes(int64_t T, int S);
lora_status_t build_schedule(const lora_addressing_t &addr, const int32_t *ranks, void *sched, size_t bytes,
                             cudaStream_t st);

lora_status_t group_by_slot(const lora_addressing_t &addr, const int32_t *ranks, int32_t *counts, int32_t *perm,
                            int32_t *num_active, void *ws, size_t ws_bytes, cudaStream_t st);
lora_status_t shrink(MultiArgs m, void *ws, size_t ws_bytes, cudaStream_t st);
lora_status_t expand(MultiArgs m, void *ws, size_t ws_bytes, cudaStream_t st);
lora_status_t apply_linear(MultiArgs m, void *ws, size_t ws_bytes, cudaStream_t st);
lora_status_t gather_shrink(MultiArgs m, cudaStream_t st);

int read_clear_error_multi();

}  // namespace lora
