// multi_tc.h -- arguments and launcher of the stream-K tensor-core shrink of
// multi_tc.cu (decode-shaped batches).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "multi.h"

namespace lora {

constexpr int kMaxTcGrid = 160;   // CTAs of the persistent grid (one per SM; more than any GB300 has)

struct MtArgs {
  const int32_t *ranks;
  const float *scal;
  const int *header;          // [1] = number of tiles
  const int4 *tiles;          // (slot, start, len, 0), at most 128 tokens of one slot
  const int32_t *perm;        // active tokens ordered by (slot, token)
  int S, R, n, T;
  int in, nk;                 // contraction length and its 64-column chunks
  int ncm;                    // columns of a partial: n * max(16, round16(R))
  float *h;                   // out: fp32 [T][ldh]
  int64_t ldh;
  float *part;                // partial sums [2 per CTA][ncm columns][128 rows]
  int *counters;              // [tiles] tickets, zero before the launch
  int a_one_slot;             // the stack has one slot (slot stride 0)
};

// Bytes of shrink partial sums for n slices of rank R.
size_t multi_tc_part_bytes(int n, int R);
lora_status_t shrink_tc_launch(const MtArgs &args, const MultiArgs &m, int64_t T, cudaStream_t st);
int read_clear_error_multi_tc();

}  // namespace lora
