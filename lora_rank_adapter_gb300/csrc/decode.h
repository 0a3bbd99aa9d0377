// decode.h -- arguments and launcher of the decode-batch shrink of decode.cu
// (tiles of at most four tokens of one slot, on CUDA cores fed by TMA).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "multi.h"

namespace lora {

constexpr int kDecTokens = 4;     // tokens per tile of a decode batch
constexpr int kMaxDecGrid = 160;  // CTAs of the persistent grid (one per SM; more than any GB300 has)

struct DecArgs {
  const int32_t *ranks;
  const int *header;          // [0] active tokens, [1] tiles, [2] sum over the tiles of round8(rank)
  const int4 *tiles;          // (slot, start, len, sum of round8(rank) over the tiles before)
  const int32_t *perm;        // active tokens ordered by (slot, token)
  int S, R, n, T;
  int nk;                     // 256-column chunks of `in`
  float *h;                   // out: fp32 [T][ldh]
  int64_t ldh;
  float *part;                // partial sums [2 per CTA][4 tokens][n * round8(R)]
  int *counters;              // [tiles] tickets, zero before the launch
  int a_one_slot;             // the stack has one slot (slot stride 0)
};

// Bytes of shrink partial sums for n slices of rank R.
size_t dec_part_bytes(int n, int R);
lora_status_t shrink_dec_launch(const DecArgs &args, const MultiArgs &m, int64_t T, cudaStream_t st);

struct DecExpMaps {
  CUtensorMap y[LORA_MAX_SLICES];      // y columns of each slice
  CUtensorMap b[LORA_MAX_SLICES][4];   // b rows of each slice: boxes of 8, 16, 32, 64 rank entries
};
// The expand of decode batches: y[t, off_i + c] += scal[slot] * h[t, slice i] . b[slot][off_i + c].
struct DecExpArgs {
  const int32_t *ranks;
  const float *scal;
  const int *header;          // as DecArgs
  const int4 *tiles;
  const int32_t *perm;
  int S, R, n, T;
  const float *h;
  int64_t ldh;
  int nbu;                              // 256-column blocks of a tile over all slices
  int blk0[LORA_MAX_SLICES + 1];        // first block of each slice
  int b_one_slot;                       // the stack b has one slot (slot stride 0)
  int bw;                               // cost of a unit's b rows, in 512-byte units
};
// Returns LORA_ERR_ALIGNMENT when y or b cannot be read through tensor maps and
// LORA_ERR_UNSUPPORTED when a 256-column unit of rank R does not fit a stage
// (R > 72); the caller then runs the plain-load expand.
lora_status_t expand_dec_launch(const DecExpArgs &args, const MultiArgs &m, int64_t T, cudaStream_t st);
int read_clear_error_decode();

}  // namespace lora
