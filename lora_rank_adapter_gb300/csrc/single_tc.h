// single_tc.h -- arguments of the tensor-core (tcgen05) single-adapter kernels
// and their host entry points.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "single_common.h"

namespace lora {

// rows_kernel: out[m, :] = In[m, :] * W for 128-row blocks, stream-K over
// (row block, 64-column chunk) units.
struct TcRowsArgs {
  int M, C, r, nc;           // rows, contraction length, rank, 64-column chunks
  int64_t U;                 // units = row blocks * nc
  int G;                     // grid
  float *part;               // partial sums [2 per CTA][128][RP]
  int *counters;             // [row block], zero before the launch
  uint8_t *blob;             // out: hi / lo bf16 tiles per row block
  float *hout;               // out (optional): fp32 rows [M][ldh], columns < r
  int64_t ldh;
  int h_vec4;                // hout rows written as float4 (16-byte aligned rows, r % 4 == 0)
  const float *hin;          // in (optional): a saved fp32 h [M][ldhin], converted
  int64_t ldhin;             //   to a blob at hblob by the epilogue warps before
  uint8_t *hblob;            //   their first block (one 128-row block per CTA in turn)
};

// col_kernel: acc[c, :] = sum_m In[m, c] * blob[m, :] for 128-column blocks,
// stream-K over (column block, 128-row tile) units; optionally the dX tiles.
struct TcColArgs {
  int M, C, r, nt;           // rows, columns of In, rank, 128-row tiles
  int64_t U;
  int G;
  float *part;               // [2 per CTA][128][RP]
  int *counters;             // [column block], zero before the launch
  const uint8_t *blob;       // hi / lo tiles per row tile
  float scale;               // dX = scale * blob * A^T
  float out_scale;           // out = out_scale * acc
  void *out;                 // out(c, j) at out[c * out_sc + j * out_sj], fp32 or bf16
  int64_t out_sc, out_sj;
  int out_bf16;
  int out_vec4;              // fp32 output rows contiguous (out_sj = 1) and 16-byte aligned
  int wait_first;            // wait for the previous launch at the start (else only before exiting)
  __nv_bfloat16 *dX;         // dX [M][lddx] (kDX)
  int64_t lddx;
};

// expand_kernel: Y += scale * h * B over (row block, 64-column chunk) units.
struct TcExpArgs {
  int M, L, nl;
  int64_t U;
  int64_t Us;                // units [0, Us) dealt evenly, [Us, U) claimed CH at a time
  int CH;
  int *next;                 // claim counter (zeroed before the launch), or null: no shared tail
  int G;
  const uint8_t *blob;       // hi / lo tiles of h per row block
  __nv_bfloat16 *Y;
  int64_t ldy;
  float scale;
};

size_t tc_ws_bytes(int op, int64_t M, int64_t K, int64_t L, int r);
lora_status_t forward_tc(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st);
lora_status_t backward_dx_da_tc(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st);
lora_status_t backward_db_tc(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st);
lora_status_t backward_tc(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st);
int read_clear_error_single_tc();

}  // namespace lora
