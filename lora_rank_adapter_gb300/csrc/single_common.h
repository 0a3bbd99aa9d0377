// single_common.h -- argument structs and helpers shared by the single-adapter
// kernels and the C ABI layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/lora.h"

namespace lora {

// Validated arguments of one single-adapter call (forward roles, strides in elements).
struct SingleArgs {
  lora_dtype_t dtype;
  int64_t M, K, L;
  int r;
  const void *X; int64_t ldx;
  const void *A; int64_t sA_k, sA_r;
  const void *B; int64_t sB_r, sB_l;
  void *Y; int64_t ldy;
  const void *dY; int64_t lddy;
  void *dX; int64_t lddx;
  float *dA; int64_t sdA_k, sdA_r;
  float *dB; int64_t sdB_r, sdB_l;
  float scale;
  float *h; int64_t ldh;      // forward: optional h = X * A out; backward: the saved h in
  int dx_acc = 0;             // backward: dX += the update (else dX = the update)
  int grad_lo = 0;            // backward: dA and dB in the input dtype (bf16), else fp32
};

// Whether A / B are repacked into the workspace, and the row strides used.
struct SingleLayout {
  bool pack_A = false, pack_B = false;
  int64_t lda = 0, ldb = 0;
};

SingleLayout plan_layout(const SingleArgs &a, bool need_A, bool need_B);
size_t f32_ws_bytes(int op, int64_t M, int64_t K, int64_t L, int r);

lora_status_t forward_f32(const SingleArgs &a, cudaStream_t st);
lora_status_t backward_dx_da_f32(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st);
lora_status_t backward_db_f32(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st);
lora_status_t backward_f32(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st);

// Strided 2-D bf16 copy into a dense [rows][ldd] layout (repacking A or B).
lora_status_t pack_bf16_2d(const void *src, int64_t s_row, int64_t s_col, int64_t rows, int64_t cols, void *dst,
                           int64_t ldd, cudaStream_t st);

// Zero fills used for degenerate shapes (outputs defined as overwritten).
lora_status_t fill_zero_2d(lora_dtype_t dt, void *p, int64_t rows, int64_t cols, int64_t s_row, int64_t s_col,
                           cudaStream_t st);

int read_clear_error_single_common();
int read_clear_error_single_f32();

}  // namespace lora
