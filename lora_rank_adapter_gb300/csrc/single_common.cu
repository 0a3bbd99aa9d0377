// single_common.cu -- operand layout of the single-adapter ops: which of A / B
// are read in place and which are repacked into the workspace, and the repack
// kernel itself.
//
// The kernels read the small operands in fixed layouts: A as Ac[j][k] (k
// contiguous; PEFT's lora_A.weight) and B as Bc[l][j] (j contiguous; PEFT's
// lora_B.weight), with 16-byte rows.  Other strides are repacked first.
#include <algorithm>

#include "common.cuh"
#include "host_common.h"
#include "single_common.h"

namespace lora {

// Strided [rows][cols] bf16 gather into a dense [rows][ldd] buffer.
__global__ void pack2d_bf16_kernel(const __nv_bfloat16 *src, int64_t s_row, int64_t s_col, int rows, int cols,
                                   __nv_bfloat16 *dst, int64_t ldd) {
  pdl_wait();
  const int64_t n = (int64_t)rows * cols;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = e / cols, j = e % cols;
    dst[i * ldd + j] = src[i * s_row + j * s_col];
  }
  pdl_launch_dependents();
}

// ----------------------------------------------------------------------------- host side
lora_status_t pack_bf16_2d(const void *src, int64_t s_row, int64_t s_col, int64_t rows, int64_t cols, void *dst,
                           int64_t ldd, cudaStream_t st) {
  const int64_t n = rows * cols;
  int blocks = (int)std::min<int64_t>(ceil_div(n, 256), 4 * num_sms());
  if (blocks < 1) blocks = 1;
  LORA_CUDA(launch(pack2d_bf16_kernel, dim3(blocks), dim3(256), 0, st, 1, true, (const __nv_bfloat16 *)src, s_row,
                   s_col, (int)rows, (int)cols, (__nv_bfloat16 *)dst, ldd));
  return LORA_OK;
}

SingleLayout plan_layout(const SingleArgs &a, bool need_A, bool need_B) {
  SingleLayout lay;
  lay.pack_A = need_A && !(a.sA_k == 1 && (a.sA_r * 2) % 16 == 0 && a.sA_r >= a.K && aligned16(a.A));
  lay.pack_B = need_B && !(a.sB_r == 1 && (a.sB_l * 2) % 16 == 0 && a.sB_l >= a.r && aligned16(a.B));
  lay.lda = lay.pack_A ? round_up(a.K, 8) : a.sA_r;
  lay.ldb = lay.pack_B ? round_up(a.r, 8) : a.sB_l;
  return lay;
}

int read_clear_error_single_common() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
  return v;
}

}  // namespace lora
