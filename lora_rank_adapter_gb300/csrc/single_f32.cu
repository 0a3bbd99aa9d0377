// single_f32.cu -- single-adapter LoRA kernels in fp32 (CUDA-core FMA), for
// sm_103a.  The fp32 workload of the benchmark is small (256 x 512 x 512, r = 8)
// and launch-bound; these kernels favour a fixed, deterministic summation order
// (warp-shuffle trees) over throughput.  Operations as in the NeMo AutoModel API
// page "nemo_automodel.components._peft.lora_kernel": lora_forward_kernel,
// lora_da_dx_kernel / lora_da_dx_update_wrapper, lora_db_kernel /
// lora_db_update_wrapper, in forward roles X (M x K), A (K x r), B (r x L).
#include <algorithm>

#include "common.cuh"
#include "host_common.h"
#include "single_common.h"

namespace lora {

constexpr int kF32Rows = 2;   // rows per block of the forward (more blocks in flight)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Y += s * (X*A)*B for 16 rows per block; h kept in shared memory.
__global__ void __launch_bounds__(256) fwd_f32_kernel(SingleArgs a) {
  __shared__ float h[kF32Rows * LORA_MAX_RANK];
  pdl_wait();
  const float *X = (const float *)a.X, *A = (const float *)a.A, *B = (const float *)a.B;
  float *Y = (float *)a.Y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int64_t m0 = (int64_t)blockIdx.x * kF32Rows;
  for (int pr = warp; pr < kF32Rows * a.r; pr += nw) {
    const int row = pr / a.r, j = pr % a.r;
    const int64_t m = m0 + row;
    // four independent partial sums per lane keep four loads in flight
    float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
    if (m < a.M) {
      const float *xr = X + m * a.ldx, *ac = A + j * a.sA_r;
      int64_t k = lane;
      for (; k + 96 < a.K; k += 128) {
        p0 += xr[k] * ac[k * a.sA_k];
        p1 += xr[k + 32] * ac[(k + 32) * a.sA_k];
        p2 += xr[k + 64] * ac[(k + 64) * a.sA_k];
        p3 += xr[k + 96] * ac[(k + 96) * a.sA_k];
      }
      for (; k < a.K; k += 32) p0 += xr[k] * ac[k * a.sA_k];
    }
    const float acc = warp_sum((p0 + p1) + (p2 + p3));
    if (lane == 0) {
      h[row * a.r + j] = acc;
      if (a.h != nullptr && m < a.M) a.h[m * a.ldh + j] = acc;   // lora_forward_h
    }
  }
  __syncthreads();
  for (int row = 0; row < kF32Rows; ++row) {
    const int64_t m = m0 + row;
    if (m >= a.M) break;
    for (int64_t l = threadIdx.x; l < a.L; l += blockDim.x) {
      float acc = 0.f;
      for (int j = 0; j < a.r; ++j) acc += h[row * a.r + j] * B[j * a.sB_r + l * a.sB_l];
      Y[m * a.ldy + l] += a.scale * acc;
    }
  }
  pdl_launch_dependents();
}

// out[m][j] = sum_c In[m][c] * W(c, j)   (W(c, j) = W[c*sw_c + j*sw_j]); one warp per (m, j)
__global__ void __launch_bounds__(256) rowdot_f32_kernel(const float *In, int64_t ld_in, int64_t M, int64_t C,
                                                         const float *W, int64_t sw_c, int64_t sw_j, int r,
                                                         float *out) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t pr = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); pr < M * r; pr += nwarps) {
    const int64_t m = pr / r;
    const int j = (int)(pr % r);
    float acc = 0.f;
    for (int64_t c = lane; c < C; c += 32) acc += In[m * ld_in + c] * W[c * sw_c + j * sw_j];
    acc = warp_sum(acc);
    if (lane == 0) out[m * r + j] = acc;
  }
  pdl_launch_dependents();
}

// dX[m][k] = s * sum_j dyb[m][j] * A(k, j); one thread per element
__global__ void __launch_bounds__(256) dx_f32_kernel(SingleArgs a, const float *dyb) {
  pdl_wait();
  const float *A = (const float *)a.A;
  float *dX = (float *)a.dX;
  const int64_t n = a.M * a.K;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = e / a.K, k = e % a.K;
    float acc = 0.f;
    for (int j = 0; j < a.r; ++j) acc += dyb[m * a.r + j] * A[k * a.sA_k + j * a.sA_r];
    const float v = a.scale * acc;
    dX[m * a.lddx + k] = a.dx_acc ? dX[m * a.lddx + k] + v : v;
  }
  pdl_launch_dependents();
}

// out(p, q) = s * sum_m U[m*su_m + p*su_p] * V[m][q]  (V row-major, ld_v); one warp per (p, q)
__global__ void __launch_bounds__(256) coldot_f32_kernel(const float *U, int64_t su_m, int64_t su_p, int64_t P,
                                                         const float *V, int64_t ld_v, int64_t Q, int64_t M,
                                                         float s, float *out, int64_t so_p, int64_t so_q) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t pr = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); pr < P * Q; pr += nwarps) {
    const int64_t p = pr / Q, q = pr % Q;
    float acc = 0.f;
    for (int64_t m = lane; m < M; m += 32) acc += U[m * su_m + p * su_p] * V[m * ld_v + q];
    acc = warp_sum(acc);
    if (lane == 0) out[p * so_p + q * so_q] = s * acc;
  }
  pdl_launch_dependents();
}

template <typename T>
__global__ void fill_zero_kernel(T *p, int64_t rows, int64_t cols, int64_t s_row, int64_t s_col) {
  pdl_wait();
  const int64_t n = rows * cols;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x)
    p[(e / cols) * s_row + (e % cols) * s_col] = T(0.f);
  pdl_launch_dependents();
}

static unsigned grid_for(int64_t units, int per_block) {
  int64_t b = ceil_div(units, per_block);
  b = std::min<int64_t>(std::max<int64_t>(b, 1), 8 * (int64_t)num_sms());
  return (unsigned)b;
}

lora_status_t fill_zero_2d(lora_dtype_t dt, void *p, int64_t rows, int64_t cols, int64_t s_row, int64_t s_col,
                           cudaStream_t st) {
  if (rows <= 0 || cols <= 0) return LORA_OK;
  if (dt == LORA_BF16)
    LORA_CUDA(launch(fill_zero_kernel<__nv_bfloat16>, dim3(grid_for(rows * cols, 256)), dim3(256), 0, st, 1, true,
                     (__nv_bfloat16 *)p, rows, cols, s_row, s_col));
  else
    LORA_CUDA(launch(fill_zero_kernel<float>, dim3(grid_for(rows * cols, 256)), dim3(256), 0, st, 1, true,
                     (float *)p, rows, cols, s_row, s_col));
  return LORA_OK;
}

size_t f32_ws_bytes(int op, int64_t M, int64_t K, int64_t L, int r) {
  (void)K;
  (void)L;
  if (M <= 0 || r <= 0) return 0;
  if (op == LORA_OP_BACKWARD_DX_DA || op == LORA_OP_BACKWARD_DB || op == LORA_OP_BACKWARD)
    return ws_round((size_t)M * r * 4);
  return 0;
}

lora_status_t forward_f32(const SingleArgs &a, cudaStream_t st) {
  LORA_CUDA(launch(fwd_f32_kernel, dim3((unsigned)ceil_div(a.M, kF32Rows)), dim3(256), 0, st, 1, true, a));
  return LORA_OK;
}

lora_status_t backward_dx_da_f32(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  WsCarver carver(ws, ws_bytes);
  float *dyb = (float *)carver.take((size_t)a.M * a.r * 4);
  if (!dyb) return LORA_ERR_WORKSPACE;
  // dyb[m][j] = sum_l dY[m][l] * B(j, l)
  LORA_CUDA(launch(rowdot_f32_kernel, dim3(grid_for(a.M * a.r, 8)), dim3(256), 0, st, 1, true,
                   (const float *)a.dY, a.lddy, a.M, a.L, (const float *)a.B, a.sB_l, a.sB_r, a.r, dyb));
  LORA_CUDA(launch(dx_f32_kernel, dim3(grid_for(a.M * a.K, 256)), dim3(256), 0, st, 1, true, a,
                   (const float *)dyb));
  // dA(k, j) = s * sum_m X[m][k] * dyb[m][j]
  LORA_CUDA(launch(coldot_f32_kernel, dim3(grid_for(a.K * a.r, 8)), dim3(256), 0, st, 1, true,
                   (const float *)a.X, a.ldx, (int64_t)1, a.K, (const float *)dyb, (int64_t)a.r, (int64_t)a.r, a.M,
                   a.scale, a.dA, a.sdA_k, a.sdA_r));
  return LORA_OK;
}

lora_status_t backward_db_f32(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  WsCarver carver(ws, ws_bytes);
  float *h = (float *)carver.take((size_t)a.M * a.r * 4);
  if (!h) return LORA_ERR_WORKSPACE;
  // h[m][j] = sum_k X[m][k] * A(k, j)
  LORA_CUDA(launch(rowdot_f32_kernel, dim3(grid_for(a.M * a.r, 8)), dim3(256), 0, st, 1, true,
                   (const float *)a.X, a.ldx, a.M, a.K, (const float *)a.A, a.sA_k, a.sA_r, a.r, h));
  // dB(j, l) = s * sum_m h[m][j] * dY[m][l]
  LORA_CUDA(launch(coldot_f32_kernel, dim3(grid_for((int64_t)a.r * a.L, 8)), dim3(256), 0, st, 1, true,
                   (const float *)h, (int64_t)a.r, (int64_t)1, (int64_t)a.r, (const float *)a.dY, a.lddy, a.L, a.M,
                   a.scale, a.dB, a.sdB_r, a.sdB_l));
  return LORA_OK;
}

// lora_backward: dX and dA as lora_backward_dx_da, dB from the saved h.
lora_status_t backward_f32(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  LORA_TRY(backward_dx_da_f32(a, ws, ws_bytes, st));
  // dB(j, l) = s * sum_m h[m][j] * dY[m][l]
  LORA_CUDA(launch(coldot_f32_kernel, dim3(grid_for((int64_t)a.r * a.L, 8)), dim3(256), 0, st, 1, true,
                   (const float *)a.h, a.ldh, (int64_t)1, (int64_t)a.r, (const float *)a.dY, a.lddy, a.L, a.M,
                   a.scale, a.dB, a.sdB_r, a.sdB_l));
  return LORA_OK;
}

int read_clear_error_single_f32() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
  return v;
}

}  // namespace lora
