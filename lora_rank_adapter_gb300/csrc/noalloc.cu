// noalloc.cu -- lora_backward_db_noalloc: lora_backward_db with its scratch in a
// file-scope device array instead of a caller-provided workspace, for callers
// that cannot allocate device memory (see include/lora.h).
#include <cuda_runtime.h>

#include <mutex>

#include "host_common.h"

namespace lora {

// The scratch every call uses; each device that loads the library holds it until exit.
static __device__ __align__(256) unsigned char g_db_scratch[LORA_DB_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_db_scratch on the current device.  In host code the
// symbol is only a host-side stand-in, so the address is looked up once per
// device, with that device current, and cached.
lora_status_t scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LORA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_db_scratch) != cudaSuccess || p == nullptr) return LORA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LORA_OK;
}
}  // namespace

}  // namespace lora

extern "C" lora_status_t lora_backward_db_noalloc(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r,
                                                  const void *X, int64_t ldx, const void *A, int64_t sA_k,
                                                  int64_t sA_r, const void *dY, int64_t lddy, float scale, float *dB,
                                                  int64_t sdB_r, int64_t sdB_l, void *stream) {
  const size_t need = lora_workspace_size(LORA_OP_BACKWARD_DB, dtype, M, K, L, r, 0);
  if (need > LORA_DB_NOALLOC_SCRATCH_BYTES) return LORA_ERR_WORKSPACE;
  void *ws = nullptr;
  lora_status_t st = lora::scratch_address(&ws);
  if (st != LORA_OK) return st;
  return lora_backward_db(dtype, M, K, L, r, X, ldx, A, sA_k, sA_r, dY, lddy, scale, dB, sdB_r, sdB_l, ws,
                          LORA_DB_NOALLOC_SCRATCH_BYTES, stream);
}
