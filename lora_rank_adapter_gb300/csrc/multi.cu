// multi.cu -- multi-adapter serving ops (placeholder until the segmented kernels land).
#include "common.cuh"
#include "host_common.h"
#include "multi.h"

namespace lora {

size_t multi_ws_bytes(int, int64_t, int64_t, int64_t, int, int) { return 0; }
lora_status_t group_by_slot(const lora_addressing_t &, const int32_t *, int32_t *, int32_t *, int32_t *, void *,
                            size_t, cudaStream_t) { return LORA_ERR_UNSUPPORTED; }
lora_status_t shrink(MultiArgs, void *, size_t, cudaStream_t) { return LORA_ERR_UNSUPPORTED; }
lora_status_t expand(MultiArgs, void *, size_t, cudaStream_t) { return LORA_ERR_UNSUPPORTED; }
lora_status_t apply_linear(MultiArgs, void *, size_t, cudaStream_t) { return LORA_ERR_UNSUPPORTED; }
lora_status_t gather_shrink(MultiArgs, cudaStream_t) { return LORA_ERR_UNSUPPORTED; }
int read_clear_error_multi() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
  return v;
}

}  // namespace lora
