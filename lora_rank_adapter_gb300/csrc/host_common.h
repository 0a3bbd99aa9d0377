// host_common.h -- host-side helpers of liblora.so: status plumbing, tensor-map
// encoding through the driver entry point, launch configuration and workspace
// carving.  No device code here.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/lora.h"

namespace lora {

#define LORA_TRY(expr)                          \
  do {                                          \
    lora_status_t st_ = (expr);                 \
    if (st_ != LORA_OK) return st_;             \
  } while (0)

#define LORA_CUDA(expr)                         \
  do {                                          \
    cudaError_t e_ = (expr);                    \
    if (e_ != cudaSuccess) return LORA_ERR_CUDA; \
  } while (0)

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Padded rank bucket of the bf16 kernels: 16, 32, 64 or 128.
inline int rank_bucket(int r) { return r <= 16 ? 16 : r <= 32 ? 32 : r <= 64 ? 64 : 128; }

// Encodes a 2-D/3-D bf16 or fp32 tiled tensor map.  dims/strides in elements
// (strides of dims 1.. in elements of the innermost type).  Returns false if
// the driver rejects it.
// `promo` is the L2 sector promotion of the copies (256-byte lines for dense
// streams; none for strided reads that use a few bytes of each row).
bool encode_tmap(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base, const uint64_t *dims,
                 const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swz,
                 CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);

// SM count of the current device, and resident blocks per SM of a kernel
// (both cached per device).
int num_sms();
int occupancy(const void *kernel, int threads, size_t smem);

// Simple bump allocator over the caller's workspace.
struct WsCarver {
  char *base;
  size_t size, used = 0;
  WsCarver(void *b, size_t s) : base(static_cast<char *>(b)), size(s) {}
  void *take(size_t bytes) {
    size_t off = (used + 255) & ~size_t(255);
    if (base == nullptr || off + bytes > size) return nullptr;
    used = off + bytes;
    return base + off;
  }
};
inline size_t ws_round(size_t b) { return (b + 255) & ~size_t(255); }

// Counts every kernel launch issued through launch() (lora_kernel_launches()).
void count_launch();

// Launch with optional cluster dimension and programmatic dependent launch.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster,
                   bool pdl, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  if (cluster > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = cluster;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Sets the dynamic shared-memory limit of `kernel` once per device.
cudaError_t ensure_smem(const void *kernel, size_t bytes);

}  // namespace lora
