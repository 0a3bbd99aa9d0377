// noalloc.cu -- lora_backward_db_noalloc: lora_backward_db with its scratch in a
// file-scope device array instead of a caller-provided workspace, for callers
// that cannot allocate device memory (see include/lora.h).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "host_common.h"

namespace lora {

// The scratch every call uses; each device that loads the library holds it until exit.
static __device__ __align__(256) unsigned char g_db_scratch[LORA_DB_NOALLOC_SCRATCH_BYTES];

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Driver entry points (the library links the CUDA runtime statically and reaches
// the driver only through the runtime's entry-point query).
struct CtxFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};
const CtxFns &ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return f;
}

// Unique id (for the life of the process) of the context current on this thread,
// 0 when none is current yet.
lora_status_t current_ctx_id(unsigned long long *id) {
  const CtxFns &f = ctx_fns();
  if (!f.get_current || !f.get_id) return LORA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS) return LORA_ERR_CUDA;
  *id = 0;
  if (ctx != nullptr && f.get_id(ctx, id) != CUDA_SUCCESS) return LORA_ERR_CUDA;
  return LORA_OK;
}

// Device addresses of g_db_scratch, one per CUDA context that has called.  In
// host code the symbol is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress in the calling thread's current context (the primary
// context of the current device for runtime-API callers) and cached under that
// context's unique id: a context created later (after cudaDeviceReset, or by an
// engine with its own cuCtxCreate) gets its own lookup, never a stale address.
constexpr int kMaxContexts = 64;
struct Entry {
  unsigned long long id;
  void *addr;
};
Entry g_cache[kMaxContexts];
int g_ncache = 0, g_next = 0;
std::mutex g_mu;

lora_status_t scratch_address(void **out) {
  unsigned long long id = 0;
  LORA_TRY(current_ctx_id(&id));
  std::lock_guard<std::mutex> lk(g_mu);
  if (id != 0) {
    for (int i = 0; i < g_ncache; ++i)
      if (g_cache[i].id == id) {
        *out = g_cache[i].addr;
        return LORA_OK;
      }
  }
  // first call in this context (or no context current yet: the lookup below
  // initialises the runtime's primary context of the current device)
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_db_scratch) != cudaSuccess || p == nullptr) return LORA_ERR_CUDA;
  if (id == 0) LORA_TRY(current_ctx_id(&id));
  if (id != 0) {
    Entry e{id, p};
    if (g_ncache < kMaxContexts) {
      g_cache[g_ncache++] = e;
    } else {
      g_cache[g_next] = e;   // more live contexts than slots: replace in turn
      g_next = (g_next + 1) % kMaxContexts;
    }
  }
  *out = p;
  return LORA_OK;
}

}  // namespace

}  // namespace lora

extern "C" lora_status_t lora_backward_db_noalloc(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r,
                                                  const void *X, int64_t ldx, const void *A, int64_t sA_k,
                                                  int64_t sA_r, const void *dY, int64_t lddy, float scale, float *dB,
                                                  int64_t sdB_r, int64_t sdB_l, void *stream) {
  // the argument checks of lora_backward_db that do not depend on the scratch come
  // first, so that a bad dtype or size is reported as such and not as a scratch overflow
  constexpr int64_t kMaxDim = (int64_t)1 << 31;
  if (dtype != LORA_F32 && dtype != LORA_BF16) return LORA_ERR_UNSUPPORTED;
  if (M < 0 || K < 0 || L < 0 || r < 0 || M >= kMaxDim || K >= kMaxDim || L >= kMaxDim)
    return LORA_ERR_INVALID_ARG;
  if (r > LORA_MAX_RANK) return LORA_ERR_UNSUPPORTED;
  if (dtype == LORA_BF16 && (K % 8 != 0 || L % 8 != 0)) return LORA_ERR_ALIGNMENT;
  const size_t need = lora_workspace_size(LORA_OP_BACKWARD_DB, dtype, M, K, L, r, 0);
  if (need > LORA_DB_NOALLOC_SCRATCH_BYTES) return LORA_ERR_WORKSPACE;
  void *ws = nullptr;
  lora_status_t st = lora::scratch_address(&ws);
  if (st != LORA_OK) return st;
  return lora_backward_db(dtype, M, K, L, r, X, ldx, A, sA_k, sA_r, dY, lddy, scale, dB, sdB_r, sdB_l, ws,
                          LORA_DB_NOALLOC_SCRATCH_BYTES, stream);
}
