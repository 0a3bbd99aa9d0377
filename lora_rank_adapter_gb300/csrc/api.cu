// api.cu -- the extern "C" entry points of liblora.so (declared in include/lora.h):
// argument validation, workspace sizing and dispatch to the sm_103a kernels,
// plus the host helpers shared by all translation units (tensor-map encoding
// through the driver entry point, SM count, occupancy, shared-memory limits).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "host_common.h"
#include "multi.h"
#include "single_common.h"
#include "single_tc.h"
#include "decode.h"

namespace lora {

// ----------------------------------------------------------------------------- host helpers
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode_tmap(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base, const uint64_t *dims,
                 const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swz,
                 CUtensorMapL2promotion promo) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  CUresult r = fn(map, dt, (cuuint32_t)rank, const_cast<void *>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static std::mutex g_mu;
static std::atomic<uint64_t> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int num_sms() {
  static std::map<int, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  cache[dev] = n;
  return n;
}

int occupancy(const void *kernel, int threads, size_t smem) {
  static std::map<std::pair<const void *, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = cache.find({kernel, dev});
    if (it != cache.end()) return it->second;
  }
  int occ = 0;
  if (ensure_smem(kernel, smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem) != cudaSuccess || occ < 1)
    occ = 1;
  std::lock_guard<std::mutex> lk(g_mu);
  cache[{kernel, dev}] = occ;
  return occ;
}

cudaError_t ensure_smem(const void *kernel, size_t bytes) {
  static std::map<std::pair<const void *, int>, size_t> done;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = done.find({kernel, dev});
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done[{kernel, dev}] = bytes;
  return e;
}

// ----------------------------------------------------------------------------- validation
static constexpr int64_t kMaxDim = (int64_t)1 << 31;

static bool size_ok(int64_t v) { return v >= 0 && v < kMaxDim; }

// Big row-major operand: rows x cols with row stride ld (elements of size e).
static lora_status_t check_big(const void *p, int64_t rows, int64_t cols, int64_t ld, int e) {
  if (rows == 0 || cols == 0) return LORA_OK;
  if (p == nullptr) return LORA_ERR_INVALID_ARG;
  if (ld < cols) return LORA_ERR_INVALID_ARG;
  if (!aligned16(p) || (ld * e) % 16 != 0) return LORA_ERR_ALIGNMENT;
  return LORA_OK;
}

static lora_status_t check_ws(void *ws, size_t ws_bytes, size_t need) {
  if (need == 0) return LORA_OK;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < need) return LORA_ERR_WORKSPACE;
  return LORA_OK;
}

static lora_status_t check_single_common(lora_dtype_t dt, int64_t M, int64_t K, int64_t L, int32_t r) {
  if (dt != LORA_F32 && dt != LORA_BF16) return LORA_ERR_UNSUPPORTED;
  if (!size_ok(M) || !size_ok(K) || !size_ok(L) || r < 0) return LORA_ERR_INVALID_ARG;
  if (r > LORA_MAX_RANK) return LORA_ERR_UNSUPPORTED;
  // bf16 Y and dX rows go out by tensor-copy stores, which write whole 16-byte
  // pieces: a row ending inside one would have its neighbour elements rewritten
  if (dt == LORA_BF16 && (K % 8 != 0 || L % 8 != 0)) return LORA_ERR_ALIGNMENT;
  return LORA_OK;
}

static size_t single_ws(int op, lora_dtype_t dt, int64_t M, int64_t K, int64_t L, int r) {
  return dt == LORA_BF16 ? tc_ws_bytes(op, M, K, L, r) : f32_ws_bytes(op, M, K, L, r);
}

// Workspace the call will actually use (packing only when a layout needs it).
static size_t single_ws_needed(int op, const SingleArgs &a) {
  if (a.dtype != LORA_BF16) return f32_ws_bytes(op, a.M, a.K, a.L, a.r);
  return tc_ws_bytes(op, a.M, a.K, a.L, a.r);
}

}  // namespace lora

using namespace lora;

extern "C" {

const char *lora_version(void) { return "lora-gb300 0.1 (sm_103a)"; }

uint64_t lora_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char *lora_status_string(lora_status_t s) {
  switch (s) {
    case LORA_OK: return "LORA_OK";
    case LORA_ERR_INVALID_ARG: return "LORA_ERR_INVALID_ARG: null pointer, negative size or inconsistent arguments";
    case LORA_ERR_UNSUPPORTED: return "LORA_ERR_UNSUPPORTED: beyond the compiled limits (rank, slices, slots, dtype)";
    case LORA_ERR_ALIGNMENT:
      return "LORA_ERR_ALIGNMENT: big operand not 16-byte aligned, row stride not 16-byte, or a bf16 extent not "
             "a multiple of 8";
    case LORA_ERR_WORKSPACE: return "LORA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case LORA_ERR_CUDA: return "LORA_ERR_CUDA: a CUDA call or kernel launch failed";
    case LORA_ERR_DEVICE: return "LORA_ERR_DEVICE: a kernel flagged a device-side error";
  }
  return "unknown lora_status_t";
}

size_t lora_workspace_size(lora_op_t op, lora_dtype_t dtype, int64_t m_or_t, int64_t k_or_in, int64_t l_or_o,
                           int32_t r_or_R, int32_t num_slots) {
  switch (op) {
    case LORA_OP_FORWARD:
    case LORA_OP_BACKWARD_DX_DA:
    case LORA_OP_BACKWARD_DB:
    case LORA_OP_BACKWARD:
      if (!size_ok(m_or_t) || !size_ok(k_or_in) || !size_ok(l_or_o) || r_or_R < 0 || r_or_R > LORA_MAX_RANK)
        return 0;
      return single_ws(op, dtype, m_or_t, k_or_in, l_or_o, r_or_R);
    case LORA_OP_GROUP_BY_SLOT:
    case LORA_OP_SHRINK:
    case LORA_OP_EXPAND:
    case LORA_OP_APPLY_LINEAR:
      if (!size_ok(m_or_t) || !size_ok(k_or_in) || !size_ok(l_or_o) || r_or_R < 1 || r_or_R > LORA_MAX_RANK ||
          num_slots < 1 || num_slots > LORA_MAX_SLOTS)
        return 0;
      return multi_ws_bytes(op, m_or_t, k_or_in, l_or_o, r_or_R, num_slots);
    case LORA_OP_GATHER_SHRINK:
      return 0;
  }
  return 0;
}

lora_status_t lora_forward(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r, const void *X, int64_t ldx,
                           const void *A, int64_t sA_k, int64_t sA_r, const void *B, int64_t sB_r, int64_t sB_l,
                           void *Y, int64_t ldy, float scale, void *ws, size_t ws_bytes, void *stream) {
  LORA_TRY(check_single_common(dtype, M, K, L, r));
  const int e = dtype == LORA_BF16 ? 2 : 4;
  if (M == 0 || L == 0 || K == 0 || r == 0) return LORA_OK;   // Y += 0
  LORA_TRY(check_big(X, M, K, ldx, e));
  LORA_TRY(check_big(Y, M, L, ldy, e));
  if (A == nullptr || B == nullptr) return LORA_ERR_INVALID_ARG;
  SingleArgs a{};
  a.dtype = dtype; a.M = M; a.K = K; a.L = L; a.r = r;
  a.X = X; a.ldx = ldx; a.A = A; a.sA_k = sA_k; a.sA_r = sA_r; a.B = B; a.sB_r = sB_r; a.sB_l = sB_l;
  a.Y = Y; a.ldy = ldy; a.scale = scale;
  LORA_TRY(check_ws(ws, ws_bytes, single_ws_needed(LORA_OP_FORWARD, a)));
  cudaStream_t st = (cudaStream_t)stream;
  return dtype == LORA_BF16 ? forward_tc(a, ws, ws_bytes, st) : forward_f32(a, st);
}

lora_status_t lora_forward_h(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r, const void *X,
                             int64_t ldx, const void *A, int64_t sA_k, int64_t sA_r, const void *B, int64_t sB_r,
                             int64_t sB_l, void *Y, int64_t ldy, float scale, float *h, int64_t ldh, void *ws,
                             size_t ws_bytes, void *stream) {
  LORA_TRY(check_single_common(dtype, M, K, L, r));
  if (M > 0 && r > 0 && (h == nullptr || ldh < r)) return LORA_ERR_INVALID_ARG;
  const int e = dtype == LORA_BF16 ? 2 : 4;
  cudaStream_t st = (cudaStream_t)stream;
  if (M == 0 || r == 0) return LORA_OK;
  if (K == 0) return fill_zero_2d(LORA_F32, h, M, r, ldh, 1, st);   // h = X * A = 0 and Y += 0
  LORA_TRY(check_big(X, M, K, ldx, e));
  LORA_TRY(check_big(Y, M, L, ldy, e));
  if (A == nullptr || (L > 0 && B == nullptr)) return LORA_ERR_INVALID_ARG;
  SingleArgs a{};
  a.dtype = dtype; a.M = M; a.K = K; a.L = L; a.r = r;
  a.X = X; a.ldx = ldx; a.A = A; a.sA_k = sA_k; a.sA_r = sA_r; a.B = B; a.sB_r = sB_r; a.sB_l = sB_l;
  a.Y = Y; a.ldy = ldy; a.scale = scale; a.h = h; a.ldh = ldh;
  LORA_TRY(check_ws(ws, ws_bytes, single_ws_needed(LORA_OP_FORWARD, a)));
  return dtype == LORA_BF16 ? forward_tc(a, ws, ws_bytes, st) : forward_f32(a, st);
}

lora_status_t lora_backward_ex(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r, const void *X,
                               int64_t ldx, const void *dY, int64_t lddy, const void *A, int64_t sA_k, int64_t sA_r,
                               const void *B, int64_t sB_r, int64_t sB_l, const float *h, int64_t ldh, float scale,
                               void *dX, int64_t lddx, void *dA, int64_t sdA_k, int64_t sdA_r, void *dB,
                               int64_t sdB_r, int64_t sdB_l, uint32_t flags, void *ws, size_t ws_bytes,
                               void *stream) {
  LORA_TRY(check_single_common(dtype, M, K, L, r));
  if (flags & ~(LORA_BWD_DX_ACCUMULATE | LORA_BWD_GRAD_INPUT_DTYPE)) return LORA_ERR_INVALID_ARG;
  const bool acc = (flags & LORA_BWD_DX_ACCUMULATE) != 0;
  // gradients in the input dtype: bf16 for LORA_BF16 (float32 inputs keep float32)
  const lora_dtype_t gdt = (flags & LORA_BWD_GRAD_INPUT_DTYPE) ? dtype : LORA_F32;
  const int e = dtype == LORA_BF16 ? 2 : 4;
  LORA_TRY(check_big(X, M, K, ldx, e));
  LORA_TRY(check_big(dY, M, L, lddy, e));
  LORA_TRY(check_big(dX, M, K, lddx, e));
  if (K > 0 && r > 0 && dA == nullptr) return LORA_ERR_INVALID_ARG;
  if (L > 0 && r > 0 && dB == nullptr) return LORA_ERR_INVALID_ARG;
  if (M > 0 && r > 0 && (h == nullptr || ldh < r)) return LORA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (M == 0 || K == 0 || L == 0 || r == 0) {
    // dyb = 0 or empty: the dX update is zero, and dA and dB are empty or zero sums
    // (dB's h = X * A is zero when K == 0)
    if (!acc) LORA_TRY(fill_zero_2d(dtype, dX, M, K, lddx, 1, st));
    LORA_TRY(fill_zero_2d(gdt, dA, K, r, sdA_k, sdA_r, st));
    return fill_zero_2d(gdt, dB, r, L, sdB_r, sdB_l, st);
  }
  if (A == nullptr || B == nullptr) return LORA_ERR_INVALID_ARG;
  SingleArgs a{};
  a.dtype = dtype; a.M = M; a.K = K; a.L = L; a.r = r;
  a.X = X; a.ldx = ldx; a.dY = dY; a.lddy = lddy; a.A = A; a.sA_k = sA_k; a.sA_r = sA_r;
  a.B = B; a.sB_r = sB_r; a.sB_l = sB_l; a.scale = scale; a.dX = dX; a.lddx = lddx;
  a.dA = (float *)dA; a.sdA_k = sdA_k; a.sdA_r = sdA_r; a.dB = (float *)dB; a.sdB_r = sdB_r; a.sdB_l = sdB_l;
  a.h = const_cast<float *>(h); a.ldh = ldh;
  a.dx_acc = acc ? 1 : 0;
  a.grad_lo = gdt == LORA_BF16 ? 1 : 0;
  LORA_TRY(check_ws(ws, ws_bytes, single_ws_needed(LORA_OP_BACKWARD, a)));
  return dtype == LORA_BF16 ? backward_tc(a, ws, ws_bytes, st) : backward_f32(a, ws, ws_bytes, st);
}

lora_status_t lora_backward(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r, const void *X, int64_t ldx,
                            const void *dY, int64_t lddy, const void *A, int64_t sA_k, int64_t sA_r, const void *B,
                            int64_t sB_r, int64_t sB_l, const float *h, int64_t ldh, float scale, void *dX,
                            int64_t lddx, float *dA, int64_t sdA_k, int64_t sdA_r, float *dB, int64_t sdB_r,
                            int64_t sdB_l, void *ws, size_t ws_bytes, void *stream) {
  return lora_backward_ex(dtype, M, K, L, r, X, ldx, dY, lddy, A, sA_k, sA_r, B, sB_r, sB_l, h, ldh, scale, dX, lddx,
                          dA, sdA_k, sdA_r, dB, sdB_r, sdB_l, 0u, ws, ws_bytes, stream);
}

lora_status_t lora_backward_dx_da(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r, const void *X,
                                  int64_t ldx, const void *dY, int64_t lddy, const void *A, int64_t sA_k,
                                  int64_t sA_r, const void *B, int64_t sB_r, int64_t sB_l, float scale, void *dX,
                                  int64_t lddx, float *dA, int64_t sdA_k, int64_t sdA_r, void *ws, size_t ws_bytes,
                                  void *stream) {
  LORA_TRY(check_single_common(dtype, M, K, L, r));
  const int e = dtype == LORA_BF16 ? 2 : 4;
  LORA_TRY(check_big(X, M, K, ldx, e));
  LORA_TRY(check_big(dY, M, L, lddy, e));
  LORA_TRY(check_big(dX, M, K, lddx, e));
  if (K > 0 && r > 0 && dA == nullptr) return LORA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (M == 0 || K == 0 || L == 0 || r == 0) {
    // dyb = 0 or empty: dX = 0 and dA = 0 wherever they have elements
    LORA_TRY(fill_zero_2d(dtype, dX, M, K, lddx, 1, st));
    LORA_TRY(fill_zero_2d(LORA_F32, dA, K, r, sdA_k, sdA_r, st));
    return LORA_OK;
  }
  if (A == nullptr || B == nullptr) return LORA_ERR_INVALID_ARG;
  SingleArgs a{};
  a.dtype = dtype; a.M = M; a.K = K; a.L = L; a.r = r;
  a.X = X; a.ldx = ldx; a.dY = dY; a.lddy = lddy; a.A = A; a.sA_k = sA_k; a.sA_r = sA_r;
  a.B = B; a.sB_r = sB_r; a.sB_l = sB_l; a.scale = scale; a.dX = dX; a.lddx = lddx;
  a.dA = dA; a.sdA_k = sdA_k; a.sdA_r = sdA_r;
  LORA_TRY(check_ws(ws, ws_bytes, single_ws_needed(LORA_OP_BACKWARD_DX_DA, a)));
  return dtype == LORA_BF16 ? backward_dx_da_tc(a, ws, ws_bytes, st) : backward_dx_da_f32(a, ws, ws_bytes, st);
}

lora_status_t lora_backward_db(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r, const void *X,
                               int64_t ldx, const void *A, int64_t sA_k, int64_t sA_r, const void *dY, int64_t lddy,
                               float scale, float *dB, int64_t sdB_r, int64_t sdB_l, void *ws, size_t ws_bytes,
                               void *stream) {
  LORA_TRY(check_single_common(dtype, M, K, L, r));
  const int e = dtype == LORA_BF16 ? 2 : 4;
  LORA_TRY(check_big(X, M, K, ldx, e));
  LORA_TRY(check_big(dY, M, L, lddy, e));
  if (L > 0 && r > 0 && dB == nullptr) return LORA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (M == 0 || K == 0 || L == 0 || r == 0) {
    LORA_TRY(fill_zero_2d(LORA_F32, dB, r, L, sdB_r, sdB_l, st));   // h = 0 or empty sum
    return LORA_OK;
  }
  if (A == nullptr) return LORA_ERR_INVALID_ARG;
  SingleArgs a{};
  a.dtype = dtype; a.M = M; a.K = K; a.L = L; a.r = r;
  a.X = X; a.ldx = ldx; a.A = A; a.sA_k = sA_k; a.sA_r = sA_r; a.dY = dY; a.lddy = lddy;
  a.scale = scale; a.dB = dB; a.sdB_r = sdB_r; a.sdB_l = sdB_l;
  LORA_TRY(check_ws(ws, ws_bytes, single_ws_needed(LORA_OP_BACKWARD_DB, a)));
  return dtype == LORA_BF16 ? backward_db_tc(a, ws, ws_bytes, st) : backward_db_f32(a, ws, ws_bytes, st);
}

// ----------------------------------------------------------------------------- multi adapter
static lora_status_t check_addr(const lora_addressing_t *addr, const int32_t *ranks) {
  if (addr == nullptr) return LORA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(addr->schedule) & 255u) != 0) return LORA_ERR_ALIGNMENT;
  if (addr->num_tokens < 0 || addr->num_slots < 1 || addr->max_rank < 1) return LORA_ERR_INVALID_ARG;
  if (addr->num_slots > LORA_MAX_SLOTS || addr->max_rank > LORA_MAX_RANK) return LORA_ERR_UNSUPPORTED;
  if (addr->num_tokens > 0 && (addr->slots == nullptr || ranks == nullptr)) return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}

static lora_status_t check_slices(const int32_t *out_slices, int32_t n, int64_t *O) {
  if (n < 1) return LORA_ERR_INVALID_ARG;
  if (n > LORA_MAX_SLICES) return LORA_ERR_UNSUPPORTED;
  if (out_slices == nullptr) return LORA_ERR_INVALID_ARG;
  int64_t o = 0;
  for (int i = 0; i < n; ++i) {
    if (out_slices[i] < 0) return LORA_ERR_INVALID_ARG;
    o += out_slices[i];
  }
  if (!size_ok(o)) return LORA_ERR_INVALID_ARG;
  *O = o;
  return LORA_OK;
}

lora_status_t lora_group_by_slot(const lora_addressing_t *addr, const int32_t *ranks, int32_t *counts, int32_t *perm,
                                 int32_t *num_active, void *ws, size_t ws_bytes, void *stream) {
  LORA_TRY(check_addr(addr, ranks));
  if (counts == nullptr || num_active == nullptr || (addr->num_tokens > 0 && perm == nullptr))
    return LORA_ERR_INVALID_ARG;
  LORA_TRY(check_ws(ws, ws_bytes, multi_ws_bytes(LORA_OP_GROUP_BY_SLOT, addr->num_tokens, 0, 0, addr->max_rank,
                                                 addr->num_slots)));
  return group_by_slot(*addr, ranks, counts, perm, num_active, ws, ws_bytes, (cudaStream_t)stream);
}

size_t lora_schedule_size(int32_t num_tokens, int32_t num_slots) {
  if (num_tokens < 0 || num_slots < 1 || num_slots > LORA_MAX_SLOTS) return 0;
  return schedule_bytes(num_tokens, num_slots);
}

lora_status_t lora_build_schedule(const lora_addressing_t *addr, const int32_t *ranks, void *schedule,
                                  size_t schedule_bytes_, void *stream) {
  LORA_TRY(check_addr(addr, ranks));
  LORA_TRY(check_ws(schedule, schedule_bytes_, schedule_bytes(addr->num_tokens, addr->num_slots)));
  return build_schedule(*addr, ranks, schedule, schedule_bytes_, (cudaStream_t)stream);
}

lora_status_t lora_shrink(const lora_addressing_t *addr, const int32_t *ranks, int64_t in, int32_t num_slices,
                          const void *x, int64_t ldx, const void *a, int64_t sa_slot, int64_t sa_row, float *h,
                          int64_t ldh, void *ws, size_t ws_bytes, void *stream) {
  LORA_TRY(check_addr(addr, ranks));
  if (!size_ok(in) || num_slices < 1) return LORA_ERR_INVALID_ARG;
  if (num_slices > LORA_MAX_SLICES) return LORA_ERR_UNSUPPORTED;
  const int64_t T = addr->num_tokens, NR = (int64_t)num_slices * addr->max_rank;
  LORA_TRY(check_big(x, T, in, ldx, 2));
  LORA_TRY(check_big(h, T, NR, ldh, 4));
  if (T > 0 && in > 0 && a == nullptr) return LORA_ERR_INVALID_ARG;
  if (in > 0 && ((sa_row * 2) % 16 != 0 || (sa_slot * 2) % 16 != 0 || !aligned16(a))) return LORA_ERR_ALIGNMENT;
  LORA_TRY(check_ws(ws, ws_bytes, multi_ws_bytes(LORA_OP_SHRINK, T, in, NR, addr->max_rank, addr->num_slots)));
  if (T == 0) return LORA_OK;
  MultiArgs m{};
  m.addr = *addr; m.ranks = ranks; m.in = in; m.n = num_slices; m.x = x; m.ldx = ldx; m.a = a;
  m.sa_slot = sa_slot; m.sa_row = sa_row; m.h = h; m.ldh = ldh;
  return shrink(m, ws, ws_bytes, (cudaStream_t)stream);
}

lora_status_t lora_expand(const lora_addressing_t *addr, const int32_t *ranks, const float *scalings,
                          const int32_t *out_slices, int32_t num_slices, const float *h, int64_t ldh, const void *b,
                          int64_t sb_slot, int64_t sb_row, int64_t sb_col, void *y, int64_t ldy, void *ws,
                          size_t ws_bytes, void *stream) {
  LORA_TRY(check_addr(addr, ranks));
  int64_t O = 0;
  LORA_TRY(check_slices(out_slices, num_slices, &O));
  const int64_t T = addr->num_tokens, NR = (int64_t)num_slices * addr->max_rank;
  LORA_TRY(check_big(h, T, NR, ldh, 4));
  LORA_TRY(check_big(y, T, O, ldy, 2));
  if (T > 0 && O > 0 && (b == nullptr || scalings == nullptr)) return LORA_ERR_INVALID_ARG;
  LORA_TRY(check_ws(ws, ws_bytes, multi_ws_bytes(LORA_OP_EXPAND, T, 0, O, addr->max_rank, addr->num_slots)));
  if (T == 0 || O == 0) return LORA_OK;
  MultiArgs m{};
  m.addr = *addr; m.ranks = ranks; m.scalings = scalings; m.n = num_slices;
  for (int i = 0; i < num_slices; ++i) m.out_slices[i] = out_slices[i];
  m.O = O; m.h = const_cast<float *>(h); m.ldh = ldh; m.b = b; m.sb_slot = sb_slot; m.sb_row = sb_row; m.sb_col = sb_col;
  m.y = y; m.ldy = ldy;
  return expand(m, ws, ws_bytes, (cudaStream_t)stream);
}

lora_status_t lora_apply_linear(const lora_addressing_t *addr, const int32_t *ranks, const float *scalings,
                                const int32_t *out_slices, int32_t num_slices, int64_t in, const void *x, int64_t ldx,
                                const void *a, int64_t sa_slot, int64_t sa_row, const void *b, int64_t sb_slot,
                                int64_t sb_row, int64_t sb_col, void *y, int64_t ldy, void *ws, size_t ws_bytes,
                                void *stream) {
  LORA_TRY(check_addr(addr, ranks));
  int64_t O = 0;
  LORA_TRY(check_slices(out_slices, num_slices, &O));
  if (!size_ok(in)) return LORA_ERR_INVALID_ARG;
  const int64_t T = addr->num_tokens;
  LORA_TRY(check_big(x, T, in, ldx, 2));
  LORA_TRY(check_big(y, T, O, ldy, 2));
  if (T > 0 && O > 0 && in > 0 && (a == nullptr || b == nullptr || scalings == nullptr)) return LORA_ERR_INVALID_ARG;
  if (in > 0 && ((sa_row * 2) % 16 != 0 || (sa_slot * 2) % 16 != 0 || !aligned16(a))) return LORA_ERR_ALIGNMENT;
  LORA_TRY(check_ws(ws, ws_bytes, multi_ws_bytes(LORA_OP_APPLY_LINEAR, T, in, O, addr->max_rank, addr->num_slots)));
  if (T == 0 || O == 0 || in == 0) return LORA_OK;   // h = 0: y += 0
  MultiArgs m{};
  m.addr = *addr; m.ranks = ranks; m.scalings = scalings; m.n = num_slices;
  for (int i = 0; i < num_slices; ++i) m.out_slices[i] = out_slices[i];
  m.O = O; m.in = in; m.x = x; m.ldx = ldx; m.a = a; m.sa_slot = sa_slot; m.sa_row = sa_row;
  m.b = b; m.sb_slot = sb_slot; m.sb_row = sb_row; m.sb_col = sb_col; m.y = y; m.ldy = ldy;
  return apply_linear(m, ws, ws_bytes, (cudaStream_t)stream);
}

lora_status_t lora_gather_shrink(const lora_addressing_t *addr, const int32_t *ranks, int64_t V, const int64_t *ids,
                                 const void *a, int64_t sa_slot, int64_t sa_row, int64_t sa_col, float *h,
                                 int64_t ldh, void *stream) {
  LORA_TRY(check_addr(addr, ranks));
  if (V < 0) return LORA_ERR_INVALID_ARG;
  const int64_t T = addr->num_tokens;
  LORA_TRY(check_big(h, T, addr->max_rank, ldh, 4));
  if (T > 0 && ids == nullptr) return LORA_ERR_INVALID_ARG;
  if (T > 0 && V > 0 && a == nullptr) return LORA_ERR_INVALID_ARG;
  if (T == 0) return LORA_OK;
  MultiArgs m{};
  m.addr = *addr; m.ranks = ranks; m.in = V; m.ids = ids; m.a = a; m.sa_slot = sa_slot; m.sa_row = sa_row;
  m.sa_col = sa_col; m.h = h; m.ldh = ldh;
  return gather_shrink(m, (cudaStream_t)stream);
}

lora_status_t lora_device_error(int32_t *code) {
  if (code == nullptr) return LORA_ERR_INVALID_ARG;
  int v = 0;
  int parts[5] = {read_clear_error_single_common(), read_clear_error_single_f32(), read_clear_error_multi(),
                  read_clear_error_single_tc(), read_clear_error_decode()};
  for (int p : parts) {
    if (p < 0) return LORA_ERR_CUDA;
    v |= p;
  }
  *code = v;
  return LORA_OK;
}

}  // extern "C"
