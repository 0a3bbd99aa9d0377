/*
 * lora.h -- C ABI of liblora.so: the LoRA low-rank adapter product on one
 * NVIDIA GB300 (sm_103a).
 *
 * Two families of operations:
 *   single adapter (training):  forward   Y += s * (X*A)*B
 *                               backward  dX = s * dY*B^T*A^T,  dA = s * X^T*(dY*B^T),
 *                                         dB = s * (X*A)^T*dY
 *   multi adapter (serving):    group_by_slot, shrink, expand, apply_linear, gather_shrink
 *
 * Sources:
 *   [NeMo lora_kernel]  NeMo AutoModel API page "nemo_automodel.components._peft.lora_kernel"
 *                       (lora_forward_kernel, lora_forward_wrapper, lora_da_dx_kernel,
 *                        lora_da_dx_update_wrapper, lora_db_kernel, lora_db_update_wrapper)
 *   [mstar lora.ops]    mstar page "mstar.engine.resources.lora.ops"
 *                       (shrink, expand_fused, apply_linear_, gather_shrink; the note on
 *                        unspecified rows of h; ops run with no host sync)
 *
 * General conventions (every entry point):
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them.  Scratch memory is passed in as
 *     `ws`/`ws_bytes`; lora_workspace_size() gives the bytes an op needs.
 *     The workspace must be 256-byte aligned and must not be shared by calls
 *     that may run concurrently.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued asynchronously; no entry point synchronises with the device or
 *     reads device data on the host.
 *   - Strides are in ELEMENTS.  "Big" row-major operands (X, Y, dY, dX, x, y)
 *     have unit column stride; their base must be 16-byte aligned and their row
 *     stride times the element size a multiple of 16 bytes, else
 *     LORA_ERR_ALIGNMENT.  With LORA_BF16 the single-adapter extents K and L
 *     must also be multiples of 8 (rows of Y and dX are stored in 16-byte
 *     pieces), else LORA_ERR_ALIGNMENT.  Small operands (A, B, a, b, dA, dB) take arbitrary
 *     strides (e.g. PEFT's lora_A.weight stored r x K is A with sA_k = 1,
 *     sA_r = K).
 *   - Dtypes: LORA_BF16 = bf16 storage with fp32 accumulation, LORA_F32 = fp32
 *     throughout.  Gradients of the adapter (dA, dB) and the intermediate h of
 *     the multi-adapter ops are always fp32.  Multi-adapter ops take bf16 x, a,
 *     b, y.  Results stored in bf16 are rounded to nearest even once, from fp32.
 *   - Host-checkable errors (NULL pointer with a nonzero extent, negative size,
 *     rank above LORA_MAX_RANK, misalignment, workspace too small) return a
 *     status without launching anything.  A failed launch returns
 *     LORA_ERR_CUDA (read with cudaGetLastError, no sync).
 *   - Kernels bound every wait; a wait that runs out sets a device error word
 *     (see lora_device_error) and the kernel returns early.
 */
#ifndef LORA_H_
#define LORA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define LORA_API __attribute__((visibility("default")))
#else
#define LORA_API
#endif

#define LORA_MAX_RANK 128          /* single adapter r, multi-adapter R */
#define LORA_MAX_SLICES 8          /* multi-adapter num_slices */
#define LORA_MAX_SLOTS 4096        /* multi-adapter num_slots */

typedef enum {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = 1,   /* NULL pointer, negative size, inconsistent arguments */
    LORA_ERR_UNSUPPORTED = 2,   /* rank / slices / slots beyond the compiled limits, bad dtype */
    LORA_ERR_ALIGNMENT = 3,     /* a big operand breaks the 16-byte rules above */
    LORA_ERR_WORKSPACE = 4,     /* ws NULL, misaligned or smaller than lora_workspace_size() */
    LORA_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    LORA_ERR_DEVICE = 6         /* returned by lora_device_error(): a kernel flagged an error */
} lora_status_t;

typedef enum { LORA_F32 = 0, LORA_BF16 = 1 } lora_dtype_t;

typedef enum {
    LORA_OP_FORWARD = 0,
    LORA_OP_BACKWARD_DX_DA = 1,
    LORA_OP_BACKWARD_DB = 2,
    LORA_OP_GROUP_BY_SLOT = 3,
    LORA_OP_SHRINK = 4,
    LORA_OP_EXPAND = 5,
    LORA_OP_APPLY_LINEAR = 6,
    LORA_OP_GATHER_SHRINK = 7,
    LORA_OP_BACKWARD = 8
} lora_op_t;

/* Token -> adapter-slot addressing of the multi-adapter ops ([mstar lora.ops]
 * LoraAddressing, read as: one slot index per token, built once per batch).
 *   slots      device int32 [num_tokens]; slot(t)
 *   num_tokens T >= 0, num_slots S in [1, LORA_MAX_SLOTS], max_rank R in [1, LORA_MAX_RANK]
 *   schedule   NULL, or the device schedule that lora_build_schedule made from
 *              these slots, ranks, T, S and R (the grouping of the tokens by slot):
 *              the ops then skip their own grouping step.  The caller keeps it
 *              unchanged while ops that use it run, and rebuilds it whenever the
 *              slots or the ranks change.
 * A token is ACTIVE when 0 <= slot(t) < S and 1 <= ranks[slot(t)] <= R.  An inactive
 * token (the zero adapter, an out-of-range slot or rank) contributes nothing: its
 * row of y is left untouched and its row of h is unspecified. */
typedef struct {
    const int32_t *slots;
    int32_t num_tokens;
    int32_t num_slots;
    int32_t max_rank;
    const void *schedule;
} lora_addressing_t;

/* Bytes of workspace that `op` needs for the given sizes (an upper bound that
 * depends only on its arguments, never on device state).
 *   single-adapter ops: (dtype, M, K, L, r, 0)
 *   multi-adapter ops:  (LORA_BF16, T, in, O, R, S)   O = sum of out_slices;
 *                       for LORA_OP_SHRINK, O = num_slices * R (the width of h),
 *                       or 0 for a bound that holds for any num_slices
 * Returns 0 when the op needs none. */
LORA_API size_t lora_workspace_size(lora_op_t op, lora_dtype_t dtype, int64_t m_or_t, int64_t k_or_in,
                           int64_t l_or_o, int32_t r_or_R, int32_t num_slots);

/* --------------------------------------------------------------------------------
 * lora_forward:  Y[M,L] += scale * (X[M,K] * A[K,r]) * B[r,L]
 * [NeMo lora_kernel] lora_forward_kernel: D = A x B x C with the input (M,K),
 * lora_A (K,N), lora_B (N,L) and the result added into the output (M,L)
 * (block_vector_mul adds; lora_forward_wrapper's `res`).  The rank-r product
 * X*A stays on chip; X is read once and Y read and written once.
 *   X  dtype [M][ldx],  A(k,j) at A[k*sA_k + j*sA_r],  B(j,l) at B[j*sB_r + l*sB_l],
 *   Y  dtype [M][ldy], in/out.  r in [0, LORA_MAX_RANK]; r == 0 or K == 0 leaves Y as is.
 *   ws: lora_workspace_size(LORA_OP_FORWARD, ...) bytes (used only when A or B
 *   is not in a layout the tensor-memory accelerator can read directly).
 * -------------------------------------------------------------------------------- */
LORA_API lora_status_t lora_forward(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r,
                           const void *X, int64_t ldx,
                           const void *A, int64_t sA_k, int64_t sA_r,
                           const void *B, int64_t sB_r, int64_t sB_l,
                           void *Y, int64_t ldy, float scale,
                           void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------------------
 * lora_forward_h:  lora_forward, and also h = X * A (the rank-r hidden rows the
 * forward computes on the way, [NeMo lora_kernel] inner_kernel) written out for
 * lora_backward, which then needs neither X * A again nor a second read of X.
 *   h     float32 [M][ldh] (caller-owned device memory, ldh >= r), overwritten.
 *   ws:   lora_workspace_size(LORA_OP_FORWARD, ...) bytes, as for lora_forward.
 * Errors as lora_forward; h == NULL or ldh < r -> LORA_ERR_INVALID_ARG.
 * -------------------------------------------------------------------------------- */
LORA_API lora_status_t lora_forward_h(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r,
                           const void *X, int64_t ldx,
                           const void *A, int64_t sA_k, int64_t sA_r,
                           const void *B, int64_t sB_r, int64_t sB_l,
                           void *Y, int64_t ldy, float scale,
                           float *h, int64_t ldh,
                           void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------------------
 * lora_backward:  dX, dA and dB in one call from the h that lora_forward_h saved:
 *   dyb = dY*B^T;  dX = scale * dyb*A^T;  dA = scale * X^T*dyb;  dB = scale * h^T*dY
 * [NeMo lora_kernel] lora_da_dx_kernel / lora_da_dx_update_wrapper (dX, dA) and
 * lora_db_kernel / lora_db_update_wrapper (dB, whose X * A is the saved h),
 * restated in the forward roles.  X is read once (by the dX / dA pass).
 *   X, dY, A, B, dX, dA as in lora_backward_dx_da;  dB as in lora_backward_db.
 *   h     float32 [M][ldh], ldh >= r: X * A as lora_forward_h wrote it.
 *   ws:   lora_workspace_size(LORA_OP_BACKWARD, ...) bytes.
 * dX, dA and dB are overwritten.  Errors as lora_backward_dx_da and
 * lora_backward_db; h == NULL or ldh < r -> LORA_ERR_INVALID_ARG.
 * -------------------------------------------------------------------------------- */
LORA_API lora_status_t lora_backward(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r,
                          const void *X, int64_t ldx, const void *dY, int64_t lddy,
                          const void *A, int64_t sA_k, int64_t sA_r,
                          const void *B, int64_t sB_r, int64_t sB_l,
                          const float *h, int64_t ldh, float scale,
                          void *dX, int64_t lddx,
                          float *dA, int64_t sdA_k, int64_t sdA_r,
                          float *dB, int64_t sdB_r, int64_t sdB_l,
                          void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------------------
 * lora_backward_ex:  lora_backward with output options, the `dtype` choice of the
 * [NeMo lora_kernel] update wrappers (lora_da_dx_update_wrapper and
 * lora_db_update_wrapper take the dtype of the gradients they return) and an
 * accumulating dX for a layer input that other branches also feed:
 *   LORA_BWD_DX_ACCUMULATE   dX += scale * dyb*A^T (dX is read, then written;
 *                            one rounding of the sum to dX's dtype per element);
 *                            without it dX is overwritten as by lora_backward.
 *   LORA_BWD_GRAD_INPUT_DTYPE  dA and dB are written in `dtype` (bf16 for
 *                            LORA_BF16, rounded to nearest even once from the
 *                            fp32 sums); without it they are float32.
 *   dA, dB  point to float or to `dtype` elements accordingly (same strides).
 *   Other arguments, the workspace (LORA_OP_BACKWARD) and errors as lora_backward;
 *   an unknown bit in flags -> LORA_ERR_INVALID_ARG.
 * -------------------------------------------------------------------------------- */
#define LORA_BWD_DX_ACCUMULATE 1u
#define LORA_BWD_GRAD_INPUT_DTYPE 2u
LORA_API lora_status_t lora_backward_ex(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r,
                          const void *X, int64_t ldx, const void *dY, int64_t lddy,
                          const void *A, int64_t sA_k, int64_t sA_r,
                          const void *B, int64_t sB_r, int64_t sB_l,
                          const float *h, int64_t ldh, float scale,
                          void *dX, int64_t lddx,
                          void *dA, int64_t sdA_k, int64_t sdA_r,
                          void *dB, int64_t sdB_r, int64_t sdB_l,
                          uint32_t flags, void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------------------
 * lora_backward_dx_da:  dyb = dY*B^T;  dX = scale * dyb*A^T;  dA = scale * X^T*dyb
 * [NeMo lora_kernel] lora_da_dx_kernel (DYB = DY x B and DX = DY x B x A, with
 * lora_B and lora_A passed transposed) and lora_da_dx_update_wrapper (dlora_A
 * reduced from the input and DYB), restated in the forward roles.
 *   X, dY  dtype [M][ldx], [M][lddy];  A, B as in lora_forward.
 *   dX  dtype [M][lddx], OVERWRITTEN (zeros when r == 0 or L == 0).
 *   dA  float, dA(k,j) at dA[k*sdA_k + j*sdA_r], OVERWRITTEN (fp32).
 *   The reduction over M is deterministic (no float atomics).
 * -------------------------------------------------------------------------------- */
LORA_API lora_status_t lora_backward_dx_da(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r,
                                  const void *X, int64_t ldx, const void *dY, int64_t lddy,
                                  const void *A, int64_t sA_k, int64_t sA_r,
                                  const void *B, int64_t sB_r, int64_t sB_l, float scale,
                                  void *dX, int64_t lddx,
                                  float *dA, int64_t sdA_k, int64_t sdA_r,
                                  void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------------------
 * lora_backward_db:  h = X*A;  dB = scale * h^T*dY
 * [NeMo lora_kernel] lora_db_kernel (AXT = A x X^T, i.e. (X*A)^T) and
 * lora_db_update_wrapper (d_lora_B from AXT and the output gradient).
 *   dB  float, dB(j,l) at dB[j*sdB_r + l*sdB_l], OVERWRITTEN (zeros when K == 0).
 * -------------------------------------------------------------------------------- */
LORA_API lora_status_t lora_backward_db(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r,
                               const void *X, int64_t ldx,
                               const void *A, int64_t sA_k, int64_t sA_r,
                               const void *dY, int64_t lddy, float scale,
                               float *dB, int64_t sdB_r, int64_t sdB_l,
                               void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------------------
 * lora_backward_db_noalloc: lora_backward_db for callers that cannot allocate
 * device memory.  The pages have no counterpart of this entry point; it exists
 * for code that runs where the surrounding system owns all device memory (an
 * operator inside another engine's memory pool, a plugin that is handed tensors
 * but no allocator) or where a cudaMalloc, with its implicit device-wide
 * synchronisation, cannot be afforded on the hot path.
 *   Arguments, results and errors are those of lora_backward_db, without ws /
 *   ws_bytes.  Scratch comes from a LORA_DB_NOALLOC_SCRATCH_BYTES array of the
 *   library's own device memory, which every GPU that loads the library holds
 *   until the process exits.  Sizes whose lora_workspace_size(LORA_OP_BACKWARD_DB,
 *   ...) exceeds it are rejected with LORA_ERR_WORKSPACE before anything is
 *   launched.  No cudaMalloc, cudaFree or allocating library call is made.
 *   Argument errors (dtype, negative or oversized extents, rank) are reported
 *   before the size check.  The first call in a CUDA context (for runtime-API
 *   callers the primary context of the current device; else the context current
 *   on the calling thread) looks up the array's device address in that context
 *   and caches it under the context's unique id, so a context created later
 *   (after cudaDeviceReset, or by an engine's own cuCtxCreate) gets its own
 *   lookup.  Make that first call before any stream capture in that context.
 *   All calls share the one array and the kernels re-clear what
 *   must start at zero on every call, but two calls that can run at the same time
 *   on the GPU (other streams, other host threads) race on it: serialise them.
 * -------------------------------------------------------------------------------- */
#define LORA_DB_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
LORA_API lora_status_t lora_backward_db_noalloc(lora_dtype_t dtype, int64_t M, int64_t K, int64_t L, int32_t r,
                               const void *X, int64_t ldx,
                               const void *A, int64_t sA_k, int64_t sA_r,
                               const void *dY, int64_t lddy, float scale,
                               float *dB, int64_t sdB_r, int64_t sdB_l, void *stream);

/* --------------------------------------------------------------------------------
 * lora_group_by_slot: the integer step in front of the segmented kernels.
 * counts[s] = number of active tokens on slot s; perm[0..n) = the active tokens
 * ordered by (slot, token index) (a stable counting sort); *num_active = n.
 * Runs on the device with no host sync ([mstar lora.ops]: no host sync and no
 * data-dependent shape).  counts: device int32 [S]; perm: device int32 [T];
 * num_active: device int32 [1].  Entries perm[n..T) are left unspecified.
 * -------------------------------------------------------------------------------- */
LORA_API lora_status_t lora_group_by_slot(const lora_addressing_t *addr, const int32_t *ranks,
                                 int32_t *counts, int32_t *perm, int32_t *num_active,
                                 void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------------------
 * lora_schedule_size / lora_build_schedule: the grouping step of the segmented
 * ops (the stable sort of the active tokens by slot and the list of tiles of at
 * most 128 tokens of one slot, as lora_group_by_slot defines it) done once, into
 * a device buffer that lora_shrink, lora_expand and lora_apply_linear then reuse
 * through addr->schedule ([mstar lora.ops]: the addressing of a batch is built
 * once and serves every adapted layer; no host sync, no data-dependent shape).
 *   schedule       device buffer of lora_schedule_size(T, S) bytes, 256-byte
 *                  aligned, written by the call (addr->schedule is ignored).
 * Errors: as lora_group_by_slot; a buffer that is NULL, misaligned or too small
 * -> LORA_ERR_WORKSPACE.
 * -------------------------------------------------------------------------------- */
LORA_API size_t lora_schedule_size(int32_t num_tokens, int32_t num_slots);
LORA_API lora_status_t lora_build_schedule(const lora_addressing_t *addr, const int32_t *ranks, void *schedule,
                                  size_t schedule_bytes, void *stream);

/* --------------------------------------------------------------------------------
 * lora_shrink:  h[t, i*R + j] = sum_k x[t,k] * a[slot(t)][i*R + j][k],  j < rank(slot(t))
 * [mstar lora.ops] shrink: h[t] = x[t] @ a[slot(t)]^T, num_slices stacked blocks.
 *   ranks   device int32 [S];  x  bf16 [T][ldx], in columns;
 *   a       bf16, element (s, row, k) at a[s*sa_slot + row*sa_row + k], rows n*R;
 *   h       float [T][ldh], n*R columns.  Rows of inactive tokens and columns
 *           past a slot's rank are unspecified (the page allows anything there).
 * -------------------------------------------------------------------------------- */
LORA_API lora_status_t lora_shrink(const lora_addressing_t *addr, const int32_t *ranks,
                          int64_t in, int32_t num_slices,
                          const void *x, int64_t ldx,
                          const void *a, int64_t sa_slot, int64_t sa_row,
                          float *h, int64_t ldh,
                          void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------------------
 * lora_expand:  y[t, off_i + c] += scalings[slot(t)] * sum_{j<rank} h[t, i*R + j] * b[slot(t)][off_i + c][j]
 * [mstar lora.ops] expand_fused: y[t, slice i] += scalings[slot(t)] * h[t, slice i] @ b[slot(t), slice i]^T.
 *   out_slices  HOST int32 [num_slices] (shape metadata); off_i = running sum; O = total.
 *   scalings    device float [S] (never read for inactive slots).
 *   h           float [T][ldh];  b bf16, element (s, c, j) at b[s*sb_slot + c*sb_row + j*sb_col];
 *   y           bf16 [T][ldy], in/out; rows of inactive tokens are untouched.
 *   Only h columns j < rank are read (the rest may hold anything, NaN included).
 * -------------------------------------------------------------------------------- */
LORA_API lora_status_t lora_expand(const lora_addressing_t *addr, const int32_t *ranks, const float *scalings,
                          const int32_t *out_slices, int32_t num_slices,
                          const float *h, int64_t ldh,
                          const void *b, int64_t sb_slot, int64_t sb_row, int64_t sb_col,
                          void *y, int64_t ldy,
                          void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------------------
 * lora_apply_linear: shrink then expand into y in one call ([mstar lora.ops]
 * apply_linear_).  The two kernels share one device-built schedule and are
 * chained with programmatic dependent launch; h passes between them through the
 * workspace (it stays in L2).  Arguments as in lora_shrink / lora_expand.
 * -------------------------------------------------------------------------------- */
LORA_API lora_status_t lora_apply_linear(const lora_addressing_t *addr, const int32_t *ranks,
                                const float *scalings, const int32_t *out_slices, int32_t num_slices,
                                int64_t in, const void *x, int64_t ldx,
                                const void *a, int64_t sa_slot, int64_t sa_row,
                                const void *b, int64_t sb_slot, int64_t sb_row, int64_t sb_col,
                                void *y, int64_t ldy,
                                void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------------------
 * lora_gather_shrink:  h[t, j] = a[slot(t)][j][ids[t]] for j < rank, if 0 <= ids[t] < V,
 *                      else h[t, 0..rank) = 0.
 * [mstar lora.ops] gather_shrink: the shrink of a token's one-hot row; an id
 * outside [0, in) contributes nothing.  An exact copy (bit-for-bit).
 *   ids  device int64 [T];  a bf16, element (s, j, v) at a[s*sa_slot + j*sa_row + v*sa_col];
 *   h    float [T][ldh]: columns j < rank written for active tokens; the rest unspecified.
 * -------------------------------------------------------------------------------- */
LORA_API lora_status_t lora_gather_shrink(const lora_addressing_t *addr, const int32_t *ranks, int64_t V,
                                 const int64_t *ids,
                                 const void *a, int64_t sa_slot, int64_t sa_row, int64_t sa_col,
                                 float *h, int64_t ldh, void *stream);

/* Human-readable name of a status code (static string). */
LORA_API const char *lora_status_string(lora_status_t status);

/* Reads and clears the device error word of the current device (a host sync on
 * the legacy default stream; diagnostics only).  *code = 0 when no kernel has
 * flagged an error, else a bit set (1: a wait timed out).  Returns LORA_OK, or
 * LORA_ERR_CUDA if the read failed. */
LORA_API lora_status_t lora_device_error(int32_t *code);

/* Number of kernels this library has launched in this process so far (all
 * devices, all streams; a relaxed counter for diagnostics and benchmarks). */
LORA_API uint64_t lora_kernel_launches(void);

/* Library version string. */
LORA_API const char *lora_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LORA_H_ */
