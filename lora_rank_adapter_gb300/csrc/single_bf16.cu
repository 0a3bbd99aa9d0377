// single_bf16.cu -- single-adapter LoRA kernels, bf16 storage / fp32 accumulate,
// for sm_103a.
//
// Operations ([NeMo lora_kernel] = NeMo AutoModel API page
// "nemo_automodel.components._peft.lora_kernel"):
//   forward      Y += s * (X*A)*B          lora_forward_kernel (inner_kernel + block_vector_mul)
//   dyb / h      partial row products      lora_da_dx_kernel's DYB = DY x B, lora_db_kernel's X*A
//   dX + dA      dX = s*dyb*A^T, dA = s*X^T*dyb      lora_da_dx_kernel / lora_da_dx_update_wrapper
//   dB           dB = s*h^T*dY                         lora_db_update_wrapper
//
// Design (all kernels): one producer warp drives the tensor-memory accelerator
// (TMA) through a ring of shared-memory stages guarded by mbarriers; four
// consumer warps run mma.sync m16n8k16 on ldmatrix fragments.  Every big
// operand tile is 64 x 64 bf16 (one 128-byte swizzled row per tile row).  Tiles
// that a kernel writes back (Y, dX) are updated in place in their stage and
// stored by the producer with a TMA store before the stage is reused.
// Out-of-range rows/columns are zero-filled by TMA on load and clipped on store.
//
// Small operands use fixed layouts: A as Ac[j][k] (k contiguous; PEFT's
// lora_A.weight) and B as Bc[l][j] (j contiguous; PEFT's lora_B.weight).  The
// host packs other layouts into the workspace first.  Rank r is padded to the
// bucket RP (16/32/64/128) by TMA zero fill.
//
// fp32 intermediates that feed a bf16 mma (h in the forward, dyb, h in dB) are
// split into bf16 hi + lo parts and multiplied twice, so the product keeps
// about 16 mantissa bits instead of 8.
#include <algorithm>

#include "common.cuh"
#include "host_common.h"
#include "single_bf16.h"

namespace lora {

constexpr int BM = 64;                  // rows per tile
constexpr int BK = 64;                  // columns per tile
constexpr int NCW = 4;                  // consumer warps (one 16-row slice each)
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr int TILE_BYTES = BM * BK * 2; // 8 KB

// Shared memory given to the stage ring of one CTA (bytes in flight per CTA);
// the number of stages of each kernel follows from its stage size.
#ifndef LORA_STAGE_BUDGET_KB
#define LORA_STAGE_BUDGET_KB 48
#endif
__host__ __device__ constexpr int stages_for(int stage_bytes, int lo = 2, int hi = 16) {
  return (LORA_STAGE_BUDGET_KB * 1024) / stage_bytes < lo   ? lo
         : (LORA_STAGE_BUDGET_KB * 1024) / stage_bytes > hi ? hi
                                                             : (LORA_STAGE_BUDGET_KB * 1024) / stage_bytes;
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Byte offset of (row, col) in a 64x64 bf16 tile (128-byte swizzle).
__device__ __forceinline__ uint32_t tile_off(int row, int col) { return swz(row, col * 2, 128); }
// Ac tile [RP rows j][64 cols k] (128-byte swizzle).
__device__ __forceinline__ uint32_t rk_off(int j, int k) { return swz(j, k * 2, 128); }
// [64 rows][RP cols] tile stored as panels of PW = min(RP, 64) columns, each with a
// (PW*2)-byte swizzle: Bc tiles, and the bf16 staging of dyb / h.
template <int RP>
__device__ __forceinline__ uint32_t lr_off(int row, int col) {
  constexpr int PW = RP < 64 ? RP : 64;
  return (col / PW) * (64 * PW * 2) + swz(row, (col % PW) * 2, PW * 2);
}

// --- fragment loaders (lane addressing of ldmatrix.x4) -------------------------
// A operand 16x16 at (r0, c0) of a row-major store [rows][contraction].
template <typename F>
__device__ __forceinline__ void ld_a(uint32_t base, int r0, int c0, F off, uint32_t (&a)[4]) {
  const int l = lane_id();
  ldsm_x4(base + off(r0 + (l & 15), c0 + ((l >> 4) << 3)), a[0], a[1], a[2], a[3]);
}
// A operand 16x16 whose rows r0.. are the COLUMNS of a store [contraction][rows].
template <typename F>
__device__ __forceinline__ void ld_a_t(uint32_t base, int r0, int c0, F off, uint32_t (&a)[4]) {
  const int l = lane_id(), q = l >> 3;
  ldsm_x4_t(base + off(c0 + (l & 7) + ((q >> 1) << 3), r0 + ((q & 1) << 3)), a[0], a[1], a[2], a[3]);
}
// B operands of two n8 tiles (n0.., n0+8..) x k16 at k0 from a store [n][k].
template <typename F>
__device__ __forceinline__ void ld_b_nk(uint32_t base, int n0, int k0, F off, uint32_t (&b)[4]) {
  const int l = lane_id();
  ldsm_x4(base + off(n0 + (l & 7) + ((l >> 4) << 3), k0 + (((l >> 3) & 1) << 3)), b[0], b[1], b[2], b[3]);
}
// Same from a store [k][n].
template <typename F>
__device__ __forceinline__ void ld_b_kn(uint32_t base, int n0, int k0, F off, uint32_t (&b)[4]) {
  const int l = lane_id();
  ldsm_x4_t(base + off(k0 + (l & 7) + (((l >> 3) & 1) << 3), n0 + ((l >> 4) << 3)), b[0], b[1], b[2], b[3]);
}

// Warp-uniform bounded wait.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait<kCluster>(bar, parity));
}

// =============================================================================
// Warp roles shared by the kernels below: warps 0..3 consume (mma.sync), warp 4
// loads (TMA), and in kernels that write tiles back, warp 5 stores (TMA).
// Barriers per stage s: full[s] (loads landed, transaction count), done[s] (the
// four consumer warps are finished with the stage) and, with a storer, free[s]
// (the store has read the stage; the loader may refill it).
// =============================================================================
constexpr int NTHREADS_LS = (NCW + 2) * 32;   // consumers + loader + storer
constexpr int kStoreDepth = 2;                // TMA stores kept in flight by the storer

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Storer loop (one lane).  For every tile g in order: wait until the consumers
// are done with its stage, issue its TMA store if store(g, s) does so, and free
// stages for the loader once their stores have read them.  At most D stores
// stay unreleased; D < NS keeps a free stage for the loader, so the loader,
// consumers and storer can always make progress.  Tiles without a store are
// freed at once.
template <int NS, typename StoreFn>
__device__ __forceinline__ void storer_run(int ntiles, uint64_t *done, uint64_t *freeb, StoreFn store) {
  static_assert(NS >= 2, "a storer needs at least two stages");
  constexpr int D = (NS - 1) < kStoreDepth ? (NS - 1) : kStoreDepth;
  int pend[D + 1];
  int np = 0;
  for (int g = 0; g < ntiles; ++g) {
    const int s = g % NS;
    if (!mbar_wait(&done[s], (g / NS) & 1)) break;
    if (store(g, s)) {
      bulk_commit();
      pend[np++] = g;
      if (np > D) {
        bulk_wait_read<D>();
        mbar_arrive(&freeb[pend[0] % NS]);
        for (int i = 1; i < np; ++i) pend[i - 1] = pend[i];
        --np;
      }
    } else {
      mbar_arrive(&freeb[s]);
    }
  }
  bulk_wait_read<0>();
  for (int i = 0; i < np; ++i) mbar_arrive(&freeb[pend[i] % NS]);
  bulk_wait_all();
}

// =============================================================================
// Forward: Y[M,L] += s * (X*Ac^T) * Bc^T
// A cluster of `cl` CTAs shares one 64-row block: CTA c runs K-chunks
// [c*nk/cl, (c+1)*nk/cl) of the shrink, the partial h are summed in cluster-rank
// order through distributed shared memory (identical in every CTA), then CTA c
// runs its share of the L-chunks of the expand.  X is read once and Y is read
// and written once; Y tiles are updated in place in their stage and written
// back by the storer warp.
// =============================================================================
template <int RP>
struct FwdCfg {
  static constexpr int SMALL = RP * 128;          // Ac [RP][64] or Bc [64][RP]
  static constexpr int STAGE = TILE_BYTES + SMALL;
  static constexpr int NS = stages_for(STAGE, 3);
  static constexpr int HBUF = BM * RP * 4;
  static constexpr int BYTES = 1024 + NS * STAGE + HBUF + 8 * (3 * NS + 2);
};

template <int RP>
__global__ void __launch_bounds__(NTHREADS_LS) fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmX,
                                                               const __grid_constant__ CUtensorMap tmA,
                                                               const __grid_constant__ CUtensorMap tmB,
                                                               const __grid_constant__ CUtensorMap tmY,
                                                               FwdArgs p) {
  using C = FwdCfg<RP>;
  constexpr int NS = C::NS;
  constexpr int PW = RP < 64 ? RP : 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  float *hbuf = reinterpret_cast<float *>(smem + NS * C::STAGE);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * C::STAGE + C::HBUF);
  uint64_t *done = full + NS;
  uint64_t *freeb = done + NS;
  uint64_t *hready = freeb + NS;
  uint64_t *hdone = hready + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cl = p.cl;
  const uint32_t crank = cl > 1 ? cluster_ctarank() : 0u;
  const int m0 = (blockIdx.x / cl) * BM;
  const int nk = (p.K + BK - 1) / BK, nl = (p.L + BK - 1) / BK;
  const int k_beg = (int)((int64_t)nk * crank / cl), k_end = (int)((int64_t)nk * (crank + 1) / cl);
  const int l_beg = (int)((int64_t)nl * crank / cl), l_end = (int)((int64_t)nl * (crank + 1) / cl);
  const int n1 = k_end - k_beg, ntiles = n1 + (l_end - l_beg);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&done[s], NCW);
      mbar_init(&freeb[s], 1);
    }
    mbar_init(hready, cl > 1 ? NCW * 32 * (cl - 1) : 1);
    mbar_init(hdone, cl > 1 ? NCW * 32 * (cl - 1) : 1);
    fence_barrier_init();
  }
  if (cl > 1) cluster_sync_all(); else __syncthreads();
  pdl_wait();

  if (warp == NCW) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      prefetch_tmap(&tmY);
      for (int g = 0; g < ntiles; ++g) {
        const int s = g % NS;
        if (g >= NS && !mbar_wait(&freeb[s], ((g / NS) & 1) ^ 1)) break;
        uint8_t *st = smem + s * C::STAGE;
        mbar_arrive_expect_tx(&full[s], C::STAGE);
        if (g < n1) {
          const int kc = k_beg + g;
          tma_load_2d(st, &tmX, &full[s], kc * BK, m0);
          tma_load_2d(st + TILE_BYTES, &tmA, &full[s], kc * BK, 0);
        } else {
          const int lc = l_beg + g - n1;
          tma_load_2d(st, &tmY, &full[s], lc * BK, m0);
#pragma unroll
          for (int pp = 0; pp < RP / PW; ++pp)
            tma_load_2d(st + TILE_BYTES + pp * (64 * PW * 2), &tmB, &full[s], pp * PW, lc * BK);
        }
      }
    }
    pdl_launch_dependents();
    return;
  }
  if (warp == NCW + 1) {
    // ------------------------------------------------------------ storer
    if (lane == 0)
      storer_run<NS>(ntiles, done, freeb, [&](int g, int s) {
        if (g < n1) return false;
        tma_store_2d(&tmY, smem + s * C::STAGE, (l_beg + g - n1) * BK, m0);
        return true;
      });
    pdl_launch_dependents();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int w = warp, gq = lane >> 2, cq = lane & 3;
  float hacc[RP / 8][4];
#pragma unroll
  for (int i = 0; i < RP / 8; ++i) hacc[i][0] = hacc[i][1] = hacc[i][2] = hacc[i][3] = 0.f;
  bool ok = true;
  int g = 0;
  for (; g < n1; ++g) {
    const int s = g % NS;
    if (!(ok = wait_all(&full[s], (g / NS) & 1))) break;
    const uint32_t tb = smem_u32(smem + s * C::STAGE), sb = tb + TILE_BYTES;
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      uint32_t a[4];
      ld_a(tb, 16 * w, kk * 16, tile_off, a);
#pragma unroll
      for (int np = 0; np < RP / 16; ++np) {
        uint32_t b[4];
        ld_b_nk(sb, np * 16, kk * 16, rk_off, b);
        mma_bf16(hacc[2 * np], a, b[0], b[1]);
        mma_bf16(hacc[2 * np + 1], a, b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&done[s]);
  }

  if (cl > 1) {
    // partial h through distributed shared memory, summed in cluster-rank order
    const int r0 = 16 * w + gq;
#pragma unroll
    for (int nt = 0; nt < RP / 8; ++nt) {
      *reinterpret_cast<float2 *>(&hbuf[r0 * RP + nt * 8 + 2 * cq]) = make_float2(hacc[nt][0], hacc[nt][1]);
      *reinterpret_cast<float2 *>(&hbuf[(r0 + 8) * RP + nt * 8 + 2 * cq]) = make_float2(hacc[nt][2], hacc[nt][3]);
    }
    for (int c = 0; c < cl; ++c)
      if (c != (int)crank) mbar_arrive_remote(hready, c);
    if (!wait_all<true>(hready, 0)) ok = false;
    if (ok) {
#pragma unroll
      for (int nt = 0; nt < RP / 8; ++nt) {
        float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
        for (int c = 0; c < cl; ++c) {
          float2 v0, v1;
          if (c == (int)crank) {
            v0 = make_float2(hacc[nt][0], hacc[nt][1]);
            v1 = make_float2(hacc[nt][2], hacc[nt][3]);
          } else {
            v0 = ld_dsmem_f2(&hbuf[r0 * RP + nt * 8 + 2 * cq], c);
            v1 = ld_dsmem_f2(&hbuf[(r0 + 8) * RP + nt * 8 + 2 * cq], c);
          }
          s0.x += v0.x; s0.y += v0.y; s1.x += v1.x; s1.y += v1.y;
        }
        hacc[nt][0] = s0.x; hacc[nt][1] = s0.y; hacc[nt][2] = s1.x; hacc[nt][3] = s1.y;
      }
    }
    for (int c = 0; c < cl; ++c)
      if (c != (int)crank) mbar_arrive_remote(hdone, c);
  }

  // the full h of this row block (identical in every CTA of the cluster): CTA 0 writes it out
  if (ok && p.h != nullptr && crank == 0) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int64_t m = m0 + 16 * w + gq + 8 * hf;
      if (m >= p.M) continue;
      float *hrow = p.h + m * p.ldh;
#pragma unroll
      for (int nt = 0; nt < RP / 8; ++nt) {
        const int j = nt * 8 + 2 * cq;
        if (j < p.r) hrow[j] = hacc[nt][2 * hf];
        if (j + 1 < p.r) hrow[j + 1] = hacc[nt][2 * hf + 1];
      }
    }
  }
  // h as A fragments (hi + lo bf16)
  uint32_t ahi[RP / 16][4], alo[RP / 16][4];
#pragma unroll
  for (int q = 0; q < RP / 16; ++q) {
    split_bf16(hacc[2 * q][0], hacc[2 * q][1], ahi[q][0], alo[q][0]);
    split_bf16(hacc[2 * q][2], hacc[2 * q][3], ahi[q][1], alo[q][1]);
    split_bf16(hacc[2 * q + 1][0], hacc[2 * q + 1][1], ahi[q][2], alo[q][2]);
    split_bf16(hacc[2 * q + 1][2], hacc[2 * q + 1][3], ahi[q][3], alo[q][3]);
  }
  const float scale = p.scale;
  for (; ok && g < ntiles; ++g) {
    const int s = g % NS;
    if (!(ok = wait_all(&full[s], (g / NS) & 1))) break;
    uint8_t *st = smem + s * C::STAGE;
    const uint32_t sb = smem_u32(st) + TILE_BYTES;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int q = 0; q < RP / 16; ++q) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b[4];
        ld_b_nk(sb, np * 16, q * 16, lr_off<RP>, b);
        mma_bf16(acc[2 * np], ahi[q], b[0], b[1]);
        mma_bf16(acc[2 * np], alo[q], b[0], b[1]);
        mma_bf16(acc[2 * np + 1], ahi[q], b[2], b[3]);
        mma_bf16(acc[2 * np + 1], alo[q], b[2], b[3]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t *yp = reinterpret_cast<uint32_t *>(st + tile_off(16 * w + gq + 8 * hf, nt * 8 + 2 * cq));
        float2 y = unpack_bf16(*yp);
        *yp = pack_bf16(y.x + scale * acc[nt][2 * hf], y.y + scale * acc[nt][2 * hf + 1]);
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&done[s]);
  }
  pdl_launch_dependents();
  if (cl > 1) wait_all<true>(hdone, 0);   // peers are done reading this CTA's hbuf
}

// =============================================================================
// Row products: out[m][j] = sum over the contraction of In[m][k] * W(k, j)
//   dyb: In = dY (M x L), W = Bc [l][j]  (kW_KN = true: the store is [k][n])
//   h:   In = X  (M x K), W = Ac [j][k]  (kW_KN = false: the store is [n][k])
// A cluster of `csplit` CTAs splits the contraction of one 64-row block; the
// partials are summed in cluster-rank order through distributed shared memory
// and written once, already split into bf16 hi/lo and laid out as the column
// pass reads them (a "blob" of 2 x 64 x RP bf16 per row block, lr_off order).
// Block 0 also zeroes the column-pass counters.
// =============================================================================
template <int RP>
struct RowsCfg {
  static constexpr int SMALL = RP * 128;
  static constexpr int STAGE = TILE_BYTES + SMALL;
  static constexpr int NS = stages_for(STAGE);
  static constexpr int HBUF = BM * RP * 4;
  static constexpr int BYTES = 1024 + NS * STAGE + HBUF + 8 * (2 * NS + 2);
};
template <int RP>
__host__ __device__ constexpr int blob_bytes() { return RP * 256; }   // hi + lo, 64 rows x RP bf16 each

template <int RP>
__device__ __forceinline__ void write_blob_rows(uint8_t *blob, int w, int gq, int cq, const float (&acc)[RP / 8][4]) {
  uint8_t *bhi = blob, *blo = blob + RP * 128;
#pragma unroll
  for (int nt = 0; nt < RP / 8; ++nt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t h, l;
      split_bf16(acc[nt][2 * hf], acc[nt][2 * hf + 1], h, l);
      const uint32_t o = lr_off<RP>(16 * w + gq + 8 * hf, nt * 8 + 2 * cq);
      *reinterpret_cast<uint32_t *>(bhi + o) = h;
      *reinterpret_cast<uint32_t *>(blo + o) = l;
    }
}

// The saved h (fp32 [M][ldh], columns j < r; zero past r and past M) as the
// column pass's hi/lo blob, one 64-row block per CTA.  Block 0 also zeroes the
// column-pass counters.
template <int RP>
__global__ void __launch_bounds__(256) hblob_kernel(const float *__restrict__ h, int64_t ldh, int64_t M, int r,
                                                    uint8_t *blob, int *counters, int ncounters) {
  pdl_wait();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < ncounters; i += blockDim.x) counters[i] = 0;
  uint8_t *bhi = blob + (size_t)blockIdx.x * blob_bytes<RP>(), *blo = bhi + RP * 128;
  const int64_t m0 = (int64_t)blockIdx.x * BM;
  for (int e = threadIdx.x; e < BM * RP / 2; e += blockDim.x) {
    const int row = e / (RP / 2), col = 2 * (e % (RP / 2));
    const int64_t m = m0 + row;
    const float v0 = m < M && col < r ? h[m * ldh + col] : 0.f;
    const float v1 = m < M && col + 1 < r ? h[m * ldh + col + 1] : 0.f;
    uint32_t hi, lo;
    split_bf16(v0, v1, hi, lo);
    const uint32_t o = lr_off<RP>(row, col);
    *reinterpret_cast<uint32_t *>(bhi + o) = hi;
    *reinterpret_cast<uint32_t *>(blo + o) = lo;
  }
  pdl_launch_dependents();
}

template <int RP, bool kW_KN>
__global__ void __launch_bounds__(NTHREADS) rows_bf16_kernel(const __grid_constant__ CUtensorMap tmIn,
                                                             const __grid_constant__ CUtensorMap tmW,
                                                             RowsArgs p) {
  using C = RowsCfg<RP>;
  constexpr int NS = C::NS;
  constexpr int PW = RP < 64 ? RP : 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  float *hbuf = reinterpret_cast<float *>(smem + NS * C::STAGE);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * C::STAGE + C::HBUF);
  uint64_t *empty = full + NS;
  uint64_t *hready = empty + NS;
  uint64_t *hdone = hready + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cs = p.csplit;
  const uint32_t c = cs > 1 ? cluster_ctarank() : 0u;
  const int rb = blockIdx.x / cs;
  const int m0 = rb * BM;
  const int nk = (p.Kc + BK - 1) / BK;
  const int k_beg = (int)((int64_t)nk * c / cs), k_end = (int)((int64_t)nk * (c + 1) / cs);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    mbar_init(hready, cs > 1 ? NCW * 32 * (cs - 1) : 1);
    mbar_init(hdone, cs > 1 ? NCW * 32 * (cs - 1) : 1);
    fence_barrier_init();
  }
  if (cs > 1) cluster_sync_all(); else __syncthreads();
  pdl_wait();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < p.ncounters; i += blockDim.x) p.counters[i] = 0;

  if (warp == NCW) {
    if (lane == 0) {
      prefetch_tmap(&tmIn);
      prefetch_tmap(&tmW);
      int g = 0;
      for (int kc = k_beg; kc < k_end; ++kc, ++g) {
        const int s = g % NS;
        if (g >= NS && !mbar_wait(&empty[s], ((g / NS) & 1) ^ 1)) break;
        uint8_t *st = smem + s * C::STAGE;
        mbar_arrive_expect_tx(&full[s], C::STAGE);
        tma_load_2d(st, &tmIn, &full[s], kc * BK, m0);
        if (kW_KN) {
#pragma unroll
          for (int pp = 0; pp < RP / PW; ++pp)
            tma_load_2d(st + TILE_BYTES + pp * (64 * PW * 2), &tmW, &full[s], pp * PW, kc * BK);
        } else {
          tma_load_2d(st + TILE_BYTES, &tmW, &full[s], kc * BK, 0);
        }
      }
    }
    pdl_launch_dependents();
    return;
  }

  const int w = warp, gq = lane >> 2, cq = lane & 3;
  float hacc[RP / 8][4];
#pragma unroll
  for (int i = 0; i < RP / 8; ++i) hacc[i][0] = hacc[i][1] = hacc[i][2] = hacc[i][3] = 0.f;
  int g = 0;
  bool ok = true;
  for (int kc = k_beg; kc < k_end; ++kc, ++g) {
    const int s = g % NS;
    if (!(ok = wait_all(&full[s], (g / NS) & 1))) break;
    const uint32_t tb = smem_u32(smem + s * C::STAGE), sb = tb + TILE_BYTES;
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      uint32_t a[4];
      ld_a(tb, 16 * w, kk * 16, tile_off, a);
#pragma unroll
      for (int np = 0; np < RP / 16; ++np) {
        uint32_t b[4];
        if (kW_KN) ld_b_kn(sb, np * 16, kk * 16, lr_off<RP>, b);
        else ld_b_nk(sb, np * 16, kk * 16, rk_off, b);
        mma_bf16(hacc[2 * np], a, b[0], b[1]);
        mma_bf16(hacc[2 * np + 1], a, b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  pdl_launch_dependents();
  uint8_t *blob = p.blob + (size_t)rb * blob_bytes<RP>();
  if (cs == 1) {
    if (ok) write_blob_rows<RP>(blob, w, gq, cq, hacc);
    return;
  }
  const int r0 = 16 * w + gq;
#pragma unroll
  for (int nt = 0; nt < RP / 8; ++nt) {
    *reinterpret_cast<float2 *>(&hbuf[r0 * RP + nt * 8 + 2 * cq]) = make_float2(hacc[nt][0], hacc[nt][1]);
    *reinterpret_cast<float2 *>(&hbuf[(r0 + 8) * RP + nt * 8 + 2 * cq]) = make_float2(hacc[nt][2], hacc[nt][3]);
  }
  for (int q = 0; q < cs; ++q)
    if (q != (int)c) mbar_arrive_remote(hready, q);
  if (!wait_all<true>(hready, 0)) ok = false;
  if (ok && (w % cs) == (int)c) {
    // this CTA reduces (and writes) the 16 rows of warp w
#pragma unroll
    for (int nt = 0; nt < RP / 8; ++nt) {
      float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
      for (int q = 0; q < cs; ++q) {
        float2 v0, v1;
        if (q == (int)c) {
          v0 = make_float2(hacc[nt][0], hacc[nt][1]);
          v1 = make_float2(hacc[nt][2], hacc[nt][3]);
        } else {
          v0 = ld_dsmem_f2(&hbuf[r0 * RP + nt * 8 + 2 * cq], q);
          v1 = ld_dsmem_f2(&hbuf[(r0 + 8) * RP + nt * 8 + 2 * cq], q);
        }
        s0.x += v0.x; s0.y += v0.y; s1.x += v1.x; s1.y += v1.y;
      }
      hacc[nt][0] = s0.x; hacc[nt][1] = s0.y; hacc[nt][2] = s1.x; hacc[nt][3] = s1.y;
    }
    write_blob_rows<RP>(blob, w, gq, cq, hacc);
  }
  for (int q = 0; q < cs; ++q)
    if (q != (int)c) mbar_arrive_remote(hdone, q);
  wait_all<true>(hdone, 0);
}

// =============================================================================
// Column pass for dX and dA.  CTA (kb, ms) owns the 64 columns k0 = 64*kb of X
// and dX and walks its share of the 64-row tiles.  Per tile the four consumer
// warps split the 64 x 64 tile into 2 x 2 quarters (m-half mh, k-half kh):
//   dX[mh, kh]  = s * dyb[mh, :] * Ac[:, kh]^T   (written over the X quarter)
//   dA[kh, :]  += X[mh, kh]^T * dyb[mh, :]       (fp32 in registers)
// so every warp reads and writes only its own quarter and no barrier is needed;
// dyb arrives as the row pass's hi/lo blob.  At the end the two m-halves of dA
// are summed, the CTA's partial goes to the workspace, and the last CTA of the
// column block (atomic ticket, no waiting) sums the msplit partials in order
// and writes dA.
// =============================================================================
template <int RP>
struct ColCfg {
  static constexpr int BLOB = blob_bytes<RP>();
  static constexpr int STAGE = TILE_BYTES + BLOB;
  static constexpr int NS = stages_for(STAGE, 3, 8);
  static constexpr int SMALL = RP * 128;       // Ac tile
  static constexpr int RED = 64 * RP * 4;      // cross-warp dA sum
  static constexpr int BYTES = 1024 + NS * STAGE + SMALL + RED + 8 * (3 * NS + 1) + 16;
};

template <int RP, bool kAccX>   // kAccX: dX += the update (p.dx_old), else dX = the update
__global__ void __launch_bounds__(NTHREADS_LS) colpass_dxda_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                   const __grid_constant__ CUtensorMap tmA,
                                                                   const __grid_constant__ CUtensorMap tmDX,
                                                                   ColArgs p) {
  using C = ColCfg<RP>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *atile = smem + NS * C::STAGE;
  float *red = reinterpret_cast<float *>(atile + C::SMALL);
  uint64_t *full = reinterpret_cast<uint64_t *>(atile + C::SMALL + C::RED);
  uint64_t *done = full + NS;
  uint64_t *freeb = done + NS;
  uint64_t *abar = freeb + NS;
  int *s_last = reinterpret_cast<int *>(abar + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = blockIdx.x / p.msplit, ms = blockIdx.x % p.msplit;
  const int k0 = kb * BK;
  const int nmt = (p.M + BM - 1) / BM;
  const int t_beg = (int)((int64_t)nmt * ms / p.msplit), t_end = (int)((int64_t)nmt * (ms + 1) / p.msplit);
  const int ntiles = t_end - t_beg;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&done[s], NCW);
      mbar_init(&freeb[s], 1);
    }
    mbar_init(abar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();

  if (warp == NCW) {
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmDX);
      mbar_arrive_expect_tx(abar, C::SMALL);
      tma_load_2d(atile, &tmA, abar, k0, 0);
      for (int g = 0; g < ntiles; ++g) {
        const int s = g % NS;
        if (g >= NS && !mbar_wait(&freeb[s], ((g / NS) & 1) ^ 1)) break;
        uint8_t *st = smem + s * C::STAGE;
        const int t = t_beg + g;
        mbar_arrive_expect_tx(&full[s], C::STAGE);
        tma_load_2d(st, &tmX, &full[s], k0, t * BM);
        bulk_load(st + TILE_BYTES, p.blob + (size_t)t * C::BLOB, C::BLOB, &full[s]);
      }
    }
    pdl_launch_dependents();
    return;
  }
  if (warp == NCW + 1) {
    if (lane == 0)
      storer_run<NS>(ntiles, done, freeb, [&](int g, int s) {
        tma_store_2d(&tmDX, smem + s * C::STAGE, k0, (t_beg + g) * BM);
        return true;
      });
    pdl_launch_dependents();
    return;
  }

  const int w = warp, gq = lane >> 2, cq = lane & 3;
  const int mh = w & 1, kh = w >> 1;
  float dacc[2][RP / 8][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < RP / 8; ++j) dacc[i][j][0] = dacc[i][j][1] = dacc[i][j][2] = dacc[i][j][3] = 0.f;
  bool ok = wait_all(abar, 0);
  const uint32_t ab = smem_u32(atile);
  const float scale = p.scale;
  for (int g = 0; ok && g < ntiles; ++g) {
    const int s = g % NS;
    if (!(ok = wait_all(&full[s], (g / NS) & 1))) break;
    uint8_t *st = smem + s * C::STAGE;
    const uint32_t tb = smem_u32(st), bh = tb + TILE_BYTES, bl = bh + RP * 128;
    // dA rows kh*32 + {0,16}: contraction over the 32 rows of this m-half
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int mrow = mh * 32 + ks * 16;
      uint32_t a[2][4];
      ld_a_t(tb, kh * 32, mrow, tile_off, a[0]);
      ld_a_t(tb, kh * 32 + 16, mrow, tile_off, a[1]);
#pragma unroll
      for (int np = 0; np < RP / 16; ++np) {
        uint32_t bhf[4], blf[4];
        ld_b_kn(bh, np * 16, mrow, lr_off<RP>, bhf);
        ld_b_kn(bl, np * 16, mrow, lr_off<RP>, blf);
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
          mma_bf16(dacc[kt][2 * np], a[kt], bhf[0], bhf[1]);
          mma_bf16(dacc[kt][2 * np], a[kt], blf[0], blf[1]);
          mma_bf16(dacc[kt][2 * np + 1], a[kt], bhf[2], bhf[3]);
          mma_bf16(dacc[kt][2 * np + 1], a[kt], blf[2], blf[3]);
        }
      }
    }
    // dX rows mh*32 + {0,16}, columns kh*32 .. +32
    float acc[2][4][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;
#pragma unroll
    for (int q = 0; q < RP / 16; ++q) {
      uint32_t ah[2][4], al[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        ld_a(bh, mh * 32 + mt * 16, q * 16, lr_off<RP>, ah[mt]);
        ld_a(bl, mh * 32 + mt * 16, q * 16, lr_off<RP>, al[mt]);
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t b[4];
        ld_b_kn(ab, kh * 32 + np * 16, q * 16, rk_off, b);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          mma_bf16(acc[mt][2 * np], ah[mt], b[0], b[1]);
          mma_bf16(acc[mt][2 * np], al[mt], b[0], b[1]);
          mma_bf16(acc[mt][2 * np + 1], ah[mt], b[2], b[3]);
          mma_bf16(acc[mt][2 * np + 1], al[mt], b[2], b[3]);
        }
      }
    }
    __syncwarp();
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int tr = mh * 32 + mt * 16 + gq + 8 * hf, tc = kh * 32 + nt * 8 + 2 * cq;
          uint32_t *dp = reinterpret_cast<uint32_t *>(st + tile_off(tr, tc));
          float v0 = scale * acc[mt][nt][2 * hf], v1 = scale * acc[mt][nt][2 * hf + 1];
          if (kAccX) {
            // accumulate: the pair (row, col), (row, col + 1) of dX before this call
            // (col is even and rows of dX are 16-byte aligned, so the pair is in the row)
            const int64_t row = (int64_t)(t_beg + g) * BM + tr;
            const int col = k0 + tc;
            if (row < p.M && col < p.K) {
              const float2 o = unpack_bf16(*reinterpret_cast<const unsigned int *>(p.dx_old + row * p.lddx + col));
              v0 += o.x;
              v1 += o.y;
            }
          }
          *dp = pack_bf16(v0, v1);
        }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&done[s]);
  }
  pdl_launch_dependents();
  if (!__all_sync(0xffffffffu, ok)) return;

  // sum the two m-halves, write this CTA's partial, ordered reduction by the last CTA
  if (mh == 1) {
#pragma unroll
    for (int kt = 0; kt < 2; ++kt)
#pragma unroll
      for (int nt = 0; nt < RP / 8; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          *reinterpret_cast<float2 *>(&red[(kh * 32 + kt * 16 + gq + 8 * hf) * RP + nt * 8 + 2 * cq]) =
              make_float2(dacc[kt][nt][2 * hf], dacc[kt][nt][2 * hf + 1]);
  }
  named_bar_sync(1, NCW * 32);
  const int64_t kpad = p.nkb * BK;
  float *part = p.part_out + (int64_t)ms * kpad * RP;
  if (mh == 0) {
#pragma unroll
    for (int kt = 0; kt < 2; ++kt)
#pragma unroll
      for (int nt = 0; nt < RP / 8; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int kr = kh * 32 + kt * 16 + gq + 8 * hf;
          const float2 o = *reinterpret_cast<const float2 *>(&red[kr * RP + nt * 8 + 2 * cq]);
          *reinterpret_cast<float2 *>(&part[(int64_t)(k0 + kr) * RP + nt * 8 + 2 * cq]) =
              make_float2(dacc[kt][nt][2 * hf] + o.x, dacc[kt][nt][2 * hf + 1] + o.y);
        }
  }
  __threadfence();
  named_bar_sync(1, NCW * 32);
  if (threadIdx.x == 0) *s_last = (atomicAdd(&p.counters[kb], 1) == p.msplit - 1);
  named_bar_sync(1, NCW * 32);
  if (*s_last) {
    __threadfence();
    for (int e = threadIdx.x; e < BK * RP; e += NCW * 32) {
      const int k = k0 + e / RP, j = e % RP;
      if (k >= p.K || j >= p.r) continue;
      float v = 0.f;
      for (int q = 0; q < p.msplit; ++q) v += __ldcg(&p.part_out[((int64_t)q * kpad + k) * RP + j]);
      const int64_t o = (int64_t)k * p.out_s0 + (int64_t)j * p.out_s1;
      if (p.out_bf16) reinterpret_cast<__nv_bfloat16 *>(p.out)[o] = __float2bfloat16_rn(scale * v);
      else p.out[o] = scale * v;
    }
    if (threadIdx.x == 0) p.counters[kb] = 0;
  }
}

// =============================================================================
// Column pass for dB.  CTA (lb, ms) owns 64 columns l0 = 64*lb of dY and walks
// its share of the 64-row tiles; warp w owns columns l0 + 16w .. +16 and all RP
// rows of dB:  dB[:, l0..] += h[m, :]^T * dY[m, l0..]  with h from the row
// pass's hi/lo blob.  Ordered cross-CTA reduction as for dA.
// =============================================================================
template <int RP>
struct DbCfg {
  static constexpr int BLOB = blob_bytes<RP>();
  static constexpr int STAGE = TILE_BYTES + BLOB;
  static constexpr int NS = stages_for(STAGE, 2, 8);
  static constexpr int BYTES = 1024 + NS * STAGE + 8 * (2 * NS) + 16;
};

template <int RP>
__global__ void __launch_bounds__(NTHREADS) colpass_db_kernel(const __grid_constant__ CUtensorMap tmDY, ColArgs p) {
  using C = DbCfg<RP>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * C::STAGE);
  uint64_t *empty = full + NS;
  int *s_last = reinterpret_cast<int *>(empty + NS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lb = blockIdx.x / p.msplit, ms = blockIdx.x % p.msplit;
  const int l0 = lb * BK;
  const int nmt = (p.M + BM - 1) / BM;
  const int t_beg = (int)((int64_t)nmt * ms / p.msplit), t_end = (int)((int64_t)nmt * (ms + 1) / p.msplit);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();

  if (warp == NCW) {
    if (lane == 0) {
      prefetch_tmap(&tmDY);
      int g = 0;
      for (int t = t_beg; t < t_end; ++t, ++g) {
        const int s = g % NS;
        if (g >= NS && !mbar_wait(&empty[s], ((g / NS) & 1) ^ 1)) break;
        uint8_t *st = smem + s * C::STAGE;
        mbar_arrive_expect_tx(&full[s], C::STAGE);
        tma_load_2d(st, &tmDY, &full[s], l0, t * BM);
        bulk_load(st + TILE_BYTES, p.blob + (size_t)t * C::BLOB, C::BLOB, &full[s]);
      }
    }
    pdl_launch_dependents();
    return;
  }

  const int w = warp, gq = lane >> 2, cq = lane & 3;
  float acc[RP / 16][2][4];
#pragma unroll
  for (int i = 0; i < RP / 16; ++i)
#pragma unroll
    for (int n = 0; n < 2; ++n) acc[i][n][0] = acc[i][n][1] = acc[i][n][2] = acc[i][n][3] = 0.f;
  bool ok = true;
  int g = 0;
  for (int t = t_beg; t < t_end; ++t, ++g) {
    const int s = g % NS;
    if (!(ok = wait_all(&full[s], (g / NS) & 1))) break;
    const uint32_t tb = smem_u32(smem + s * C::STAGE), hb = tb + TILE_BYTES, lbb = hb + RP * 128;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t b[4];
      ld_b_kn(tb, 16 * w, kk * 16, tile_off, b);   // dY columns l0+16w .. +16, contraction rows
#pragma unroll
      for (int mt = 0; mt < RP / 16; ++mt) {
        uint32_t ah[4], al[4];
        ld_a_t(hb, mt * 16, kk * 16, lr_off<RP>, ah);
        ld_a_t(lbb, mt * 16, kk * 16, lr_off<RP>, al);
        mma_bf16(acc[mt][0], ah, b[0], b[1]);
        mma_bf16(acc[mt][0], al, b[0], b[1]);
        mma_bf16(acc[mt][1], ah, b[2], b[3]);
        mma_bf16(acc[mt][1], al, b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  pdl_launch_dependents();
  if (!__all_sync(0xffffffffu, ok)) return;

  const int64_t lpad = p.nkb * BK;
  float *part = p.part_out + (int64_t)ms * RP * lpad;
#pragma unroll
  for (int mt = 0; mt < RP / 16; ++mt)
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int j = mt * 16 + gq + 8 * hf;
        const int l = l0 + 16 * w + n * 8 + 2 * cq;
        *reinterpret_cast<float2 *>(&part[(int64_t)j * lpad + l]) =
            make_float2(acc[mt][n][2 * hf], acc[mt][n][2 * hf + 1]);
      }
  __threadfence();
  named_bar_sync(1, NCW * 32);
  if (threadIdx.x == 0) *s_last = (atomicAdd(&p.counters[lb], 1) == p.msplit - 1);
  named_bar_sync(1, NCW * 32);
  if (*s_last) {
    __threadfence();
    const float scale = p.scale;
    for (int e = threadIdx.x; e < RP * BK; e += NCW * 32) {
      const int j = e / BK, l = l0 + e % BK;
      if (j >= p.r || l >= p.K) continue;   // p.K holds L for this kernel
      float v = 0.f;
      for (int q = 0; q < p.msplit; ++q) v += __ldcg(&p.part_out[((int64_t)q * RP + j) * lpad + l]);
      const int64_t o = (int64_t)j * p.out_s0 + (int64_t)l * p.out_s1;
      if (p.out_bf16) reinterpret_cast<__nv_bfloat16 *>(p.out)[o] = __float2bfloat16_rn(scale * v);
      else p.out[o] = scale * v;
    }
    if (threadIdx.x == 0) p.counters[lb] = 0;
  }
}

// =============================================================================
// Helpers: strided 2-D copy into a dense bf16 layout (packing A / B), fills.
// =============================================================================
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

namespace {

CUtensorMapSwizzle swz_for(int row_bytes) {
  return row_bytes >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
         : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                           : CU_TENSOR_MAP_SWIZZLE_32B;
}

// Big row-major bf16 operand [rows][cols] with row stride ld: 64x64 boxes.
bool map_big(CUtensorMap *m, const void *p, int64_t rows, int64_t cols, int64_t ld) {
  uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  uint64_t str[1] = {(uint64_t)ld * 2};
  uint32_t box[2] = {64, 64};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// Ac [r][K] (row stride lda): boxes of 64 k x RP rows.
bool map_ac(CUtensorMap *m, const void *p, int64_t K, int r, int64_t lda, int RP) {
  uint64_t dims[2] = {(uint64_t)K, (uint64_t)r};
  uint64_t str[1] = {(uint64_t)lda * 2};
  uint32_t box[2] = {64, (uint32_t)RP};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// Bc [L][r] (row stride ldb): boxes of PW j x 64 rows.
bool map_bc(CUtensorMap *m, const void *p, int64_t L, int r, int64_t ldb, int RP) {
  const int PW = RP < 64 ? RP : 64;
  uint64_t dims[2] = {(uint64_t)r, (uint64_t)L};
  uint64_t str[1] = {(uint64_t)ldb * 2};
  uint32_t box[2] = {(uint32_t)PW, 64};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p, dims, str, box, swz_for(PW * 2));
}
int pick_pow2(int64_t units, int64_t capacity, int maxv) {
  int c = 1;
  while (c * 2 <= maxv && units * c * 2 <= capacity) c *= 2;
  return c;
}

constexpr int kCpMax = 4;        // row-pass cluster size (contraction split)
constexpr int kMsplitMax = 16;   // column-pass split of M

}  // namespace

SingleLayout plan_layout(const SingleArgs &a, bool need_A, bool need_B) {
  SingleLayout lay;
  lay.pack_A = need_A && !(a.sA_k == 1 && (a.sA_r * 2) % 16 == 0 && a.sA_r >= a.K && aligned16(a.A));
  lay.pack_B = need_B && !(a.sB_r == 1 && (a.sB_l * 2) % 16 == 0 && a.sB_l >= a.r && aligned16(a.B));
  lay.lda = lay.pack_A ? round_up(a.K, 8) : a.sA_r;
  lay.ldb = lay.pack_B ? round_up(a.r, 8) : a.sB_l;
  return lay;
}

size_t bf16_ws_bytes(int op, int64_t M, int64_t K, int64_t L, int r) {
  if (M <= 0 || K < 0 || L < 0 || r <= 0) return 0;
  const int RP = rank_bucket(r);
  const size_t packA = ws_round((size_t)r * round_up(K, 8) * 2);
  const size_t packB = ws_round((size_t)L * round_up(r, 8) * 2);
  const size_t blob = ws_round((size_t)ceil_div(M, BM) * RP * 256);   // hi/lo bf16 of dyb or h
  if (op == LORA_OP_FORWARD) return packA + packB;
  if (op == LORA_OP_BACKWARD_DX_DA) {
    const int64_t nkb = ceil_div(K, 64);
    return packA + packB + blob + ws_round((size_t)kMsplitMax * nkb * 64 * RP * 4) + ws_round((size_t)nkb * 4);
  }
  if (op == LORA_OP_BACKWARD_DB) {
    const int64_t nlb = ceil_div(L, 64);
    return packA + blob + ws_round((size_t)kMsplitMax * RP * nlb * 64 * 4) + ws_round((size_t)nlb * 4);
  }
  if (op == LORA_OP_BACKWARD) {
    const int64_t nlb = ceil_div(L, 64);
    return bf16_ws_bytes(LORA_OP_BACKWARD_DX_DA, M, K, L, r) + blob +
           ws_round((size_t)kMsplitMax * RP * nlb * 64 * 4) + ws_round((size_t)nlb * 4);
  }
  return 0;
}

static lora_status_t pack_operands(const SingleArgs &a, const SingleLayout &lay, WsCarver &ws, const void **Ac,
                                   const void **Bc, cudaStream_t st, bool pdl) {
  if (lay.pack_A) {
    void *d = ws.take((size_t)a.r * lay.lda * 2);
    if (!d) return LORA_ERR_WORKSPACE;
    const int64_t n = (int64_t)a.r * a.K;
    int blocks = (int)std::min<int64_t>(ceil_div(n, 256), 4 * num_sms());
    if (blocks < 1) blocks = 1;
    LORA_CUDA(launch(pack2d_bf16_kernel, dim3(blocks), dim3(256), 0, st, 1, pdl,
                     (const __nv_bfloat16 *)a.A, (int64_t)a.sA_r, (int64_t)a.sA_k, a.r, (int)a.K,
                     (__nv_bfloat16 *)d, (int64_t)lay.lda));
    *Ac = d;
    pdl = true;
  } else if (Ac) {
    *Ac = a.A;
  }
  if (lay.pack_B) {
    void *d = ws.take((size_t)a.L * lay.ldb * 2);
    if (!d) return LORA_ERR_WORKSPACE;
    const int64_t n = (int64_t)a.r * a.L;
    int blocks = (int)std::min<int64_t>(ceil_div(n, 256), 4 * num_sms());
    if (blocks < 1) blocks = 1;
    LORA_CUDA(launch(pack2d_bf16_kernel, dim3(blocks), dim3(256), 0, st, 1, pdl,
                     (const __nv_bfloat16 *)a.B, (int64_t)a.sB_l, (int64_t)a.sB_r, (int)a.L, a.r,
                     (__nv_bfloat16 *)d, (int64_t)lay.ldb));
    *Bc = d;
  } else if (Bc) {
    *Bc = a.B;
  }
  return LORA_OK;
}

template <int RP>
static lora_status_t forward_rp(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  SingleLayout lay = plan_layout(a, true, a.L > 0);
  WsCarver carver(ws, ws_bytes);
  const void *Ac = nullptr, *Bc = nullptr;
  LORA_TRY(pack_operands(a, lay, carver, &Ac, &Bc, st, true));
  CUtensorMap tX, tA, tB, tY;
  if (!map_big(&tX, a.X, a.M, a.K, a.ldx) || !map_ac(&tA, Ac, a.K, a.r, lay.lda, RP)) return LORA_ERR_ALIGNMENT;
  if (a.L == 0) {
    // h only (lora_forward_h with no output columns): no Y or B tile is ever loaded
    tB = tA;
    tY = tX;
  } else if (!map_bc(&tB, Bc, a.L, a.r, lay.ldb, RP) || !map_big(&tY, a.Y, a.M, a.L, a.ldy)) {
    return LORA_ERR_ALIGNMENT;
  }
  auto kern = fwd_bf16_kernel<RP>;
  const size_t smem = FwdCfg<RP>::BYTES;
  LORA_CUDA(ensure_smem((const void *)kern, smem));
  const int occ = occupancy((const void *)kern, NTHREADS_LS, smem);
  const int64_t nrb = ceil_div(a.M, BM);
  const int64_t nk = ceil_div(a.K, BK), nl = ceil_div(a.L, BK);
  int cl = pick_pow2(nrb, (int64_t)occ * num_sms(), 8);
  while (cl > 1 && (nk < cl || nl < cl)) cl /= 2;
  FwdArgs p{(int)a.M, (int)a.K, (int)a.L, a.scale, cl, a.h, a.ldh, a.r};
  LORA_CUDA(launch(kern, dim3((unsigned)(nrb * cl)), dim3(NTHREADS_LS), smem, st, cl, true, tX, tA, tB, tY, p));
  return LORA_OK;
}

lora_status_t forward_bf16(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  switch (rank_bucket(a.r)) {
    case 16: return forward_rp<16>(a, ws, ws_bytes, st);
    case 32: return forward_rp<32>(a, ws, ws_bytes, st);
    case 64: return forward_rp<64>(a, ws, ws_bytes, st);
    default: return forward_rp<128>(a, ws, ws_bytes, st);
  }
}

// Row pass for dyb (kW_KN) or h: writes the hi/lo blob.
template <int RP, bool kW_KN>
static lora_status_t launch_rows(const void *in, int64_t ld_in, int64_t Kc, const CUtensorMap &tW, int64_t M,
                                 uint8_t *blob, int *counters, int ncounters, cudaStream_t st) {
  CUtensorMap tIn;
  if (!map_big(&tIn, in, M, Kc, ld_in)) return LORA_ERR_ALIGNMENT;
  auto kern = rows_bf16_kernel<RP, kW_KN>;
  const size_t smem = RowsCfg<RP>::BYTES;
  LORA_CUDA(ensure_smem((const void *)kern, smem));
  const int occ = occupancy((const void *)kern, NTHREADS, smem);
  const int64_t nrb = ceil_div(M, BM);
  int cp = pick_pow2(nrb, (int64_t)occ * num_sms(), kCpMax);
  while (cp > 1 && ceil_div(Kc, BK) < cp) cp /= 2;
  RowsArgs p{(int)M, (int)Kc, cp, blob, counters, ncounters};
  LORA_CUDA(launch(kern, dim3((unsigned)(nrb * cp)), dim3(NTHREADS), smem, st, cp, true, tIn, tW, p));
  return LORA_OK;
}

static int choose_msplit(int64_t ncol_blocks, int64_t M, const void *kern, int threads, size_t smem) {
  const int occ = occupancy(kern, threads, smem);
  const int64_t cap = (int64_t)occ * num_sms();
  int64_t ms = cap / std::max<int64_t>(ncol_blocks, 1);
  ms = std::min<int64_t>(ms, kMsplitMax);
  ms = std::min<int64_t>(ms, ceil_div(M, BM));
  return (int)std::max<int64_t>(ms, 1);
}

template <int RP>
static lora_status_t dxda_rp(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  SingleLayout lay = plan_layout(a, true, true);
  WsCarver carver(ws, ws_bytes);
  const void *Ac = nullptr, *Bc = nullptr;
  LORA_TRY(pack_operands(a, lay, carver, &Ac, &Bc, st, true));
  const int64_t nkb = ceil_div(a.K, BK);
  CUtensorMap tA, tB;
  if (!map_ac(&tA, Ac, a.K, a.r, lay.lda, RP) || !map_bc(&tB, Bc, a.L, a.r, lay.ldb, RP))
    return LORA_ERR_ALIGNMENT;
  uint8_t *blob = (uint8_t *)carver.take((size_t)ceil_div(a.M, BM) * RP * 256);
  float *partA = (float *)carver.take((size_t)kMsplitMax * nkb * 64 * RP * 4);
  int *counters = (int *)carver.take((size_t)nkb * 4);
  if (!blob || !partA || !counters) return LORA_ERR_WORKSPACE;
  LORA_TRY((launch_rows<RP, true>(a.dY, a.lddy, a.L, tB, a.M, blob, counters, (int)nkb, st)));

  auto kern = a.dx_acc ? colpass_dxda_kernel<RP, true> : colpass_dxda_kernel<RP, false>;
  const size_t smem = ColCfg<RP>::BYTES;
  LORA_CUDA(ensure_smem((const void *)kern, smem));
  const int ms = choose_msplit(nkb, a.M, (const void *)kern, NTHREADS_LS, smem);
  CUtensorMap tX, tDX;
  if (!map_big(&tX, a.X, a.M, a.K, a.ldx) || !map_big(&tDX, a.dX, a.M, a.K, a.lddx)) return LORA_ERR_ALIGNMENT;
  ColArgs p{};
  p.M = (int)a.M;
  p.K = (int)a.K;
  p.r = a.r;
  p.msplit = ms;
  p.nkb = (int)nkb;
  p.scale = a.scale;
  p.part_out = partA;
  p.counters = counters;
  p.out = a.dA;
  p.out_s0 = a.sdA_k;
  p.out_s1 = a.sdA_r;
  p.out_bf16 = a.grad_lo;
  p.blob = blob;
  p.dx_old = a.dx_acc ? (const __nv_bfloat16 *)a.dX : nullptr;
  p.lddx = a.lddx;
  LORA_CUDA(launch(kern, dim3((unsigned)(nkb * ms)), dim3(NTHREADS_LS), smem, st, 1, true, tX, tA, tDX, p));
  return LORA_OK;
}

lora_status_t backward_dx_da_bf16(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  switch (rank_bucket(a.r)) {
    case 16: return dxda_rp<16>(a, ws, ws_bytes, st);
    case 32: return dxda_rp<32>(a, ws, ws_bytes, st);
    case 64: return dxda_rp<64>(a, ws, ws_bytes, st);
    default: return dxda_rp<128>(a, ws, ws_bytes, st);
  }
}

template <int RP>
static lora_status_t launch_colpass_db(const SingleArgs &a, const uint8_t *blob, float *partB, int *counters,
                                       cudaStream_t st);

template <int RP>
static lora_status_t db_rp(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  SingleLayout lay = plan_layout(a, true, false);
  WsCarver carver(ws, ws_bytes);
  const void *Ac = nullptr;
  LORA_TRY(pack_operands(a, lay, carver, &Ac, nullptr, st, true));
  const int64_t nlb = ceil_div(a.L, BK);
  CUtensorMap tA;
  if (!map_ac(&tA, Ac, a.K, a.r, lay.lda, RP)) return LORA_ERR_ALIGNMENT;
  uint8_t *blob = (uint8_t *)carver.take((size_t)ceil_div(a.M, BM) * RP * 256);
  float *partB = (float *)carver.take((size_t)kMsplitMax * RP * nlb * 64 * 4);
  int *counters = (int *)carver.take((size_t)nlb * 4);
  if (!blob || !partB || !counters) return LORA_ERR_WORKSPACE;
  LORA_TRY((launch_rows<RP, false>(a.X, a.ldx, a.K, tA, a.M, blob, counters, (int)nlb, st)));
  return launch_colpass_db<RP>(a, blob, partB, counters, st);
}

// dB = s * h^T * dY from the h blob (the column pass of lora_backward_db).
template <int RP>
static lora_status_t launch_colpass_db(const SingleArgs &a, const uint8_t *blob, float *partB, int *counters,
                                       cudaStream_t st) {
  const int64_t nlb = ceil_div(a.L, BK);
  auto kern = colpass_db_kernel<RP>;
  const size_t smem = DbCfg<RP>::BYTES;
  LORA_CUDA(ensure_smem((const void *)kern, smem));
  const int ms = choose_msplit(nlb, a.M, (const void *)kern, NTHREADS, smem);
  CUtensorMap tDY;
  if (!map_big(&tDY, a.dY, a.M, a.L, a.lddy)) return LORA_ERR_ALIGNMENT;
  ColArgs p{};
  p.M = (int)a.M;
  p.K = (int)a.L;
  p.r = a.r;
  p.msplit = ms;
  p.nkb = (int)nlb;
  p.scale = a.scale;
  p.part_out = partB;
  p.counters = counters;
  p.out = a.dB;
  p.out_bf16 = a.grad_lo;
  p.out_s0 = a.sdB_r;
  p.out_s1 = a.sdB_l;
  p.blob = const_cast<uint8_t *>(blob);
  LORA_CUDA(launch(kern, dim3((unsigned)(nlb * ms)), dim3(NTHREADS), smem, st, 1, true, tDY, p));
  return LORA_OK;
}

// lora_backward: the dX / dA passes of lora_backward_dx_da, then dB from the saved h.
template <int RP>
static lora_status_t backward_rp(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  const size_t n1 = bf16_ws_bytes(LORA_OP_BACKWARD_DX_DA, a.M, a.K, a.L, a.r);
  if (ws_bytes < n1) return LORA_ERR_WORKSPACE;
  LORA_TRY(dxda_rp<RP>(a, ws, n1, st));
  WsCarver carver(static_cast<char *>(ws) + n1, ws_bytes - n1);
  const int64_t nlb = ceil_div(a.L, BK), nrb = ceil_div(a.M, BM);
  uint8_t *blob = (uint8_t *)carver.take((size_t)nrb * RP * 256);
  float *partB = (float *)carver.take((size_t)kMsplitMax * RP * nlb * 64 * 4);
  int *counters = (int *)carver.take((size_t)nlb * 4);
  if (!blob || !partB || !counters) return LORA_ERR_WORKSPACE;
  LORA_CUDA(launch(hblob_kernel<RP>, dim3((unsigned)nrb), dim3(256), 0, st, 1, true, (const float *)a.h, a.ldh, a.M,
                   a.r, blob, counters, (int)nlb));
  return launch_colpass_db<RP>(a, blob, partB, counters, st);
}

lora_status_t backward_bf16(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  switch (rank_bucket(a.r)) {
    case 16: return backward_rp<16>(a, ws, ws_bytes, st);
    case 32: return backward_rp<32>(a, ws, ws_bytes, st);
    case 64: return backward_rp<64>(a, ws, ws_bytes, st);
    default: return backward_rp<128>(a, ws, ws_bytes, st);
  }
}

lora_status_t backward_db_bf16(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  switch (rank_bucket(a.r)) {
    case 16: return db_rp<16>(a, ws, ws_bytes, st);
    case 32: return db_rp<32>(a, ws, ws_bytes, st);
    case 64: return db_rp<64>(a, ws, ws_bytes, st);
    default: return db_rp<128>(a, ws, ws_bytes, st);
  }
}

int read_clear_error_single_bf16() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
  return v;
}

}  // namespace lora
