// multi.cu -- multi-adapter (serving) LoRA ops for sm_103a.
//
// Operations (mstar page "mstar.engine.resources.lora.ops"):
//   shrink         h[t, i*R + j] = x[t] . a[slot(t)][i*R + j]            (j < rank)
//   expand_fused   y[t, slice i] += scalings[slot] * h[t, slice i] @ b[slot, slice i]^T
//   apply_linear_  shrink then expand into y
//   gather_shrink  h[t] = a[slot(t)][:, ids[t]]  (ids outside [0, V) give zeros)
// and the integer step in front of them (group_by_slot): a stable counting sort
// of the active tokens by slot and a list of tiles of at most 64 tokens of one
// slot, built on the device with no host sync (the page requires the ops to run
// without one).
//
// shrink_kernel: one (token tile, slice) per cluster of `cl` CTAs; the
// contraction is split over the cluster and the partial h are summed in
// cluster-rank order through distributed shared memory.
// expand_kernel: one (token tile, slice, group of 64-column blocks) per CTA;
// only that slice's h is held in registers, y blocks stream through a ring with
// a loader and a storer warp.
// apply_linear runs both, chained by programmatic dependent launch, with h in
// the workspace (it stays in L2 between the two kernels).
// Rows are gathered (a tile's tokens need not be contiguous) with one 1-D bulk
// copy per row into padded shared-memory rows (conflict-free ldmatrix).
// Adapter padding (rows / columns past a slot's rank, which may hold anything)
// is masked in registers, never trusted.
#include <algorithm>

#include "common.cuh"
#include "host_common.h"
#include "multi.h"

namespace lora {

namespace {

constexpr int MBM = 64;      // token rows per tile
constexpr int KW = 64;       // contraction columns per shrink stage
constexpr int XP = KW * 2 + 16;   // padded row pitch (bytes) of x / a / y rows in shared memory
constexpr int CBW = 64;      // output columns per expand block
constexpr int kMaxHC = 256;  // n * R columns of h held on chip by the shrink

constexpr int EX_CW = 4;     // expand consumer warps (16 rows each)

struct MArgs {
  const int32_t *ranks;
  const float *scal;
  const int *header;   // [0] number of active tokens, [1] number of tiles
  const int4 *tiles;   // (slot, start, len, 0)
  const int32_t *perm;
  int S, R, n, cl, gb, ngroups;
  int64_t in;
  const __nv_bfloat16 *x; int64_t ldx;
  const __nv_bfloat16 *a; int64_t sa_slot, sa_row;
  const __nv_bfloat16 *b; int64_t sb_slot, sb_row;
  float *h; int64_t ldh;
  __nv_bfloat16 *y; int64_t ldy;
  int off[LORA_MAX_SLICES + 1];   // output column offset of each slice
  int tma_ok;                     // the tensor maps of x / y are valid
};

// Byte offset of (row, col) in a 64 x 64 bf16 tile written by TMA with the
// 128-byte swizzle (tile base 1024-byte aligned).
__device__ __forceinline__ uint32_t swz_off(int row, int col) { return swz(row, col * 2, 128); }

// A tile is "dense" when its 64 tokens are consecutive rows: then x / y tiles
// can move as one TMA box instead of 64 gathered rows (LORA_MULTI_TMA selects
// which kernels use that path: bit 0 the shrink, bit 1 the expand).
#ifndef LORA_MULTI_TMA
#define LORA_MULTI_TMA 1
#endif
__device__ __forceinline__ bool dense_tile(const int32_t *perm, int start, int len) {
  return len == 64 && perm[start + 63] - perm[start] == 63;
}

__device__ __forceinline__ uint32_t mask_pair(uint32_t v, int j0, int lim) {
  // keep the bf16 halves whose column j0 (low) / j0 + 1 (high) is below lim
  const uint32_t lo = j0 < lim ? 0x0000ffffu : 0u, hi = j0 + 1 < lim ? 0xffff0000u : 0u;
  return v & (lo | hi);
}

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Warp-uniform bounded wait.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait<kCluster>(bar, parity));
}

// A operand (16x16 at rows r0.., cols c0..) / B operands (two n8 tiles) from padded rows.
__device__ __forceinline__ void lda_p(uint32_t base, int pitch, int r0, int c0, uint32_t (&a)[4]) {
  const int l = lane_id();
  ldsm_x4(base + (r0 + (l & 15)) * pitch + (c0 + ((l >> 4) << 3)) * 2, a[0], a[1], a[2], a[3]);
}
__device__ __forceinline__ void ldb_p(uint32_t base, int pitch, int n0, int k0, uint32_t (&b)[4]) {
  const int l = lane_id();
  ldsm_x4(base + (n0 + (l & 7) + ((l >> 4) << 3)) * pitch + (k0 + (((l >> 3) & 1) << 3)) * 2, b[0], b[1], b[2],
          b[3]);
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace

// =============================================================================
// group_by_slot: one CTA.  Each warp owns a contiguous range of tokens; pass 1
// counts active tokens per (warp, slot) (warp-level __match_any_sync, no
// atomics), a block scan turns the counts into per-(warp, slot) cursors, and
// pass 2 revisits the ranges in the same order and scatters each token to its
// cursor: a stable counting sort by slot.  Tiles of at most `bmt` tokens of one
// slot are listed in slot order.  Slots are read in batches of 8 per lane so
// their loads overlap.
// =============================================================================
__device__ __forceinline__ void block_scan2(int a, int b, int &ea, int &eb, int &ta, int &tb, int *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int va = __shfl_up_sync(0xffffffffu, ia, o), vb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += va;
      ib += vb;
    }
  }
  if (lane == 31) {
    sh[warp] = ia;
    sh[32 + warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    int va = lane < nw ? sh[lane] : 0, vb = lane < nw ? sh[32 + lane] : 0;
    int sa = va, sb = vb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xa = __shfl_up_sync(0xffffffffu, sa, o), xb = __shfl_up_sync(0xffffffffu, sb, o);
      if (lane >= o) {
        sa += xa;
        sb += xb;
      }
    }
    if (lane < nw) {
      sh[64 + lane] = sa - va;
      sh[96 + lane] = sb - vb;
    }
    if (lane == 31) {
      sh[128] = sa;
      sh[129] = sb;
    }
  }
  __syncthreads();
  ea = sh[64 + warp] + ia - a;
  eb = sh[96 + warp] + ib - b;
  ta = sh[128];
  tb = sh[129];
  __syncthreads();
}

constexpr int GU = 8;   // tokens per lane per batch in group_kernel
// Tokens per warp the grouping aims for (fewer warps: shorter scans and barriers).
#ifndef LORA_GROUP_TOKENS_PER_WARP
#define LORA_GROUP_TOKENS_PER_WARP 256
#endif

__global__ void __launch_bounds__(1024) group_kernel(const int32_t *__restrict__ slots, int T, int S, int R,
                                                     const int32_t *__restrict__ ranks, int32_t *counts_out,
                                                     int32_t *perm_out, int32_t *num_active_out, int *header,
                                                     int4 *tiles, int bmt) {
  extern __shared__ int gsm[];
  const int nw = blockDim.x >> 5;
  int *hist = gsm;                 // [nw][S]
  int *srank = gsm + nw * S;       // [S]
  int *sh = srank + S;             // scan scratch (160 ints)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  const int t_lo = (int)((int64_t)T * warp / nw), t_hi = (int)((int64_t)T * (warp + 1) / nw);
  const bool one_batch = t_hi - t_lo <= 32 * GU;   // the warp's slots stay in registers for both passes
  int sv[GU];
#pragma unroll
  for (int u = 0; u < GU; ++u) {
    const int t = t_lo + u * 32 + lane;
    sv[u] = t < t_hi ? slots[t] : -1;
  }
  for (int i = threadIdx.x; i < nw * S; i += blockDim.x) hist[i] = 0;
  for (int i = threadIdx.x; i < S; i += blockDim.x) srank[i] = ranks[i];
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  auto active = [&](int s) { return s >= 0 && s < S && srank[s] >= 1 && srank[s] <= R; };
  for (int t0 = t_lo; t0 < t_hi; t0 += 32 * GU) {
    if (t0 != t_lo) {
#pragma unroll
      for (int u = 0; u < GU; ++u) {
        const int t = t0 + u * 32 + lane;
        sv[u] = t < t_hi ? slots[t] : -1;
      }
    }
#pragma unroll
    for (int u = 0; u < GU; ++u) {
      const bool act = active(sv[u]);
      const unsigned m = __match_any_sync(0xffffffffu, act ? sv[u] : -(lane + 1));
      if (act && (m & lt) == 0) hist[warp * S + sv[u]] += __popc(m);
      __syncwarp();
    }
  }
  __syncthreads();
  int run = 0, trun = 0;
  for (int c0 = 0; c0 < S; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    int cnt = 0;
    if (s < S)
      for (int w = 0; w < nw; ++w) cnt += hist[w * S + s];
    const int nt = (cnt + bmt - 1) / bmt;
    int ec, et, tc, tt;
    block_scan2(cnt, nt, ec, et, tc, tt, sh);
    if (s < S) {
      const int base = run + ec, tb = trun + et;
      counts_out[s] = cnt;
      int cur = base;
      for (int w = 0; w < nw; ++w) {
        const int hcount = hist[w * S + s];
        hist[w * S + s] = cur;
        cur += hcount;
      }
      for (int i = 0; i < nt; ++i) tiles[tb + i] = make_int4(s, base + i * bmt, min(bmt, cnt - i * bmt), 0);
    }
    run += tc;
    trun += tt;
  }
  if (threadIdx.x == 0) {
    *num_active_out = run;
    header[0] = run;
    header[1] = trun;
  }
  __syncthreads();
  for (int t0 = t_lo; t0 < t_hi; t0 += 32 * GU) {
    if (!one_batch) {
#pragma unroll
      for (int u = 0; u < GU; ++u) {
        const int t = t0 + u * 32 + lane;
        sv[u] = t < t_hi ? slots[t] : -1;
      }
    }
#pragma unroll
    for (int u = 0; u < GU; ++u) {
      const int t = t0 + u * 32 + lane;
      const bool act = active(sv[u]);
      const unsigned m = __match_any_sync(0xffffffffu, act ? sv[u] : -(lane + 1));
      int cur = 0;
      if (act) cur = hist[warp * S + sv[u]];
      __syncwarp();
      if (act) {
        perm_out[cur + __popc(m & lt)] = t;
        if ((m & lt) == 0) hist[warp * S + sv[u]] = cur + __popc(m);
      }
      __syncwarp();
    }
  }
  pdl_launch_dependents();
}

// 16-byte asynchronous global -> shared copies (src_bytes < 16 zero-fills the
// rest), and an mbarrier arrival once all of this thread's earlier copies landed.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ uint32_t clamp16(int v) { return v <= 0 ? 0u : v >= 16 ? 16u : (uint32_t)v; }

constexpr int LDW = 2;                 // loader warps (64 threads) of the multi-adapter kernels
constexpr int LDT = LDW * 32;
constexpr int RPT = MBM * 8 / LDT;     // tile rows handled per loader thread (8 sixteen-byte chunks a row)

// =============================================================================
// shrink_kernel: CTA (tile, slice i) computes h[t, i*R + j] = x[t] . a[slot][i*R + j]
// for j < rank.  A cluster of `cl` CTAs splits the contraction (decode tiles are
// few) and sums the partial h in cluster-rank order through distributed shared
// memory.  Four consumer warps own 16 rows each; two loader warps gather the
// tile's x rows (one TMA box when the tile is dense) and the slice's a rows
// with 16-byte cp.async copies.
// =============================================================================
constexpr int SH_CWN = 4;   // shrink consumer warps

template <int RP>
struct ShCfg {
  static constexpr int STAGE = ((MBM + RP) * XP + 1023) / 1024 * 1024;   // x rows + a rows of one slice
  static constexpr int NS = (54 * 1024) / STAGE < 2 ? 2 : (54 * 1024) / STAGE > 6 ? 6 : (54 * 1024) / STAGE;
  static constexpr int BYTES = 1024 + NS * STAGE + 8 * (2 * NS + 2) + 64;
  static constexpr int THREADS = (SH_CWN + LDW) * 32;
  static_assert(MBM * RP * 4 <= NS * STAGE, "the h exchange must fit in the stage ring");
};

template <int RP>
__global__ void __launch_bounds__(ShCfg<RP>::THREADS, RP >= 128 ? 2 : 4)
    shrink_kernel(const __grid_constant__ CUtensorMap tmX, MArgs p) {
  using C = ShCfg<RP>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * C::STAGE);
  uint64_t *empty = full + NS;
  uint64_t *hready = empty + NS, *hdone = hready + 1;
  float *hbuf = reinterpret_cast<float *>(smem);   // the exchange reuses the ring once the loads are over

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cl = p.cl;
  const int item = blockIdx.x / cl;
  const int tile = item / p.n, i = item % p.n;
  pdl_wait();
  if (tile >= p.header[1]) return;   // the whole cluster: beyond the device-side tile count
  const uint32_t crank = cl > 1 ? cluster_ctarank() : 0u;
  const int4 td = p.tiles[tile];
  const int slot = td.x, start = td.y, len = td.z;
  const int rank = p.ranks[slot];
  const bool dense = (LORA_MULTI_TMA & 1) && p.tma_ok && dense_tile(p.perm, start, len);
  const int nk = (int)((p.in + KW - 1) / KW);
  const int k_beg = (int)((int64_t)nk * crank / cl), k_end = (int)((int64_t)nk * (crank + 1) / cl);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], LDT + 1);
      mbar_init(&empty[s], SH_CWN);
    }
    mbar_init(hready, cl > 1 ? SH_CWN * 32 * (cl - 1) : 1);
    mbar_init(hdone, cl > 1 ? SH_CWN * 32 * (cl - 1) : 1);
    fence_barrier_init();
  }
  if (cl > 1) cluster_sync_all(); else __syncthreads();

  if (warp >= SH_CWN) {
    // ---------------------------------------------------------------- loaders (64 threads)
    const int lt = threadIdx.x - SH_CWN * 32;
    const int ch = lt & 7;                         // 16-byte chunk of a row
    const int t0 = p.perm[start];
    if (lt == 0 && dense) prefetch_tmap(&tmX);
    const __nv_bfloat16 *xrow[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      const int r = (lt >> 3) + k * (LDT / 8);
      xrow[k] = r < len ? p.x + (int64_t)p.perm[start + r] * p.ldx : p.x;
    }
    const __nv_bfloat16 *as = p.a + (int64_t)slot * p.sa_slot + (int64_t)i * p.R * p.sa_row;
    for (int g = 0; g < k_end - k_beg; ++g) {
      const int s = g % NS;
      if (g >= NS && !mbar_wait(&empty[s], ((g / NS) & 1) ^ 1)) break;
      uint8_t *st = smem + s * C::STAGE;
      const int64_t k0 = (int64_t)(k_beg + g) * KW;
      const int64_t krem = p.in - k0 < (int64_t)KW ? p.in - k0 : (int64_t)KW;
      const uint32_t nb = clamp16((int)krem * 2 - ch * 16);
      if (dense) {
        if (lt == 0) {
          mbar_arrive_expect_tx(&full[s], MBM * KW * 2);
          tma_load_2d(st, &tmX, &full[s], (int)k0, t0);
        }
      } else {
#pragma unroll
        for (int k = 0; k < RPT; ++k) {
          const int r = (lt >> 3) + k * (LDT / 8);
          cp_async16(st + r * XP + ch * 16, xrow[k] + k0 + ch * 8, r < len ? nb : 0u);
        }
        if (lt == 0) mbar_arrive(&full[s]);
      }
      for (int j = lt >> 3; j < rank; j += LDT / 8)
        cp_async16(st + (MBM + j) * XP + ch * 16, as + (int64_t)j * p.sa_row + k0 + ch * 8, nb);
      cp_async_arrive(&full[s]);
    }
    pdl_launch_dependents();
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int w = warp, gq = lane >> 2, cq = lane & 3;
  const bool live = 16 * w < len;
  float hacc[RP / 8][4];
#pragma unroll
  for (int t = 0; t < RP / 8; ++t) hacc[t][0] = hacc[t][1] = hacc[t][2] = hacc[t][3] = 0.f;
  bool ok = true;
  const int l = lane_id();
  for (int g = 0; g < k_end - k_beg; ++g) {
    const int s = g % NS;
    if (!(ok = wait_all(&full[s], (g / NS) & 1))) break;
    const uint32_t xb = smem_u32(smem + s * C::STAGE), ab = xb + MBM * XP;
    const int64_t k0 = (int64_t)(k_beg + g) * KW;
    if (live) {
#pragma unroll
      for (int kk = 0; kk < KW / 16; ++kk) {
        if (k0 + kk * 16 >= p.in) break;
        uint32_t a[4];
        const int ar = 16 * w + (l & 15), ac = kk * 16 + ((l >> 4) << 3);
        ldsm_x4(xb + (dense ? swz_off(ar, ac) : (uint32_t)(ar * XP + ac * 2)), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int np = 0; np < RP / 16; ++np) {
          if (np * 16 >= rank) break;
          uint32_t b[4];
          ldb_p(ab, XP, np * 16, kk * 16, b);
          mma_bf16(hacc[2 * np], a, b[0], b[1]);
          mma_bf16(hacc[2 * np + 1], a, b[2], b[3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  // columns past the slot's rank come from unloaded (stale) rows of a: zero them
#pragma unroll
  for (int nt = 0; nt < RP / 8; ++nt) {
    const int j = nt * 8 + 2 * cq;
    if (j >= rank) hacc[nt][0] = hacc[nt][2] = 0.f;
    if (j + 1 >= rank) hacc[nt][1] = hacc[nt][3] = 0.f;
  }
  const int r0 = 16 * w + gq;
  if (cl > 1) {
    named_bar_sync(1, SH_CWN * 32);   // every consumer warp is done with the ring
#pragma unroll
    for (int nt = 0; nt < RP / 8; ++nt) {
      *reinterpret_cast<float2 *>(&hbuf[r0 * RP + nt * 8 + 2 * cq]) = make_float2(hacc[nt][0], hacc[nt][1]);
      *reinterpret_cast<float2 *>(&hbuf[(r0 + 8) * RP + nt * 8 + 2 * cq]) = make_float2(hacc[nt][2], hacc[nt][3]);
    }
    for (int q = 0; q < cl; ++q)
      if (q != (int)crank) mbar_arrive_remote(hready, q);
    if (!wait_all<true>(hready, 0)) ok = false;
    if (ok && live && (w % cl) == (int)crank) {
#pragma unroll
      for (int nt = 0; nt < RP / 8; ++nt) {
        float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
        for (int q = 0; q < cl; ++q) {
          float2 v0, v1;
          if (q == (int)crank) {
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
    }
    for (int q = 0; q < cl; ++q)
      if (q != (int)crank) mbar_arrive_remote(hdone, q);
  }
  // h rows < len, columns j < rank of slice i; cluster CTA q writes the warps w % cl == q
  if (ok && live && (w % cl) == (int)crank) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int r = r0 + 8 * hf;
      if (r >= len) continue;
      float *hrow = p.h + (int64_t)p.perm[start + r] * p.ldh + (int64_t)i * p.R;
#pragma unroll
      for (int nt = 0; nt < RP / 8; ++nt) {
        const int j = nt * 8 + 2 * cq;
        if (j + 1 < rank) {
          *reinterpret_cast<float2 *>(&hrow[j]) = make_float2(hacc[nt][2 * hf], hacc[nt][2 * hf + 1]);
        } else if (j < rank) {
          hrow[j] = hacc[nt][2 * hf];
        }
      }
    }
  }
  pdl_launch_dependents();
  if (cl > 1) wait_all<true>(hdone, 0);   // peers are done reading this CTA's ring
}

// =============================================================================
// expand_kernel: CTA (tile, group) adds slice i's product for the 64-column
// blocks [b0, b0 + nb) of that slice:  y[t, c] += scal * sum_{j<rank} h[t, i*R+j] * b[slot][c][j].
// Two loader warps fetch y (one TMA box for a full block of a dense tile, else
// 64 gathered rows with 16-byte cp.async) and the slot's b rows (cp.async); two
// storer warps write y back (one TMA store, or 16-byte stores per row).
// =============================================================================
constexpr int STW = 2;                 // storer warps
constexpr int STT = STW * 32;

template <int RP>
struct ExCfg {
  static constexpr int BPITCH = RP * 2 + 16;                       // b row pitch (bytes)
  static constexpr int STAGE = ((MBM * XP + CBW * BPITCH) + 1023) / 1024 * 1024;
  static constexpr int NS = (72 * 1024) / STAGE < 3 ? 3 : (72 * 1024) / STAGE > 6 ? 6 : (72 * 1024) / STAGE;
  static constexpr int BYTES = 1024 + NS * STAGE + 8 * (3 * NS) + 64;
  static constexpr int THREADS = (EX_CW + LDW + STW) * 32;
};

template <int RP>
__global__ void __launch_bounds__(ExCfg<RP>::THREADS, RP >= 128 ? 2 : 3)
    expand_kernel(const __grid_constant__ CUtensorMap tmY, MArgs p) {
  using C = ExCfg<RP>;
  constexpr int NS = C::NS;
  constexpr int BP = C::BPITCH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * C::STAGE);
  uint64_t *done = full + NS;
  uint64_t *freeb = done + NS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / p.ngroups, grp = blockIdx.x % p.ngroups;
  pdl_wait();
  if (tile >= p.header[1]) return;
  // group -> (slice i, first block b0, number of blocks nb)
  int i = 0, gleft = grp, b0 = 0, nb = 0;
  for (; i < p.n; ++i) {
    const int nblk = (p.off[i + 1] - p.off[i] + CBW - 1) / CBW;
    const int ng = (nblk + p.gb - 1) / p.gb;
    if (gleft < ng) {
      b0 = gleft * p.gb;
      nb = min(p.gb, nblk - b0);
      break;
    }
    gleft -= ng;
  }
  if (i >= p.n || nb <= 0) return;
  const int4 td = p.tiles[tile];
  const int slot = td.x, start = td.y, len = td.z;
  const int rank = p.ranks[slot];
  const int rank8 = (rank + 7) & ~7;
  const int col_end = p.off[i + 1];
  const bool dense = (LORA_MULTI_TMA & 2) && p.tma_ok && dense_tile(p.perm, start, len);
  const int t0 = p.perm[start];
  // block g covers columns [c0, c0 + ocols); it moves by TMA when the tile is dense and the block full
  auto block = [&](int g, int &c0, int &ocols) {
    c0 = p.off[i] + (b0 + g) * CBW;
    ocols = min(CBW, col_end - c0);
    return dense && ocols == CBW;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], LDT + 1);
      mbar_init(&done[s], EX_CW);
      mbar_init(&freeb[s], STW);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp >= EX_CW && warp < EX_CW + LDW) {
    // ---------------------------------------------------------------- loaders (64 threads)
    const int lt = threadIdx.x - EX_CW * 32;
    const int ch = lt & 7;
    if (lt == 0 && dense) prefetch_tmap(&tmY);
    __nv_bfloat16 *yrow[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      const int r = (lt >> 3) + k * (LDT / 8);
      yrow[k] = r < len ? p.y + (int64_t)p.perm[start + r] * p.ldy : p.y;
    }
    const __nv_bfloat16 *bs = p.b + (int64_t)slot * p.sb_slot;
    const int bchunks = rank8 / 8;   // 16-byte chunks of a b row
    for (int g = 0; g < nb; ++g) {
      const int s = g % NS;
      if (g >= NS && !mbar_wait(&freeb[s], ((g / NS) & 1) ^ 1)) break;
      uint8_t *st = smem + s * C::STAGE;
      int c0, ocols;
      if (block(g, c0, ocols)) {
        if (lt == 0) {
          mbar_arrive_expect_tx(&full[s], MBM * CBW * 2);
          tma_load_2d(st, &tmY, &full[s], c0, t0);
        }
      } else {
        const uint32_t nbytes = clamp16(ocols * 2 - ch * 16);
#pragma unroll
        for (int k = 0; k < RPT; ++k) {
          const int r = (lt >> 3) + k * (LDT / 8);
          cp_async16(st + r * XP + ch * 16, yrow[k] + c0 + ch * 8, r < len ? nbytes : 0u);
        }
        if (lt == 0) mbar_arrive(&full[s]);
      }
      for (int it = lt; it < ocols * bchunks; it += LDT) {
        const int cc = it / bchunks, q = it % bchunks;
        cp_async16(st + MBM * XP + cc * BP + q * 16, bs + (int64_t)(c0 + cc) * p.sb_row + q * 8, 16u);
      }
      cp_async_arrive(&full[s]);
    }
    pdl_launch_dependents();
    return;
  }
  if (warp >= EX_CW + LDW) {
    // ---------------------------------------------------------------- storers (64 threads)
    const int tt = threadIdx.x - (EX_CW + LDW) * 32;
    const int ch = tt & 7;
    const bool tma_lane = tt == 0;   // issues the TMA stores and releases their stages
    constexpr int D = (NS - 1) < 2 ? (NS - 1) : 2;
    int pend[D + 1];
    int np = 0;
    __nv_bfloat16 *yrow[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      const int r = (tt >> 3) + k * (STT / 8);
      yrow[k] = r < len ? p.y + (int64_t)p.perm[start + r] * p.ldy : p.y;
    }
    for (int g = 0; g < nb; ++g) {
      const int s = g % NS;
      if (!mbar_wait(&done[s], (g / NS) & 1)) break;
      const uint8_t *st = smem + s * C::STAGE;
      int c0, ocols;
      if (block(g, c0, ocols)) {
        if (tma_lane) {
          tma_store_2d(&tmY, st, c0, t0);
          bulk_commit();
          pend[np++] = g;
          if (np > D) {
            bulk_wait_read<D>();
            mbar_arrive(&freeb[pend[0] % NS]);
            for (int k = 1; k < np; ++k) pend[k - 1] = pend[k];
            --np;
          }
        } else if (lane == 0) {
          mbar_arrive(&freeb[s]);     // the other storer warp has nothing to write
        }
      } else {
        if (ch * 8 < ocols) {
#pragma unroll
          for (int k = 0; k < RPT; ++k) {
            const int r = (tt >> 3) + k * (STT / 8);
            if (r < len)
              *reinterpret_cast<int4 *>(yrow[k] + c0 + ch * 8) = *reinterpret_cast<const int4 *>(st + r * XP + ch * 16);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&freeb[s]);
      }
    }
    if (tma_lane) {
      bulk_wait_read<0>();
      for (int k = 0; k < np; ++k) mbar_arrive(&freeb[pend[k] % NS]);
      bulk_wait_all();
    }
    pdl_launch_dependents();
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int w = warp, gq = lane >> 2, cq = lane & 3;
  const bool live = 16 * w < len;
  // slice i of h for rows 16w.., as bf16 A fragments; columns >= rank are zero.  One
  // bf16 rounding of h (relative error 2^-9 per term) sits well inside what the
  // bf16 result of the add can hold.
  uint32_t ah[RP / 16][4];
  {
    float hv[RP / 8][4];
#pragma unroll
    for (int nt = 0; nt < RP / 8; ++nt) hv[nt][0] = hv[nt][1] = hv[nt][2] = hv[nt][3] = 0.f;
    if (live) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = 16 * w + gq + 8 * hf;
        if (r >= len) continue;
        const float *hrow = p.h + (int64_t)p.perm[start + r] * p.ldh + (int64_t)i * p.R;
#pragma unroll
        for (int nt = 0; nt < RP / 8; ++nt) {
          const int j = nt * 8 + 2 * cq;
          if (j < rank) hv[nt][2 * hf] = __ldg(&hrow[j]);
          if (j + 1 < rank) hv[nt][2 * hf + 1] = __ldg(&hrow[j + 1]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < RP / 16; ++q) {
      ah[q][0] = pack_bf16(hv[2 * q][0], hv[2 * q][1]);
      ah[q][1] = pack_bf16(hv[2 * q][2], hv[2 * q][3]);
      ah[q][2] = pack_bf16(hv[2 * q + 1][0], hv[2 * q + 1][1]);
      ah[q][3] = pack_bf16(hv[2 * q + 1][2], hv[2 * q + 1][3]);
    }
  }
  const float sc = p.scal[slot];
  for (int g = 0; g < nb; ++g) {
    const int s = g % NS;
    if (!wait_all(&full[s], (g / NS) & 1)) break;
    uint8_t *st = smem + s * C::STAGE;
    int c0, ocols;
    const bool tmab = block(g, c0, ocols);
    if (live) {
      const uint32_t bb = smem_u32(st) + MBM * XP;
      float acc[8][4];
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll
      for (int q = 0; q < RP / 16; ++q) {
        if (q * 16 >= rank) break;
        const int j0 = q * 16;
        const bool part = j0 + 16 > rank;   // the b padding past the rank (any value) is masked
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b[4];
          ldb_p(bb, BP, np * 16, j0, b);
          if (part) {
            b[0] = mask_pair(b[0], j0 + 2 * cq, rank);
            b[1] = mask_pair(b[1], j0 + 8 + 2 * cq, rank);
            b[2] = mask_pair(b[2], j0 + 2 * cq, rank);
            b[3] = mask_pair(b[3], j0 + 8 + 2 * cq, rank);
          }
          mma_bf16(acc[2 * np], ah[q], b[0], b[1]);
          mma_bf16(acc[2 * np + 1], ah[q], b[2], b[3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int cc = nt * 8 + 2 * cq;
        if (cc >= ocols) continue;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = 16 * w + gq + 8 * hf;
          if (r >= len) continue;
          uint32_t *yp = reinterpret_cast<uint32_t *>(st + (tmab ? swz_off(r, cc) : (uint32_t)(r * XP + cc * 2)));
          const float2 yv = unpack_bf16(*yp);
          *yp = pack_bf16(yv.x + sc * acc[nt][2 * hf], yv.y + sc * acc[nt][2 * hf + 1]);
        }
      }
    }
    if (tmab) fence_proxy_async_smem();   // the TMA store reads what these threads wrote
    __syncwarp();
    if (lane == 0) mbar_arrive(&done[s]);
  }
  pdl_launch_dependents();
}

// =============================================================================
// gather_shrink: one warp per token; h[t, j] = a[slot][j][id] for j < rank
// (zeros when id is outside [0, V)); an exact copy widened to fp32.
// =============================================================================
__global__ void __launch_bounds__(256) gather_kernel(const int32_t *__restrict__ slots, int T, int S, int R,
                                                     const int32_t *__restrict__ ranks,
                                                     const int64_t *__restrict__ ids, int64_t V,
                                                     const __nv_bfloat16 *__restrict__ a, int64_t sa_slot,
                                                     int64_t sa_row, int64_t sa_col, float *h, int64_t ldh) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += nwarps) {
    const int s = slots[t];
    if (s < 0 || s >= S) continue;
    const int rank = ranks[s];
    if (rank < 1 || rank > R) continue;
    const int64_t id = ids[t];
    const bool valid = id >= 0 && id < V;
    const __nv_bfloat16 *col = a + (int64_t)s * sa_slot + (valid ? id : 0) * sa_col;
    for (int j = lane; j < rank; j += 32)
      h[t * ldh + j] = valid ? __bfloat162float(col[(int64_t)j * sa_row]) : 0.f;
  }
  pdl_launch_dependents();
}


// ----------------------------------------------------------------------------- host side
namespace {

int max_tiles(int64_t T, int S) { return (int)(ceil_div(T, MBM) + std::min<int64_t>(S, T)); }

struct SchedPtrs {
  int *header, *counts;
  int32_t *perm;
  int4 *tiles;
};

size_t sched_bytes(int64_t T, int S) {
  return ws_round(256) + ws_round((size_t)S * 4) + ws_round((size_t)std::max<int64_t>(T, 1) * 4) +
         ws_round((size_t)max_tiles(T, S) * 16);
}
// h of apply_linear, kept between its two kernels (n * R <= kMaxHC columns)
size_t hbuf_bytes(int64_t T, int R) { return ws_round((size_t)T * std::min(kMaxHC, LORA_MAX_SLICES * R) * 4); }

bool carve_sched(WsCarver &c, int64_t T, int S, SchedPtrs &sp) {
  sp.header = (int *)c.take(256);
  sp.counts = (int *)c.take((size_t)S * 4);
  sp.perm = (int32_t *)c.take((size_t)std::max<int64_t>(T, 1) * 4);
  sp.tiles = (int4 *)c.take((size_t)max_tiles(T, S) * 16);
  return sp.header && sp.counts && sp.perm && sp.tiles;
}

lora_status_t launch_group(const lora_addressing_t &ad, const int32_t *ranks, int32_t *counts, int32_t *perm,
                           int32_t *num_active, int *header, int4 *tiles, cudaStream_t st) {
  const int S = ad.num_slots;
  int nw = (int)std::max<int64_t>(1, (160 * 1024 / 4 - 256 - S) / S);   // shared-memory bound
  nw = std::min<int64_t>({nw, 32, std::max<int64_t>(1, ceil_div(ad.num_tokens, LORA_GROUP_TOKENS_PER_WARP))});
  const size_t smem = (size_t)(nw * S + S + 160) * 4;
  LORA_CUDA(ensure_smem((const void *)group_kernel, smem));
  LORA_CUDA(launch(group_kernel, dim3(1), dim3(nw * 32), smem, st, 1, true, ad.slots, ad.num_tokens, S,
                   ad.max_rank, ranks, counts, perm, num_active, header, tiles, (int)MBM));
  return LORA_OK;
}

// 64 x 64 bf16 tiles of a row-major [rows][cols] operand (128-byte swizzle).
bool map_rows(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld) {
  uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  uint64_t str[1] = {(uint64_t)ld * 2};
  uint32_t box[2] = {64, 64};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int RP>
lora_status_t launch_shrink(MArgs a, int64_t T, cudaStream_t st) {
  auto kern = shrink_kernel<RP>;
  const size_t smem = ShCfg<RP>::BYTES;
  LORA_CUDA(ensure_smem((const void *)kern, smem));
  CUtensorMap tmX;
  a.tma_ok = map_rows(&tmX, a.x, T, a.in, a.ldx) ? 1 : 0;
  const int occ = occupancy((const void *)kern, ShCfg<RP>::THREADS, smem);
  const int64_t items = (int64_t)max_tiles(T, a.S) * a.n, cap = (int64_t)occ * num_sms();
  int cl = 1;
  while (cl * 2 <= 8 && items * cl * 2 <= cap) cl *= 2;
  while (cl > 1 && ceil_div(a.in, KW) < cl) cl /= 2;
  a.cl = cl;
  LORA_CUDA(launch(kern, dim3((unsigned)(items * cl)), dim3(ShCfg<RP>::THREADS), smem, st, cl, true, tmX, a));
  return LORA_OK;
}

lora_status_t dispatch_shrink(const MArgs &a, int64_t T, cudaStream_t st) {
  switch (rank_bucket(a.R)) {
    case 16: return launch_shrink<16>(a, T, st);
    case 32: return launch_shrink<32>(a, T, st);
    case 64: return launch_shrink<64>(a, T, st);
    default: return launch_shrink<128>(a, T, st);
  }
}

template <int RP>
lora_status_t launch_expand(MArgs a, int64_t T, cudaStream_t st) {
  auto kern = expand_kernel<RP>;
  const size_t smem = ExCfg<RP>::BYTES;
  LORA_CUDA(ensure_smem((const void *)kern, smem));
  const int occ = occupancy((const void *)kern, ExCfg<RP>::THREADS, smem);
  const int64_t tiles = max_tiles(T, a.S), cap = (int64_t)occ * num_sms();
  int64_t blocks = 0;
  for (int i = 0; i < a.n; ++i) blocks += ceil_div(a.off[i + 1] - a.off[i], CBW);
  // column blocks per CTA: about three waves of CTAs over the tile bound
  const int64_t gb = std::max<int64_t>(1, ceil_div(tiles * blocks, 3 * cap));
  int64_t ng = 0;
  for (int i = 0; i < a.n; ++i) ng += ceil_div(ceil_div(a.off[i + 1] - a.off[i], CBW), gb);
  if (ng == 0) return LORA_OK;
  a.gb = (int)gb;
  a.ngroups = (int)ng;
  CUtensorMap tmY;
  a.tma_ok = map_rows(&tmY, a.y, T, a.off[a.n], a.ldy) ? 1 : 0;
  LORA_CUDA(launch(kern, dim3((unsigned)(tiles * ng)), dim3(ExCfg<RP>::THREADS), smem, st, 1, true, tmY, a));
  return LORA_OK;
}

lora_status_t dispatch_expand(const MArgs &a, int64_t T, cudaStream_t st) {
  switch (rank_bucket(a.R)) {
    case 16: return launch_expand<16>(a, T, st);
    case 32: return launch_expand<32>(a, T, st);
    case 64: return launch_expand<64>(a, T, st);
    default: return launch_expand<128>(a, T, st);
  }
}

// Argument checks of the segmented ops beyond those of the ABI layer.
lora_status_t check_seg(const MultiArgs &m, bool need_in, bool need_out) {
  const int R = m.addr.max_rank;
  if ((int64_t)m.n * R > kMaxHC) return LORA_ERR_UNSUPPORTED;
  if (R % 8 != 0) return LORA_ERR_UNSUPPORTED;
  if (need_in && m.in % 8 != 0) return LORA_ERR_UNSUPPORTED;
  if (need_out) {
    for (int i = 0; i < m.n; ++i)
      if (m.out_slices[i] % 8 != 0) return LORA_ERR_UNSUPPORTED;
    if (m.sb_col != 1) return LORA_ERR_UNSUPPORTED;   // b rows must be contiguous along the rank
    if (!aligned16(m.b) || (m.sb_row * 2) % 16 != 0 || (m.sb_slot * 2) % 16 != 0) return LORA_ERR_ALIGNMENT;
  }
  return LORA_OK;
}

MArgs margs(const MultiArgs &m, const SchedPtrs &sp) {
  MArgs a{};
  a.ranks = m.ranks;
  a.scal = m.scalings;
  a.header = sp.header;
  a.tiles = sp.tiles;
  a.perm = sp.perm;
  a.S = m.addr.num_slots;
  a.R = m.addr.max_rank;
  a.n = m.n;
  a.in = m.in;
  a.x = (const __nv_bfloat16 *)m.x;
  a.ldx = m.ldx;
  a.a = (const __nv_bfloat16 *)m.a;
  a.sa_slot = m.sa_slot;
  a.sa_row = m.sa_row;
  a.b = (const __nv_bfloat16 *)m.b;
  a.sb_slot = m.sb_slot;
  a.sb_row = m.sb_row;
  a.h = m.h;
  a.ldh = m.ldh;
  a.y = (__nv_bfloat16 *)m.y;
  a.ldy = m.ldy;
  int off = 0;
  for (int i = 0; i < m.n; ++i) {
    a.off[i] = off;
    off += m.out_slices[i];
  }
  a.off[m.n] = off;
  return a;
}

lora_status_t schedule(const MultiArgs &m, WsCarver &c, SchedPtrs &sp, cudaStream_t st) {
  if (!carve_sched(c, m.addr.num_tokens, m.addr.num_slots, sp)) return LORA_ERR_WORKSPACE;
  return launch_group(m.addr, m.ranks, sp.counts, sp.perm, sp.header, sp.header, sp.tiles, st);
}

}  // namespace

size_t multi_ws_bytes(int op, int64_t T, int64_t in, int64_t O, int R, int S) {
  (void)in;
  (void)O;
  if (T <= 0) return 0;
  if (op == LORA_OP_GROUP_BY_SLOT || op == LORA_OP_SHRINK || op == LORA_OP_EXPAND) return sched_bytes(T, S);
  if (op == LORA_OP_APPLY_LINEAR) return sched_bytes(T, S) + hbuf_bytes(T, R);
  return 0;
}

lora_status_t group_by_slot(const lora_addressing_t &addr, const int32_t *ranks, int32_t *counts, int32_t *perm,
                            int32_t *num_active, void *ws, size_t ws_bytes, cudaStream_t st) {
  if (addr.num_tokens == 0) {
    // no tokens: every count is zero and no token is active
    LORA_CUDA(cudaMemsetAsync(counts, 0, (size_t)addr.num_slots * 4, st));
    LORA_CUDA(cudaMemsetAsync(num_active, 0, 4, st));
    return LORA_OK;
  }
  WsCarver c(ws, ws_bytes);
  SchedPtrs sp;
  if (!carve_sched(c, addr.num_tokens, addr.num_slots, sp)) return LORA_ERR_WORKSPACE;
  return launch_group(addr, ranks, counts, perm, num_active, sp.header, sp.tiles, st);
}

lora_status_t shrink(MultiArgs m, void *ws, size_t ws_bytes, cudaStream_t st) {
  LORA_TRY(check_seg(m, true, false));
  WsCarver c(ws, ws_bytes);
  SchedPtrs sp;
  LORA_TRY(schedule(m, c, sp, st));
  return dispatch_shrink(margs(m, sp), m.addr.num_tokens, st);
}

lora_status_t expand(MultiArgs m, void *ws, size_t ws_bytes, cudaStream_t st) {
  LORA_TRY(check_seg(m, false, true));
  WsCarver c(ws, ws_bytes);
  SchedPtrs sp;
  LORA_TRY(schedule(m, c, sp, st));
  return dispatch_expand(margs(m, sp), m.addr.num_tokens, st);
}

lora_status_t apply_linear(MultiArgs m, void *ws, size_t ws_bytes, cudaStream_t st) {
  LORA_TRY(check_seg(m, true, true));
  WsCarver c(ws, ws_bytes);
  SchedPtrs sp;
  LORA_TRY(schedule(m, c, sp, st));
  float *h = (float *)c.take(hbuf_bytes(m.addr.num_tokens, m.addr.max_rank));
  if (!h) return LORA_ERR_WORKSPACE;
  MArgs a = margs(m, sp);
  a.h = h;
  a.ldh = (int64_t)m.n * m.addr.max_rank;
  LORA_TRY(dispatch_shrink(a, m.addr.num_tokens, st));
  return dispatch_expand(a, m.addr.num_tokens, st);
}

lora_status_t gather_shrink(MultiArgs m, cudaStream_t st) {
  const int64_t T = m.addr.num_tokens;
  const int64_t blocks = std::min<int64_t>(ceil_div(T, 8), 8 * (int64_t)num_sms());
  LORA_CUDA(launch(gather_kernel, dim3((unsigned)std::max<int64_t>(blocks, 1)), dim3(256), 0, st, 1, true,
                   m.addr.slots, (int)T, m.addr.num_slots, m.addr.max_rank, m.ranks, m.ids, m.in,
                   (const __nv_bfloat16 *)m.a, m.sa_slot, m.sa_row, m.sa_col, m.h, m.ldh));
  return LORA_OK;
}

int read_clear_error_multi() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
  return v;
}

}  // namespace lora
