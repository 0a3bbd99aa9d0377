// multi.cu -- multi-adapter (serving) LoRA ops for sm_103a.
//
// Operations (mstar page "mstar.engine.resources.lora.ops"):
//   shrink         h[t, i*R + j] = x[t] . a[slot(t)][i*R + j]            (j < rank)
//   expand_fused   y[t, slice i] += scalings[slot] * h[t, slice i] @ b[slot, slice i]^T
//   apply_linear_  shrink then expand into y
//   gather_shrink  h[t] = a[slot(t)][:, ids[t]]  (ids outside [0, V) give zeros)
// and the integer step in front of them (group_by_slot): a stable counting sort
// of the active tokens by slot and a list of tiles of at most 128 tokens of one
// slot, built on the device with no host sync (the page requires the ops to run
// without one).
//
// shrink_kernel: one token tile (all slices) per cluster of `cl` CTAs; the
// contraction is split over the cluster and the partial h are summed in
// cluster-rank order through distributed shared memory.
// expand_kernel: one (token tile, slice, group of 64-column blocks) per CTA;
// only that slice's h is held in registers, y blocks stream through a ring with
// a loader and a storer warp.
// apply_linear runs both, chained by programmatic dependent launch, with h in
// the workspace (it stays in L2 between the two kernels).
// Rows of a tile whose tokens are not consecutive are gathered with 16-byte
// cp.async copies; consecutive rows and the adapter rows move as TMA boxes.
// Adapter padding (rows / columns past a slot's rank, which may hold anything)
// is masked in registers, never trusted.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "host_common.h"
#include "multi.h"
#include "decode.h"

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
  int tma_a;                      // the tensor map of a is valid (shrink)
  int sh_ns, sh_stage;            // shrink: stages in the ring, bytes per stage
  int nk;                         // shrink: stages (64 columns of `in`) per tile
  int T;                          // number of tokens (rows of x)
  int tc_cols;                    // shrink: tensor-memory columns of the accumulator
  int a_one_slot;                 // shrink: the adapter map has one slot (slot stride 0)
  int nsub;                       // expand: 64-row sub-tiles per tile
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

// Warp-uniform bounded wait: lane 0 polls the barrier, the warp barrier then
// orders what lane 0 observed before every lane's later reads.
#ifndef LORA_POLL_ONE
#define LORA_POLL_ONE 1
#endif
template <bool kCluster = false>
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
#if LORA_POLL_ONE
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait<kCluster>(bar, parity);
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
#else
  return __all_sync(0xffffffffu, mbar_wait<kCluster>(bar, parity));
#endif
}

// B operands (two n8 tiles) from padded rows.
__device__ __forceinline__ void ldb_p(uint32_t base, int pitch, int n0, int k0, uint32_t (&b)[4]) {
  const int l = lane_id();
  ldsm_x4(base + (n0 + (l & 7) + ((l >> 4) << 3)) * pitch + (k0 + (((l >> 3) & 1) << 3)) * 2, b[0], b[1], b[2],
          b[3]);
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace

// Lanes holding the same key (a warp-wide match; the common case where all 32
// lanes agree is checked first with one vote).
__device__ __forceinline__ unsigned same_key_lanes(int key) {
  const int k0 = __shfl_sync(0xffffffffu, key, 0);
  if (__all_sync(0xffffffffu, key == k0)) return 0xffffffffu;
  return __match_any_sync(0xffffffffu, key);
}

// =============================================================================
// group_by_slot: one CTA.  Each warp owns a contiguous range of tokens; pass 1
// counts active tokens per (warp, slot) (warp-level __match_any_sync, no
// atomics), a block scan turns the counts into per-(warp, slot) cursors, and
// pass 2 revisits the ranges in the same order and scatters each token to its
// cursor: a stable counting sort by slot.  Tiles of at most `bmt` tokens of one
// slot are listed in slot order.  Slots are read in batches of 8 per lane so
// their loads overlap.
// =============================================================================
// Exclusive block-wide scan of three values per thread: e[k] the sum over the
// threads before this one, t[k] the block total.  sh: 3 * 64 + 3 ints.
__device__ __forceinline__ void block_scan3(const int (&v)[3], int (&e)[3], int (&t)[3], int *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int in[3] = {v[0], v[1], v[2]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int x = __shfl_up_sync(0xffffffffu, in[k], o);
      if (lane >= o) in[k] += x;
    }
  }
  if (lane == 31)
#pragma unroll
    for (int k = 0; k < 3; ++k) sh[32 * k + warp] = in[k];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int w = lane < nw ? sh[32 * k + lane] : 0;
      int sc = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, sc, o);
        if (lane >= o) sc += x;
      }
      if (lane < nw) sh[96 + 32 * k + lane] = sc - w;
      if (lane == 31) sh[192 + k] = sc;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    e[k] = sh[96 + 32 * k + warp] + in[k] - v[k];
    t[k] = sh[192 + k];
  }
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
                                                     int4 *tiles, int bmt, int *zero, int nzero) {
  extern __shared__ int gsm[];
  const int nw = blockDim.x >> 5;
  int *hist = gsm;                 // [S][nw]: a slot's warp counts contiguous
  int *srank = gsm + nw * S;       // [S]
  int *scnt = srank + S;           // [S] active tokens of each slot
  int *sbase = scnt + S;           // [S] first position of each slot in the permutation
  int *sh = sbase + S;             // scan scratch (224 ints)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  // the tickets of the kernel that follows start at zero
  for (int k = threadIdx.x; k < nzero; k += blockDim.x) zero[k] = 0;
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
      // inactive lanes share one class (fewer distinct values: a faster match)
      const bool act = active(sv[u]);
      const unsigned m = same_key_lanes(act ? sv[u] : -1);
      if (act && (m & lt) == 0) hist[sv[u] * nw + warp] += __popc(m);
      __syncwarp();
    }
  }
  __syncthreads();
  // per slot, a warp scans the warps' counts (lane w: warp w): hist becomes each
  // warp's offset inside the slot, scnt the slot's total
  for (int s = warp; s < S; s += nw) {
    const int v = lane < nw ? hist[s * nw + lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    if (lane < nw) hist[s * nw + lane] = inc - v;
    if (lane == 31) scnt[s] = inc;
  }
  __syncthreads();
  // tile t = (slot, start, len, rows): rows = the sum over the tiles before t of
  // round8(rank), the adapter rows per slice that a contraction over those
  // tiles reads (the cost weights of the stream-K shrink)
  int run = 0, trun = 0, rrun = 0;
  for (int c0 = 0; c0 < S; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    const int cnt = s < S ? scnt[s] : 0;
    const int nt = (cnt + bmt - 1) / bmt;
    const int r8 = cnt > 0 ? (srank[s] + 7) & ~7 : 0;
    const int v[3] = {cnt, nt, nt * r8};
    int e[3], tot[3];
    block_scan3(v, e, tot, sh);
    if (s < S) {
      const int base = run + e[0], tb = trun + e[1], rb = rrun + e[2];
      counts_out[s] = cnt;
      sbase[s] = base;
      for (int i = 0; i < nt; ++i)
        tiles[tb + i] = make_int4(s, base + i * bmt, min(bmt, cnt - i * bmt), rb + i * r8);
    }
    run += tot[0];
    trun += tot[1];
    rrun += tot[2];
  }
  if (threadIdx.x == 0) {
    *num_active_out = run;
    header[0] = run;
    header[1] = trun;
    header[2] = rrun;
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
      const unsigned m = same_key_lanes(act ? sv[u] : -1);
      int cur = 0;
      if (act) cur = sbase[sv[u]] + hist[sv[u] * nw + warp];
      __syncwarp();
      if (act) {
        perm_out[cur + __popc(m & lt)] = t;
        if ((m & lt) == 0) hist[sv[u] * nw + warp] = cur - sbase[sv[u]] + __popc(m);
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
// shrink_kernel: h[t, i*R + j] = x[t] . a[slot][i*R + j] for every slice i and
// j < rank, over the slot-sorted tiles of at most 128 tokens, on the
// fifth-generation tensor cores.  One tile per cluster of `cl` CTAs; CTA q of
// the cluster takes stages [nk q / cl, nk (q + 1) / cl) of the contraction (64
// columns of `in` a stage).  A warp keeps one tensor-copy instruction in flight
// at a time (its lanes' copies run together), so the stages are dealt
// round-robin to several loader warps: x loaders take the tile's 128 x rows (one
// 128-row box when the tile's tokens are consecutive rows, else lane q gathers
// rows 4q..4q+3 with one four-row gather copy), adapter loaders the first rank16
// rows of every slice of a[slot] (lane b: the b-th box of 64, 32 or 16 rows),
// all with the 128-byte swizzle.  Lane 0 of the MMA warp issues four
// 128 x (n * rank16) x 16 MMAs per stage into a tensor-memory accumulator (x read
// once per tile for all slices); warps 4-7 drain it, one token row per thread.
// CTAs q > 0 leave their partial sums in their own shared memory; CTA 0 adds
// them to its own through distributed shared memory in cluster-rank order, so
// the result does not depend on timing.
// =============================================================================
constexpr int TC_M = 128;                  // tokens per tile (accumulator rows)
constexpr int TC_XB = TC_M * KW * 2;       // x bytes of one stage (16 KB)
// Warp roles: x loaders [0, TC_XW), drain [4, 8), the MMA warp, adapter loaders
// [TC_AW0, TC_AW0 + TC_AW).
constexpr int TC_THREADS = 352, TC_XW = 4, TC_MMA_WARP = 8, TC_AW0 = 9, TC_AW = 2;
constexpr int TC_RING = 200 * 1024;
constexpr int TC_BYTES = 1024 + 1024 + TC_RING;

__global__ void __launch_bounds__(TC_THREADS, 1)
    shrink_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXd,
                  const __grid_constant__ CUtensorMap tmA16, const __grid_constant__ CUtensorMap tmA32,
                  const __grid_constant__ CUtensorMap tmA64, MArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = align1024(smem_raw);
  uint64_t *full = reinterpret_cast<uint64_t *>(base);
  uint64_t *empty = full + 16;
  uint64_t *accf = empty + 16;                         // accumulator written
  uint64_t *xready = accf + 1, *xdone = xready + 1;    // partial sums in shared memory / read by CTA 0
  uint64_t *mdone = xdone + 1;                         // every MMA of this CTA has completed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mdone + 1);
  uint8_t *ring = base + 1024;
  float *xbuf = reinterpret_cast<float *>(ring);       // [column][128 rows] once the ring is drained
  const int NS = p.sh_ns, STAGE = p.sh_stage, nk = p.nk, cl = p.cl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / cl;
  const uint32_t q = cl > 1 ? cluster_ctarank() : 0u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    mbar_init(xready, cl > 1 ? 128 * (cl - 1) : 1);   // every drain thread of every other CTA
    mbar_init(xdone, 128);                             // every drain thread of CTA 0
    mbar_init(mdone, 1);
    fence_barrier_init();
  }
  if (warp == TC_MMA_WARP) tmem_alloc(tmem_slot, (uint32_t)p.tc_cols);
  tc_fence_before();
  if (cl > 1) cluster_sync_all(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  const bool any = tile < p.header[1];                // the whole cluster alike
  const int kb = (int)((int64_t)nk * q / cl), ke = (int)((int64_t)nk * (q + 1) / cl);
  const bool has_k = p.in > 0;
  int4 td = make_int4(0, 0, 0, 0);
  int rank = 0;
  if (any) {
    td = p.tiles[tile];
    rank = p.ranks[td.x];
  }
  const int slot = td.x, start = td.y, len = td.z;
  const int r16 = (rank + 15) & ~15, ncols = p.n * r16;

  const bool aw = warp >= TC_AW0 && warp < TC_AW0 + TC_AW;   // adapter loader
  if (any && (warp < TC_XW || aw)) {
    // ---------------------------------------------------------------- loader warps
    const int par = aw ? warp - TC_AW0 : warp, nw = aw ? TC_AW : TC_XW;   // stages s % nw == par
    if (lane == 0 && has_k) {
      if (aw) {
        prefetch_tmap(&tmA16);
        prefetch_tmap(&tmA32);
        prefetch_tmap(&tmA64);
      } else {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmXd);
      }
    }
    // consecutive token rows: one 128-row box (rows past len belong to other
    // tokens, or lie past the last row and read as zeros, and only reach
    // accumulator rows that are never written)
    const int t0 = p.perm[start];
    const bool dense = p.perm[start + len - 1] - t0 == len - 1;
    int rr[4] = {0, 0, 0, 0};
    const CUtensorMap *bmap = nullptr;
    int bdst = 0, brow = 0;
    if (!aw) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = 4 * lane + e;
        rr[e] = r < len ? p.perm[start + r] : p.T;   // past the last row: zeros
      }
    } else {
      // lane b issues the stage's b-th adapter box (each slice's rank16 rows as
      // boxes of 64, 32 and 16 rows; at most 24)
      int b = 0;
      for (int i = 0; i < p.n && !bmap; ++i)
        for (int j0 = 0; j0 < r16;) {
          const int hb = r16 - j0 >= 64 ? 64 : r16 - j0 >= 32 ? 32 : 16;
          if (b++ == lane) {
            bmap = hb == 64 ? &tmA64 : hb == 32 ? &tmA32 : &tmA16;
            bdst = (i * r16 + j0) * 128;
            brow = i * p.R + j0;
            break;
          }
          j0 += hb;
        }
    }
    const int aslot = p.a_one_slot ? 0 : slot;
    const uint32_t tx = has_k ? (uint32_t)(TC_XB + ncols * KW * 2) : 0u;
    for (int k = kb, g = 0; k < ke; ++k, ++g) {
      // a loader warp owns stages s with s % nw == par and takes all their uses in
      // order, so its wait on a stage's empty barrier is always for the use just
      // before (a later use could otherwise pass an earlier one of the same parity)
      if ((g % NS) % nw != par) continue;
      const int s = g % NS;
      if (g >= NS && !wait_all(&empty[s], ((g / NS) & 1) ^ 1)) break;
      uint8_t *st = ring + s * STAGE;
      const int k0 = k * KW;
      if (!aw) {
        if (lane == 0) {
          if (tx) mbar_arrive_expect_tx(&full[s], tx);
          else mbar_arrive(&full[s]);
        }
        __syncwarp();
        if (has_k) {
          if (!dense) tma_gather4(st + lane * 512, &tmX, &full[s], k0, rr[0], rr[1], rr[2], rr[3]);
          else if (lane == 0) tma_load_2d(st, &tmXd, &full[s], k0, t0);
        }
      } else if (bmap && has_k) {
        tma_load_3d(st + TC_XB + bdst, bmap, &full[s], k0, brow, aslot);
      }
    }
  } else if (any && warp == TC_MMA_WARP) {
    // ---------------------------------------------------------------- MMA issuer (one thread)
    if (lane == 0) {
      const uint32_t idesc = tc_idesc_bf16(TC_M, ncols);
      bool ok = true;
      for (int k = kb, g = 0; k < ke; ++k, ++g) {
        const int s = g % NS;
        if (!mbar_wait(&full[s], (g / NS) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t xa = smem_u32(ring + s * STAGE), aa = xa + TC_XB;
#pragma unroll
        for (int kk = 0; kk < KW / 16; ++kk)
          if ((int64_t)k * KW + kk * 16 < p.in)
            tc_mma_bf16(tmem, tc_desc_sw128(xa + kk * 32), tc_desc_sw128(aa + kk * 32), idesc,
                        (k > kb || kk > 0) ? 1u : 0u);
        tc_commit(&empty[s]);   // the stage is free once these MMAs have read it
      }
      if (ok) tc_commit(accf);
      tc_commit(mdone);
      mbar_wait(mdone, 0);
    }
    __syncwarp();
  } else if (any && warp >= 4 && warp < 8) {
    // ---------------------------------------------------------------- drain: one token row per thread
    const int r = 32 * (warp & 3) + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    // an empty share (more CTAs than stages) leaves zeros
    const bool mine = ke > kb && has_k;
    bool ok = !mine || wait_all(accf, 0);
    if (ok) tc_fence_after();
    if (ok && q > 0) {
      // partial sums to this CTA's shared memory (the ring is no longer read), column-major
      for (int c0 = 0; c0 < ncols; c0 += 16) {
        float v[16];
        if (mine) {
          tmem_ld16(trow + (uint32_t)c0, v);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) xbuf[(c0 + e) * TC_M + r] = v[e];
      }
      mbar_arrive_remote(xready, 0);                    // released to CTA 0
      wait_all<true>(xdone, 0);                          // CTA 0 has read it
    } else if (ok) {
      if (cl > 1) ok = wait_all<true>(xready, 0);
      float *hrow = r < len ? p.h + (int64_t)p.perm[start + r] * p.ldh : nullptr;
      for (int c0 = 0; ok && c0 < ncols; c0 += 16) {
        float v[16];
        if (mine) {
          tmem_ld16(trow + (uint32_t)c0, v);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
        }
        // the other CTAs' partial sums, in cluster-rank order (16 loads in flight)
        for (int qq = 1; qq < cl; ++qq) {
          float u[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) u[e] = ld_dsmem_f1(&xbuf[(c0 + e) * TC_M + r], (uint32_t)qq);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] += u[e];
        }
        const int i = c0 / r16, j0 = c0 - i * r16;
        if (hrow) {
          float *hp = hrow + (int64_t)i * p.R + j0;
          if (j0 + 16 <= rank) {
#pragma unroll
            for (int e = 0; e < 16; e += 4)
              *reinterpret_cast<float4 *>(hp + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
          } else {
            // columns past the rank come from padding rows of a
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (j0 + e < rank) hp[e] = v[e];
          }
        }
      }
      for (int qq = 1; qq < cl; ++qq) mbar_arrive_remote(xdone, (uint32_t)qq);
    }
  }
  pdl_launch_dependents();
  // every MMA has completed (the issuer waited for its last commit): free the tensor memory
  tc_fence_before();
  __syncthreads();
  if (warp == TC_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)p.tc_cols);
  }
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
  // CTA (tile, group, 64-row sub-tile)
  const int sub = blockIdx.x % p.nsub, rest = blockIdx.x / p.nsub;
  const int tile = rest / p.ngroups, grp = rest % p.ngroups;
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
  const int slot = td.x, start = td.y + MBM * sub, len = min(MBM, td.z - MBM * sub);
  if (len <= 0) return;
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
// expand_decode_kernel: the expand for tiles of a few tokens (decode batches,
// where every token may carry its own adapter).  The work is streaming the
// slots' b rows b[slot][c][0 .. rank).  A block takes one tile, one slice i and
// a range of output columns holding 2048 sixteen-byte pieces of b: a column's
// ceil(rank / 8) pieces sit in P consecutive lanes (P = that count rounded up
// to a power of two), so every block reads about the same bytes whatever the
// rank, and a thread keeps eight pieces in flight.  A lane multiplies its piece
// by the matching eight entries of each token's h row (held in shared memory),
// the P lanes of a column add their partial sums with shuffles, and the first
// of them adds scal * sum into y[t][c].  Columns j >= rank of h and b are never
// used (the pieces are masked past the rank).
// =============================================================================
constexpr int DX_THREADS = 256;
constexpr int DX_PIECES = 8;    // sixteen-byte pieces of b per thread
constexpr int DX_BLOCK_PIECES = DX_THREADS * DX_PIECES;

// Columns a block covers for pieces-per-column P.
__host__ __device__ __forceinline__ int dx_cols(int P) { return DX_BLOCK_PIECES / P; }

template <int RP>
__global__ void __launch_bounds__(DX_THREADS, 4) expand_decode_kernel(MArgs p) {
  extern __shared__ float hs[];   // [len][RP] of the tile's h rows (slice i), then [len] token rows
  pdl_wait();
  const int nblk = p.ngroups;     // blocks per tile (over all slices)
  const int tile = blockIdx.x / nblk, bi = blockIdx.x % nblk;
  if (tile >= p.header[1]) return;
  // block -> slice i and its index inside the slice (the host sized the grid
  // for P = RP / 8, the most pieces a column can have)
  int i = 0, left = bi;
  for (; i < p.n; ++i) {
    const int nb = (p.off[i + 1] - p.off[i] + dx_cols(RP / 8) - 1) / dx_cols(RP / 8);
    if (left < nb) break;
    left -= nb;
  }
  if (i >= p.n) return;
  const int4 td = p.tiles[tile];
  const int slot = td.x, start = td.y, len = td.z;
  const int rank = min(p.ranks[slot], RP);
  const int npc = (rank + 7) >> 3;
  int lgP = 0;
  while ((1 << lgP) < npc) ++lgP;
  const int P = 1 << lgP;
  const int width = p.off[i + 1] - p.off[i];
  const int col0 = left * dx_cols(P);
  if (col0 >= width) return;   // fewer pieces per column: fewer blocks cover the slice
  const int tid = threadIdx.x, pc = tid & (P - 1);
  // b pieces first (their loads in flight while h is staged)
  const __nv_bfloat16 *bs = p.b + (int64_t)slot * p.sb_slot + (int64_t)p.off[i] * p.sb_row;
  uint4 w[DX_PIECES];
#pragma unroll
  for (int k = 0; k < DX_PIECES; ++k) {
    const int c = col0 + ((k * DX_THREADS + tid) >> lgP);
    w[k] = c < width && pc < npc ? *reinterpret_cast<const uint4 *>(bs + (int64_t)c * p.sb_row + pc * 8)
                                 : make_uint4(0u, 0u, 0u, 0u);
  }
  int *rows = reinterpret_cast<int *>(hs + len * RP);
  for (int e = tid; e < len * RP; e += DX_THREADS) {
    const int t = e / RP, j = e % RP;
    hs[e] = j < rank ? p.h[(int64_t)p.perm[start + t] * p.ldh + (int64_t)i * p.R + j] : 0.f;
  }
  for (int t = tid; t < len; t += DX_THREADS) rows[t] = p.perm[start + t];
  const float sc = p.scal[slot];
  // entries past the rank in this lane's pieces may hold anything: a mask per
  // 32-bit word (two entries) clears them
  const int tail = rank - pc * 8;
  const uint32_t m0 = tail >= 2 ? ~0u : tail == 1 ? 0xffffu : 0u, m1 = tail >= 4 ? ~0u : tail == 3 ? 0xffffu : 0u,
                 m2 = tail >= 6 ? ~0u : tail == 5 ? 0xffffu : 0u, m3 = tail >= 8 ? ~0u : tail == 7 ? 0xffffu : 0u;
  __syncthreads();
#pragma unroll
  for (int k = 0; k < DX_PIECES; ++k) {
    const float2 b0 = unpack_bf16(w[k].x & m0), b1 = unpack_bf16(w[k].y & m1), b2 = unpack_bf16(w[k].z & m2),
                 b3 = unpack_bf16(w[k].w & m3);
    const int c = col0 + ((k * DX_THREADS + tid) >> lgP);
    const bool store = pc == 0 && c < width;
    for (int t = 0; t < len; ++t) {
      const float4 h0 = *reinterpret_cast<const float4 *>(hs + t * RP + pc * 8);
      const float4 h1 = *reinterpret_cast<const float4 *>(hs + t * RP + pc * 8 + 4);
      float acc = h0.x * b0.x + h0.y * b0.y + h0.z * b1.x + h0.w * b1.y + h1.x * b2.x + h1.y * b2.y +
                  h1.z * b3.x + h1.w * b3.y;
      for (int o = 1; o < P; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (store) {
        __nv_bfloat16 *yp = p.y + (int64_t)rows[t] * p.ldy + p.off[i] + c;
        *yp = __float2bfloat16_rn(__bfloat162float(*yp) + sc * acc);
      }
    }
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
    // the slot and the id are independent loads: issue both before either is used
    const int s = __ldg(&slots[t]);
    const int64_t id = __ldg(&ids[t]);
    if (s < 0 || s >= S) continue;
    const int rank = __ldg(&ranks[s]);
    if (rank < 1 || rank > R) continue;
    const bool valid = id >= 0 && id < V;
    const __nv_bfloat16 *col = a + (int64_t)s * sa_slot + (valid ? id : 0) * sa_col;
    // up to 4 rank entries per lane, all loads in flight before the stores
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = lane + 32 * q;
      v[q] = valid && j < rank ? __bfloat162float(col[(int64_t)j * sa_row]) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = lane + 32 * q;
      if (j < rank) h[t * ldh + j] = v[q];
    }
  }
  pdl_launch_dependents();
}


// ----------------------------------------------------------------------------- host side
// Decode batches: at most four tokens per slot on average.
bool decode_shape(int64_t T, int S) { return T <= 4 * (int64_t)S; }

namespace {

// Tokens per tile: decode batches (a few tokens per slot) are cut into tiles of
// at most four tokens for the CUDA-core shrink and expand, prefill batches into
// tiles of at most TC_M tokens for the tiled kernels.
int tile_tokens(int64_t T, int S) { return decode_shape(T, S) ? kDecTokens : TC_M; }
// At most one partial tile per slot.
int max_tiles(int64_t T, int S) { return (int)(ceil_div(T, tile_tokens(T, S)) + std::min<int64_t>(S, T)); }

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
                           int32_t *num_active, int *header, int4 *tiles, cudaStream_t st, int *zero = nullptr,
                           int nzero = 0) {
  const int S = ad.num_slots;
  int nw = (int)std::max<int64_t>(1, (160 * 1024 / 4 - 256 - 3 * S) / S);   // shared-memory bound
  // enough warps for the tokens, and for the per-slot scans (a warp scans the
  // slots s = w, w + nw, ...): at most 8 slots per warp
  const int64_t want = std::max<int64_t>(ceil_div(ad.num_tokens, LORA_GROUP_TOKENS_PER_WARP), ceil_div(S, 8));
  nw = std::min<int64_t>({nw, 32, std::max<int64_t>(1, want)});
  const size_t smem = (size_t)(nw * S + 3 * S + 224) * 4;
  LORA_CUDA(ensure_smem((const void *)group_kernel, smem));
  LORA_CUDA(launch(group_kernel, dim3(1), dim3(nw * 32), smem, st, 1, true, ad.slots, ad.num_tokens, S,
                   ad.max_rank, ranks, counts, perm, num_active, header, tiles, tile_tokens(ad.num_tokens, S), zero,
                   nzero));
  return LORA_OK;
}

// 64 x 64 bf16 tiles of a row-major [rows][cols] operand (128-byte swizzle).
bool map_rows(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld) {
  uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  uint64_t str[1] = {(uint64_t)ld * 2};
  uint32_t box[2] = {64, 64};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Boxes of `box_rows` rows x 64 columns of the adapter stack a[S][rows][cols] (128-byte swizzle).
bool map_adapter(CUtensorMap *m, const void *base, int64_t S, int64_t rows, int64_t cols, int64_t s_slot,
                 int64_t s_row, uint32_t box_rows) {
  uint64_t dims[3] = {(uint64_t)cols, (uint64_t)rows, (uint64_t)S};
  uint64_t str[2] = {(uint64_t)s_row * 2, (uint64_t)s_slot * 2};
  uint32_t box[3] = {64, box_rows, 1};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Boxes of `box_rows` rows x 64 columns of a row-major [rows][cols] operand (128-byte swizzle).
bool map_box(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows) {
  uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  uint64_t str[1] = {(uint64_t)ld * 2};
  uint32_t box[2] = {64, box_rows};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Rows of x, one 64-column box a row (the four-row gather copies of the shrink).
bool map_gather_rows(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld) {
  uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  uint64_t str[1] = {(uint64_t)ld * 2};
  uint32_t box[2] = {64, 1};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Cluster size of the shrink (CTAs splitting a tile's contraction); 0 picks one
// from the tile bound so that the clusters about cover the SMs once.
#ifndef LORA_SHRINK_CL
#define LORA_SHRINK_CL 0
#endif

lora_status_t launch_shrink(MArgs a, int64_t T, cudaStream_t st) {
  LORA_CUDA(ensure_smem((const void *)shrink_kernel, TC_BYTES));
  CUtensorMap tmX, tmXd, tmA16, tmA32, tmA64;
  memset(&tmX, 0, sizeof(tmX));
  memset(&tmXd, 0, sizeof(tmXd));
  memset(&tmA16, 0, sizeof(tmA16));
  memset(&tmA32, 0, sizeof(tmA32));
  memset(&tmA64, 0, sizeof(tmA64));
  a.T = (int)T;
  const int nc = a.n * (int)round_up(a.R, 16);   // most columns a slot can have
  a.tc_cols = 32;
  while (a.tc_cols < nc) a.tc_cols *= 2;
  a.sh_stage = TC_XB + nc * KW * 2;
  a.sh_ns = std::min(16, TC_RING / a.sh_stage);
  if (a.sh_ns < 2 || nc > kMaxHC || a.tc_cols > 512) return LORA_ERR_UNSUPPORTED;
  a.nk = (int)std::max<int64_t>(1, ceil_div(a.in, KW));
  const int64_t tiles = max_tiles(T, a.S);
  int cl = LORA_SHRINK_CL;
  if (cl <= 0) {
    // about ceil(T / 128) + S / 2 tiles are real; cover the SMs once
    const int64_t est = ceil_div(T, TC_M) + std::min<int64_t>(a.S, T) / 2, sms = num_sms();
    cl = 1;
    while (cl < 8 && est * cl * 2 * 4 <= sms * 5) cl *= 2;
  }
  while (cl > 1 && a.nk < cl) cl /= 2;
  a.cl = cl;
  if (a.in > 0) {
    // one adapter when the slot stride is zero: a map over one slot, slot coordinate 0
    a.a_one_slot = a.sa_slot == 0 ? 1 : 0;
    const int64_t arows = (int64_t)a.n * a.R, aS = a.a_one_slot ? 1 : a.S;
    const int64_t sslot = a.a_one_slot ? arows * a.sa_row : a.sa_slot;
    if (!map_gather_rows(&tmX, a.x, T, a.in, a.ldx) || !map_box(&tmXd, a.x, T, a.in, a.ldx, TC_M) ||
        !map_adapter(&tmA16, a.a, aS, arows, a.in, sslot, a.sa_row, 16) ||
        !map_adapter(&tmA32, a.a, aS, arows, a.in, sslot, a.sa_row, 32) ||
        !map_adapter(&tmA64, a.a, aS, arows, a.in, sslot, a.sa_row, 64))
      return LORA_ERR_ALIGNMENT;
  }
  LORA_CUDA(launch(shrink_kernel, dim3((unsigned)(tiles * cl)), dim3(TC_THREADS), TC_BYTES, st, cl, true, tmX,
                   tmXd, tmA16, tmA32, tmA64, a));
  return LORA_OK;
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
  const int64_t gb = std::max<int64_t>(1, ceil_div(tiles * (TC_M / MBM) * blocks, 3 * cap));
  int64_t ng = 0;
  for (int i = 0; i < a.n; ++i) ng += ceil_div(ceil_div(a.off[i + 1] - a.off[i], CBW), gb);
  if (ng == 0) return LORA_OK;
  a.gb = (int)gb;
  a.ngroups = (int)ng;
  a.nsub = TC_M / MBM;
  CUtensorMap tmY;
  a.tma_ok = map_rows(&tmY, a.y, T, a.off[a.n], a.ldy) ? 1 : 0;
  LORA_CUDA(launch(kern, dim3((unsigned)(tiles * ng * a.nsub)), dim3(ExCfg<RP>::THREADS), smem, st, 1, true, tmY,
                   a));
  return LORA_OK;
}

template <int RP>
lora_status_t launch_expand_decode(MArgs a, int64_t T, cudaStream_t st) {
  int nblk = 0;
  for (int i = 0; i < a.n; ++i) nblk += (int)ceil_div(a.off[i + 1] - a.off[i], dx_cols(RP / 8));
  if (nblk == 0) return LORA_OK;
  a.ngroups = nblk;
  const int64_t tiles = max_tiles(T, a.S);
  const size_t smem = (size_t)TC_M * (RP + 1) * 4;   // h rows and token rows of the largest tile
  LORA_CUDA(ensure_smem((const void *)expand_decode_kernel<RP>, smem));
  LORA_CUDA(
      launch(expand_decode_kernel<RP>, dim3((unsigned)(tiles * nblk)), dim3(DX_THREADS), smem, st, 1, true, a));
  return LORA_OK;
}

// Decode batches (a few tokens per slot on average) stream the b rows on the
// CUDA cores; prefill batches run the tiled expand.

lora_status_t dispatch_expand(const MArgs &a, int64_t T, cudaStream_t st) {
  if (decode_shape(T, a.S)) {
    switch (rank_bucket(a.R)) {
      case 16: return launch_expand_decode<16>(a, T, st);
      case 32: return launch_expand_decode<32>(a, T, st);
      case 64: return launch_expand_decode<64>(a, T, st);
      default: return launch_expand_decode<128>(a, T, st);
    }
  }
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

// The schedule of the call: the caller's prebuilt one (no launch), else built
// into the workspace by the grouping kernel.
lora_status_t schedule(const MultiArgs &m, WsCarver &c, SchedPtrs &sp, cudaStream_t st) {
  if (m.addr.schedule != nullptr) {
    WsCarver pre(const_cast<void *>(m.addr.schedule), sched_bytes(m.addr.num_tokens, m.addr.num_slots));
    return carve_sched(pre, m.addr.num_tokens, m.addr.num_slots, sp) ? LORA_OK : LORA_ERR_WORKSPACE;
  }
  if (!carve_sched(c, m.addr.num_tokens, m.addr.num_slots, sp)) return LORA_ERR_WORKSPACE;
  return launch_group(m.addr, m.ranks, sp.counts, sp.perm, sp.header, sp.header, sp.tiles, st);
}

// Schedule, then the shrink itself (h written to `h`).
lora_status_t schedule_and_shrink(const MultiArgs &m, WsCarver &c, SchedPtrs &sp, MArgs *out, float *h,
                                  int64_t ldh, cudaStream_t st) {
  LORA_TRY(schedule(m, c, sp, st));
  MArgs a = margs(m, sp);
  a.h = h;
  a.ldh = ldh;
  *out = a;
  return launch_shrink(a, m.addr.num_tokens, st);
}

// Tickets of the stream-K shrink (one per tile).
size_t tc_counter_bytes(int64_t T, int S) { return ws_round((size_t)(max_tiles(T, S) + 1) * 4); }
// Width of the shrink output h for the workspace bound (n * R when known).
int shrink_cols(int64_t n_times_R, int R) {
  return (int)std::min<int64_t>(256, n_times_R > 0 ? n_times_R : (int64_t)LORA_MAX_SLICES * R);
}

DecArgs dec_args(const MultiArgs &m, const SchedPtrs &sp) {
  DecArgs a{};
  a.ranks = m.ranks;
  a.header = sp.header;
  a.tiles = sp.tiles;
  a.perm = sp.perm;
  a.S = m.addr.num_slots;
  a.R = m.addr.max_rank;
  a.n = m.n;
  a.T = m.addr.num_tokens;
  a.nk = (int)std::max<int64_t>(1, ceil_div(m.in, 256));
  a.h = m.h;
  a.ldh = m.ldh;
  return a;
}

// The schedule, then the shrink that suits the batch's shape: decode batches (a
// few tokens per slot) split (tile, chunk) units by cost over a persistent grid
// (their adapter rows read through a view that needs `in` a multiple of 64);
// prefill batches, and the rest, give each tile a cluster of CTAs.
lora_status_t schedule_then_shrink(const MultiArgs &m, WsCarver &c, SchedPtrs &sp, cudaStream_t st) {
  if (!decode_shape(m.addr.num_tokens, m.addr.num_slots) || m.in % 64 != 0) {
    MArgs a;
    return schedule_and_shrink(m, c, sp, &a, m.h, m.ldh, st);
  }
  // the tickets (one per tile) start at zero: the grouping kernel clears them,
  // or a memset when the caller's schedule is reused
  const int nc = max_tiles(m.addr.num_tokens, m.addr.num_slots) + 1;
  int *cnt = nullptr;
  if (m.addr.schedule != nullptr) {
    LORA_TRY(schedule(m, c, sp, st));
    cnt = (int *)c.take((size_t)nc * 4);
    if (!cnt) return LORA_ERR_WORKSPACE;
    LORA_CUDA(cudaMemsetAsync(cnt, 0, (size_t)nc * 4, st));
  } else {
    if (!carve_sched(c, m.addr.num_tokens, m.addr.num_slots, sp)) return LORA_ERR_WORKSPACE;
    cnt = (int *)c.take((size_t)nc * 4);
    if (!cnt) return LORA_ERR_WORKSPACE;
    LORA_TRY(launch_group(m.addr, m.ranks, sp.counts, sp.perm, sp.header, sp.header, sp.tiles, st, cnt, nc));
  }
  DecArgs a = dec_args(m, sp);
  a.counters = cnt;
  a.part = (float *)c.take(dec_part_bytes(m.n, m.addr.max_rank));
  if (!a.part) return LORA_ERR_WORKSPACE;
  return shrink_dec_launch(a, m, m.addr.num_tokens, st);
}

}  // namespace

size_t schedule_bytes(int64_t T, int S) { return T > 0 ? sched_bytes(T, S) : 0; }

lora_status_t build_schedule(const lora_addressing_t &addr, const int32_t *ranks, void *sched, size_t bytes,
                             cudaStream_t st) {
  if (addr.num_tokens == 0) return LORA_OK;
  WsCarver c(sched, bytes);
  SchedPtrs sp;
  if (!carve_sched(c, addr.num_tokens, addr.num_slots, sp)) return LORA_ERR_WORKSPACE;
  return launch_group(addr, ranks, sp.counts, sp.perm, sp.header, sp.header, sp.tiles, st);
}

size_t multi_ws_bytes(int op, int64_t T, int64_t in, int64_t O, int R, int S) {
  (void)in;
  if (T <= 0) return 0;
  if (op == LORA_OP_GROUP_BY_SLOT) return sched_bytes(T, S);
  if (op == LORA_OP_EXPAND) return sched_bytes(T, S) + tc_counter_bytes(T, S);
  // shrink: O carries the width of h (num_slices * R), 0 when unknown
  if (op == LORA_OP_SHRINK) {
    const int nc = shrink_cols(O, R);
    return sched_bytes(T, S) + tc_counter_bytes(T, S) + ws_round(dec_part_bytes(1, nc));
  }
  if (op == LORA_OP_APPLY_LINEAR)
    return sched_bytes(T, S) + tc_counter_bytes(T, S) + ws_round(dec_part_bytes(1, shrink_cols(0, R))) +
           hbuf_bytes(T, R);
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
  if (m.in == 0) {
    // h = x * a = 0: every entry the page specifies is zero (the others may be anything)
    LORA_CUDA(cudaMemset2DAsync(m.h, (size_t)m.ldh * 4, 0, (size_t)m.n * m.addr.max_rank * 4,
                                (size_t)m.addr.num_tokens, st));
    return LORA_OK;
  }
  WsCarver c(ws, ws_bytes);
  SchedPtrs sp;
  return schedule_then_shrink(m, c, sp, st);
}

// The expand of a scheduled batch: decode batches stream b through TMA on the
// persistent decode kernel (the plain-load kernel when y or b cannot be read
// through tensor maps, or R > 72); prefill batches run the tiled expand.
lora_status_t expand_scheduled(const MultiArgs &m, const SchedPtrs &sp, cudaStream_t st) {
  if (decode_shape(m.addr.num_tokens, m.addr.num_slots)) {
    DecExpArgs a{};
    a.ranks = m.ranks;
    a.scal = m.scalings;
    a.header = sp.header;
    a.tiles = sp.tiles;
    a.perm = sp.perm;
    a.S = m.addr.num_slots;
    a.R = m.addr.max_rank;
    a.n = m.n;
    a.T = m.addr.num_tokens;
    a.h = m.h;
    a.ldh = m.ldh;
    const lora_status_t r = expand_dec_launch(a, m, m.addr.num_tokens, st);
    if (r != LORA_ERR_ALIGNMENT && r != LORA_ERR_UNSUPPORTED) return r;
  }
  return dispatch_expand(margs(m, sp), m.addr.num_tokens, st);
}

lora_status_t expand(MultiArgs m, void *ws, size_t ws_bytes, cudaStream_t st) {
  LORA_TRY(check_seg(m, false, true));
  WsCarver c(ws, ws_bytes);
  SchedPtrs sp;
  LORA_TRY(schedule(m, c, sp, st));
  return expand_scheduled(m, sp, st);
}

lora_status_t apply_linear(MultiArgs m, void *ws, size_t ws_bytes, cudaStream_t st) {
  LORA_TRY(check_seg(m, true, true));
  WsCarver c(ws, ws_bytes);
  float *h = (float *)c.take(hbuf_bytes(m.addr.num_tokens, m.addr.max_rank));
  if (!h) return LORA_ERR_WORKSPACE;
  SchedPtrs sp;
  m.h = h;
  m.ldh = (int64_t)m.n * m.addr.max_rank;
  LORA_TRY(schedule_then_shrink(m, c, sp, st));
  return expand_scheduled(m, sp, st);
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
