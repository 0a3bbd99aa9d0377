// multi.cu -- multi-adapter (serving) LoRA ops for sm_103a.
//
// Operations (mstar page "mstar.engine.resources.lora.ops"):
//   shrink         h[t, i*R + j] = x[t] . a[slot(t)][i*R + j]            (j < rank)
//   expand_fused   y[t, slice i] += scalings[slot] * h[t, slice i] @ b[slot, slice i]^T
//   apply_linear_  shrink then expand (fused here; h never leaves the chip)
//   gather_shrink  h[t] = a[slot(t)][:, ids[t]]  (ids outside [0, V) give zeros)
// and the integer step in front of them (group_by_slot): a stable counting sort
// of the active tokens by slot and a list of tiles of at most 64 tokens of one
// slot, built on the device with no host sync (the page requires the ops to run
// without one).
//
// The segmented kernel runs one token tile per cluster of `cl` CTAs.  Phase 1
// (shrink) splits the contraction over the cluster and sums the partial h in
// cluster-rank order through distributed shared memory; phase 2 (expand) splits
// the output column blocks over the cluster.  Rows are gathered (the tile's
// tokens need not be contiguous) with one 1-D bulk copy per row into padded
// shared-memory rows (144-byte pitch, conflict-free ldmatrix); y rows go back
// the same way from a storer warp.  Adapter padding (rows / columns past a
// slot's rank, which may hold anything) is masked in registers, never trusted.
#include <algorithm>

#include "common.cuh"
#include "host_common.h"
#include "multi.h"

namespace lora {

namespace {

constexpr int MBM = 64;                   // token rows per tile
constexpr int MCW = 4;                    // consumer warps
constexpr int MTHREADS = (MCW + 2) * 32;  // + loader + storer
constexpr int KW = 64;                    // contraction columns per phase-1 stage
constexpr int XP = KW * 2 + 16;           // padded row pitch (bytes) of x / a / y rows
constexpr int CBW = 64;                   // output columns per phase-2 block
constexpr int kMaxHC = 256;               // n * R columns of h held on chip

enum Mode { kShrink = 0, kExpand = 1, kApply = 2 };

struct SegArgs {
  const int32_t *slots, *ranks;
  const float *scal;
  const int *header;   // [0] number of active tokens, [1] number of tiles
  const int4 *tiles;   // (slot, start, len, 0)
  const int32_t *perm;
  int T, S, R, n, cl;
  int64_t in;
  const __nv_bfloat16 *x; int64_t ldx;
  const __nv_bfloat16 *a; int64_t sa_slot, sa_row;
  const __nv_bfloat16 *b; int64_t sb_slot, sb_row;
  float *h; int64_t ldh;
  __nv_bfloat16 *y; int64_t ldy;
  int nb;                      // number of (slice, column block) pairs
  int off[LORA_MAX_SLICES + 1];
  int blk0[LORA_MAX_SLICES + 1];   // first block index of each slice
};

__device__ __forceinline__ uint32_t mask_pair(uint32_t v, int j0, int lim) {
  // keep the bf16 halves whose column j0 (low) / j0 + 1 (high) is below lim
  const uint32_t lo = j0 < lim ? 0x0000ffffu : 0u, hi = j0 + 1 < lim ? 0xffff0000u : 0u;
  return v & (lo | hi);
}

template <int N>
__device__ __forceinline__ void bulk_wait_read_n() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

template <int HC>
struct SegCfg {
  static constexpr int P1 = (MBM + HC) * XP;              // x rows + a rows
  static constexpr int BP = 2 * 128 + 16;                 // max b-row pitch (R <= 128)
  static constexpr int P2 = MBM * XP + CBW * BP;          // y rows + b rows
  static constexpr int STAGE = ((P1 > P2 ? P1 : P2) + 1023) / 1024 * 1024;
  static constexpr int NS = (72 * 1024) / STAGE < 2 ? 2 : (72 * 1024) / STAGE > 6 ? 6 : (72 * 1024) / STAGE;
  static constexpr int BYTES = 1024 + NS * STAGE + 8 * (3 * NS + 4) + 64;
  static_assert(MBM * HC * 4 <= NS * STAGE, "h exchange must fit in the stage ring");
};

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

}  // namespace

// =============================================================================
// group_by_slot: one CTA.  Each warp owns a contiguous range of tokens; pass 1
// counts active tokens per (warp, slot) (warp-level __match_any_sync, no
// atomics), a block scan turns the counts into per-(warp, slot) cursors, and
// pass 2 revisits the ranges in the same order and scatters each token to its
// cursor: a stable counting sort by slot.  Tiles of at most `bmt` tokens of one
// slot are then listed in slot order.
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

__global__ void __launch_bounds__(1024) group_kernel(const int32_t *__restrict__ slots, int T, int S, int R,
                                                     const int32_t *__restrict__ ranks, int32_t *counts_out,
                                                     int32_t *perm_out, int32_t *num_active_out, int *header,
                                                     int4 *tiles, int bmt) {
  extern __shared__ int gsm[];
  const int nw = blockDim.x >> 5;
  int *hist = gsm;                 // [nw][S]
  int *sh = gsm + nw * S;          // scan scratch (160 ints)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  for (int i = threadIdx.x; i < nw * S; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int t_lo = (int)((int64_t)T * warp / nw), t_hi = (int)((int64_t)T * (warp + 1) / nw);
  const unsigned lt = (1u << lane) - 1u;
  for (int t0 = t_lo; t0 < t_hi; t0 += 32) {
    const int t = t0 + lane;
    const int s = t < t_hi ? slots[t] : -1;
    const bool act = t < t_hi && s >= 0 && s < S && ranks[s] >= 1 && ranks[s] <= R;
    const unsigned m = __match_any_sync(0xffffffffu, act ? s : -(lane + 1));
    if (act && (m & lt) == 0) hist[warp * S + s] += __popc(m);
    __syncwarp();
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
  for (int t0 = t_lo; t0 < t_hi; t0 += 32) {
    const int t = t0 + lane;
    const int s = t < t_hi ? slots[t] : -1;
    const bool act = t < t_hi && s >= 0 && s < S && ranks[s] >= 1 && ranks[s] <= R;
    const unsigned m = __match_any_sync(0xffffffffu, act ? s : -(lane + 1));
    int cur = 0;
    if (act) cur = hist[warp * S + s];
    __syncwarp();
    if (act) {
      perm_out[cur + __popc(m & lt)] = t;
      if ((m & lt) == 0) hist[warp * S + s] = cur + __popc(m);
    }
    __syncwarp();
  }
  pdl_launch_dependents();
}

// =============================================================================
// The segmented kernel.  MODE kShrink: phase 1 and the h write; kExpand: h read
// and phase 2; kApply: phase 1 then phase 2 with h in registers.
// =============================================================================
template <int HC, int MODE>
__global__ void __launch_bounds__(MTHREADS) seg_kernel(SegArgs p) {
  using C = SegCfg<HC>;
  constexpr int NS = C::NS;
  constexpr bool P1 = MODE != kExpand, P2 = MODE != kShrink;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * C::STAGE);
  uint64_t *done = full + NS;
  uint64_t *freeb = done + NS;
  uint64_t *hready = freeb + NS, *hdone = hready + 1, *xready = hready + 2;
  float *hbuf = reinterpret_cast<float *>(smem);   // the h exchange reuses the stage ring

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cl = p.cl;
  const int tile = blockIdx.x / cl;
  pdl_wait();
  if (tile >= p.header[1]) return;   // whole cluster: beyond the device-side tile count
  const uint32_t crank = cl > 1 ? cluster_ctarank() : 0u;
  const int4 td = p.tiles[tile];
  const int slot = td.x, start = td.y, len = td.z;
  const int rank = p.ranks[slot];
  const int R = p.R, n = p.n;
  const int nk = P1 ? (int)((p.in + KW - 1) / KW) : 0;
  const int k_beg = (int)((int64_t)nk * crank / cl), k_end = (int)((int64_t)nk * (crank + 1) / cl);
  const int b_beg = P2 ? (int)((int64_t)p.nb * crank / cl) : 0, b_end = P2 ? (int)((int64_t)p.nb * (crank + 1) / cl) : 0;
  const int n1 = k_end - k_beg, ntiles = n1 + (b_end - b_beg);
  const int r16 = (R + 15) & ~15, rank8 = (rank + 7) & ~7;
  const int bp = r16 * 2 + 16;   // b-row pitch in bytes

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 32);
      mbar_init(&done[s], MCW);
      mbar_init(&freeb[s], 1);
    }
    mbar_init(hready, cl > 1 ? MCW * 32 * (cl - 1) : 1);
    mbar_init(hdone, cl > 1 ? MCW * 32 * (cl - 1) : 1);
    mbar_init(xready, MCW * 32);
    fence_barrier_init();
  }
  if (cl > 1) cluster_sync_all(); else __syncthreads();

  // (slice, column block) of phase-2 block index q
  auto blk = [&](int q, int &i, int &c0, int &ocols) {
    i = 0;
    while (i + 1 < n && q >= p.blk0[i + 1]) ++i;
    c0 = p.off[i] + (q - p.blk0[i]) * CBW;
    ocols = min(CBW, p.off[i + 1] - c0);
  };

  if (warp == MCW) {
    // ---------------------------------------------------------------- loader (32 lanes)
    for (int g = 0; g < ntiles; ++g) {
      const int s = g % NS;
      if (g >= NS && !mbar_wait(&freeb[s], ((g / NS) & 1) ^ 1)) break;
      if (P1 && P2 && cl > 1 && g == n1 && !mbar_wait(xready, 0)) break;   // stage ring holds the exchange
      uint8_t *st = smem + s * C::STAGE;
      uint32_t bytes = 0;
      if (g < n1) {
        const int64_t k0 = (int64_t)(k_beg + g) * KW;
        const int kb = (int)(p.in - k0 < (int64_t)KW ? p.in - k0 : (int64_t)KW);
        const uint32_t rb = kb * 2;
        // expect first, then copies, then (after zeroing a ragged tail) arrive
        int cnt = 0;
        for (int r = lane; r < len; r += 32) ++cnt;
        for (int c = lane; c < n * R; c += 32)
          if (c % R < rank) ++cnt;
        mbar_expect_tx(&full[s], cnt * rb);
        for (int r = lane; r < len; r += 32)
          bulk_load(st + r * XP, p.x + (int64_t)p.perm[start + r] * p.ldx + k0, rb, &full[s]);
        const __nv_bfloat16 *as = p.a + (int64_t)slot * p.sa_slot + k0;
        for (int c = lane; c < n * R; c += 32)
          if (c % R < rank) bulk_load(st + (MBM + c) * XP, as + (int64_t)c * p.sa_row, rb, &full[s]);
        if (kb < KW) {   // zero the tail columns of every loaded row (they enter the contraction)
          for (int r = lane; r < len; r += 32)
            for (int cc = rb; cc < KW * 2; cc += 16) *reinterpret_cast<int4 *>(st + r * XP + cc) = make_int4(0, 0, 0, 0);
          for (int c = lane; c < n * R; c += 32)
            if (c % R < rank)
              for (int cc = rb; cc < KW * 2; cc += 16)
                *reinterpret_cast<int4 *>(st + (MBM + c) * XP + cc) = make_int4(0, 0, 0, 0);
        }
        (void)bytes;
      } else {
        int i, c0, ocols;
        blk(b_beg + g - n1, i, c0, ocols);
        const uint32_t yb = ocols * 2, bb = rank8 * 2;
        int cnt = 0;
        for (int r = lane; r < len; r += 32) ++cnt;
        int cb = 0;
        for (int cc = lane; cc < ocols; cc += 32) ++cb;
        mbar_expect_tx(&full[s], cnt * yb + cb * bb);
        for (int r = lane; r < len; r += 32)
          bulk_load(st + r * XP, p.y + (int64_t)p.perm[start + r] * p.ldy + c0, yb, &full[s]);
        const __nv_bfloat16 *bs = p.b + (int64_t)slot * p.sb_slot;
        for (int cc = lane; cc < ocols; cc += 32)
          bulk_load(st + MBM * XP + cc * bp, bs + (int64_t)(c0 + cc) * p.sb_row, bb, &full[s]);
      }
      mbar_arrive(&full[s]);
    }
    pdl_launch_dependents();
    return;
  }
  if (warp == MCW + 1) {
    // ---------------------------------------------------------------- storer (32 lanes)
    constexpr int D = (NS - 1) < 2 ? (NS - 1) : 2;
    int pend[D + 1];
    int np = 0;
    for (int g = 0; g < ntiles; ++g) {
      const int s = g % NS;
      if (!mbar_wait(&done[s], (g / NS) & 1)) break;
      if (g < n1) {
        if (lane == 0) mbar_arrive(&freeb[s]);
        continue;
      }
      int i, c0, ocols;
      blk(b_beg + g - n1, i, c0, ocols);
      uint8_t *st = smem + s * C::STAGE;
      for (int r = lane; r < len; r += 32)
        bulk_store(p.y + (int64_t)p.perm[start + r] * p.ldy + c0, st + r * XP, ocols * 2);
      bulk_commit();
      pend[np++] = g;
      if (np > D) {
        bulk_wait_read_n<D>();
        __syncwarp();
        if (lane == 0) mbar_arrive(&freeb[pend[0] % NS]);
        for (int k = 1; k < np; ++k) pend[k - 1] = pend[k];
        --np;
      }
    }
    bulk_wait_read_n<0>();
    __syncwarp();
    if (lane == 0)
      for (int k = 0; k < np; ++k) mbar_arrive(&freeb[pend[k] % NS]);
    bulk_wait_all();
    pdl_launch_dependents();
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int w = warp, gq = lane >> 2, cq = lane & 3;
  const bool rows_live = 16 * w < len;
  float hacc[HC / 8][4];
#pragma unroll
  for (int i = 0; i < HC / 8; ++i) hacc[i][0] = hacc[i][1] = hacc[i][2] = hacc[i][3] = 0.f;
  bool ok = true;
  int g = 0;
  if (P1) {
    for (; g < n1; ++g) {
      const int s = g % NS;
      if (!(ok = wait_all(&full[s], (g / NS) & 1))) break;
      const uint32_t xb = smem_u32(smem + s * C::STAGE), ab = xb + MBM * XP;
      const int64_t k0 = (int64_t)(k_beg + g) * KW;
      if (rows_live) {
#pragma unroll
        for (int kk = 0; kk < KW / 16; ++kk) {
          if (k0 + kk * 16 >= p.in) break;
          uint32_t a[4];
          lda_p(xb, XP, 16 * w, kk * 16, a);
#pragma unroll
          for (int np = 0; np < HC / 16; ++np) {
            if (np * 16 >= n * R) break;
            uint32_t b[4];
            ldb_p(ab, XP, np * 16, kk * 16, b);
            mma_bf16(hacc[2 * np], a, b[0], b[1]);
            mma_bf16(hacc[2 * np + 1], a, b[2], b[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&done[s]);
    }
    // columns past the slot's rank come from unloaded rows of a: zero them
#pragma unroll
    for (int nt = 0; nt < HC / 8; ++nt) {
      const int c = nt * 8 + 2 * cq;
      const bool v0 = c < n * R && (c % R) < rank, v1 = c + 1 < n * R && ((c + 1) % R) < rank;
      if (!v0) hacc[nt][0] = hacc[nt][2] = 0.f;
      if (!v1) hacc[nt][1] = hacc[nt][3] = 0.f;
    }
    if (cl > 1) {
      // exchange partial h through distributed shared memory (in the stage ring)
      named_bar_sync(1, MCW * 32);   // every consumer warp is done with the last phase-1 stage
      const int r0 = 16 * w + gq;
#pragma unroll
      for (int nt = 0; nt < HC / 8; ++nt) {
        *reinterpret_cast<float2 *>(&hbuf[r0 * HC + nt * 8 + 2 * cq]) = make_float2(hacc[nt][0], hacc[nt][1]);
        *reinterpret_cast<float2 *>(&hbuf[(r0 + 8) * HC + nt * 8 + 2 * cq]) = make_float2(hacc[nt][2], hacc[nt][3]);
      }
      for (int c = 0; c < cl; ++c)
        if (c != (int)crank) mbar_arrive_remote(hready, c);
      if (!wait_all<true>(hready, 0)) ok = false;
      if (ok && rows_live) {
#pragma unroll
        for (int nt = 0; nt < HC / 8; ++nt) {
          float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
          for (int c = 0; c < cl; ++c) {
            float2 v0, v1;
            if (c == (int)crank) {
              v0 = make_float2(hacc[nt][0], hacc[nt][1]);
              v1 = make_float2(hacc[nt][2], hacc[nt][3]);
            } else {
              v0 = ld_dsmem_f2(&hbuf[r0 * HC + nt * 8 + 2 * cq], c);
              v1 = ld_dsmem_f2(&hbuf[(r0 + 8) * HC + nt * 8 + 2 * cq], c);
            }
            s0.x += v0.x; s0.y += v0.y; s1.x += v1.x; s1.y += v1.y;
          }
          hacc[nt][0] = s0.x; hacc[nt][1] = s0.y; hacc[nt][2] = s1.x; hacc[nt][3] = s1.y;
        }
      }
      for (int c = 0; c < cl; ++c)
        if (c != (int)crank) mbar_arrive_remote(hdone, c);
      wait_all<true>(hdone, 0);       // peers are done reading this CTA's part of the ring
      mbar_arrive(xready);            // the loader may refill the ring
    }
    if (MODE == kShrink) {
      // write h rows (< len) and columns j < rank; cluster CTA c writes the rows of warps w % cl == c
      if (ok && rows_live && (w % cl) == (int)crank) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = 16 * w + gq + 8 * hf;
          if (r >= len) continue;
          float *hrow = p.h + (int64_t)p.perm[start + r] * p.ldh;
#pragma unroll
          for (int nt = 0; nt < HC / 8; ++nt) {
            const int c = nt * 8 + 2 * cq;
            if (c < n * R && (c % R) < rank) hrow[c] = hacc[nt][2 * hf];
            if (c + 1 < n * R && ((c + 1) % R) < rank) hrow[c + 1] = hacc[nt][2 * hf + 1];
          }
        }
      }
      pdl_launch_dependents();
      return;
    }
  } else {
    // expand: h rows of the tile from global memory (columns past the rank are masked)
    if (rows_live) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = 16 * w + gq + 8 * hf;
        if (r >= len) continue;
        const float *hrow = p.h + (int64_t)p.perm[start + r] * p.ldh;
#pragma unroll
        for (int nt = 0; nt < HC / 8; ++nt) {
          const int c = nt * 8 + 2 * cq;
          if (c < n * R && (c % R) < rank) hacc[nt][2 * hf] = __ldg(&hrow[c]);
          if (c + 1 < n * R && ((c + 1) % R) < rank) hacc[nt][2 * hf + 1] = __ldg(&hrow[c + 1]);
        }
      }
    }
  }

  // ------------------------------------------------------------------ phase 2
  uint32_t ahi[HC / 16][4], alo[HC / 16][4];
#pragma unroll
  for (int q = 0; q < HC / 16; ++q) {
    split_bf16(hacc[2 * q][0], hacc[2 * q][1], ahi[q][0], alo[q][0]);
    split_bf16(hacc[2 * q][2], hacc[2 * q][3], ahi[q][1], alo[q][1]);
    split_bf16(hacc[2 * q + 1][0], hacc[2 * q + 1][1], ahi[q][2], alo[q][2]);
    split_bf16(hacc[2 * q + 1][2], hacc[2 * q + 1][3], ahi[q][3], alo[q][3]);
  }
  const float sc = p.scal[slot];
  for (; ok && g < ntiles; ++g) {
    const int s = g % NS;
    if (!(ok = wait_all(&full[s], (g / NS) & 1))) break;
    uint8_t *st = smem + s * C::STAGE;
    if (rows_live) {
      int i, c0, ocols;
      blk(b_beg + g - n1, i, c0, ocols);
      const uint32_t bb = smem_u32(st) + MBM * XP;
      float acc[8][4];
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
      const int cs = i * R;   // first h column of slice i
#pragma unroll
      for (int q = 0; q < HC / 16; ++q) {
        if (q * 16 < cs || q * 16 >= cs + rank) continue;
        const int j0 = q * 16 - cs;
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b[4];
          ldb_p(bb, bp, np * 16, j0, b);
          b[0] = mask_pair(b[0], j0 + 2 * cq, rank);
          b[1] = mask_pair(b[1], j0 + 8 + 2 * cq, rank);
          b[2] = mask_pair(b[2], j0 + 2 * cq, rank);
          b[3] = mask_pair(b[3], j0 + 8 + 2 * cq, rank);
          mma_bf16(acc[2 * np], ahi[q], b[0], b[1]);
          mma_bf16(acc[2 * np], alo[q], b[0], b[1]);
          mma_bf16(acc[2 * np + 1], ahi[q], b[2], b[3]);
          mma_bf16(acc[2 * np + 1], alo[q], b[2], b[3]);
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
          uint32_t *yp = reinterpret_cast<uint32_t *>(st + r * XP + cc * 2);
          const float2 yv = unpack_bf16(*yp);
          *yp = pack_bf16(yv.x + sc * acc[nt][2 * hf], yv.y + sc * acc[nt][2 * hf + 1]);
        }
      }
    }
    fence_proxy_async_smem();
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
  int nw = (int)std::min<int64_t>(32, std::max<int64_t>(1, (160 * 1024 / 4 - 256) / S));
  nw = std::min(nw, 32);
  const size_t smem = (size_t)(nw * S + 160) * 4;
  LORA_CUDA(ensure_smem((const void *)group_kernel, smem));
  LORA_CUDA(launch(group_kernel, dim3(1), dim3(nw * 32), smem, st, 1, true, ad.slots, ad.num_tokens, S,
                   ad.max_rank, ranks, counts, perm, num_active, header, tiles, (int)MBM));
  return LORA_OK;
}

template <int HC, int MODE>
lora_status_t launch_seg(SegArgs a, int64_t T, cudaStream_t st) {
  auto kern = seg_kernel<HC, MODE>;
  const size_t smem = SegCfg<HC>::BYTES;
  LORA_CUDA(ensure_smem((const void *)kern, smem));
  const int occ = occupancy((const void *)kern, MTHREADS, smem);
  const int64_t tiles = max_tiles(T, a.S);
  const int64_t cap = (int64_t)occ * num_sms();
  int cl = 1;
  while (cl * 2 <= 8 && tiles * cl * 2 <= cap) cl *= 2;
  if (MODE != kExpand)
    while (cl > 1 && ceil_div(a.in, KW) < cl) cl /= 2;
  if (MODE != kShrink)
    while (cl > 1 && a.nb < cl) cl /= 2;
  a.cl = cl;
  LORA_CUDA(launch(kern, dim3((unsigned)(tiles * cl)), dim3(MTHREADS), smem, st, cl, true, a));
  return LORA_OK;
}

template <int MODE>
lora_status_t dispatch_seg(SegArgs a, int64_t T, cudaStream_t st) {
  const int hc = a.n * a.R;
  if (hc <= 64) return launch_seg<64, MODE>(a, T, st);
  if (hc <= 128) return launch_seg<128, MODE>(a, T, st);
  if (hc <= 192) return launch_seg<192, MODE>(a, T, st);
  return launch_seg<256, MODE>(a, T, st);
}

// Shared argument checks of the segmented ops (beyond those of the ABI layer).
lora_status_t check_seg(const MultiArgs &m, bool need_in, bool need_out) {
  const int R = m.addr.max_rank;
  if ((int64_t)m.n * R > kMaxHC) return LORA_ERR_UNSUPPORTED;
  if (R % 8 != 0 || (m.n > 1 && R % 16 != 0)) return LORA_ERR_UNSUPPORTED;
  if (need_in && m.in % 8 != 0) return LORA_ERR_UNSUPPORTED;
  if (need_out) {
    for (int i = 0; i < m.n; ++i)
      if (m.out_slices[i] % 8 != 0) return LORA_ERR_UNSUPPORTED;
    if (m.sb_col != 1) return LORA_ERR_UNSUPPORTED;   // b rows must be contiguous along the rank
    if (!aligned16(m.b) || (m.sb_row * 2) % 16 != 0 || (m.sb_slot * 2) % 16 != 0) return LORA_ERR_ALIGNMENT;
  }
  return LORA_OK;
}

SegArgs seg_args(const MultiArgs &m, const SchedPtrs &sp) {
  SegArgs a{};
  a.slots = m.addr.slots;
  a.ranks = m.ranks;
  a.scal = m.scalings;
  a.header = sp.header;
  a.tiles = sp.tiles;
  a.perm = sp.perm;
  a.T = m.addr.num_tokens;
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
  int off = 0, nb = 0;
  for (int i = 0; i < m.n; ++i) {
    a.off[i] = off;
    a.blk0[i] = nb;
    off += m.out_slices[i];
    nb += (m.out_slices[i] + CBW - 1) / CBW;
  }
  a.off[m.n] = off;
  a.blk0[m.n] = nb;
  a.nb = nb;
  return a;
}

}  // namespace

size_t multi_ws_bytes(int op, int64_t T, int64_t in, int64_t O, int R, int S) {
  (void)in;
  (void)O;
  (void)R;
  if (op == LORA_OP_GROUP_BY_SLOT || op == LORA_OP_SHRINK || op == LORA_OP_EXPAND || op == LORA_OP_APPLY_LINEAR)
    return T > 0 ? sched_bytes(T, S) : 0;
  return 0;
}

lora_status_t group_by_slot(const lora_addressing_t &addr, const int32_t *ranks, int32_t *counts, int32_t *perm,
                            int32_t *num_active, void *ws, size_t ws_bytes, cudaStream_t st) {
  WsCarver c(ws, ws_bytes);
  SchedPtrs sp;
  if (addr.num_tokens > 0 && !carve_sched(c, addr.num_tokens, addr.num_slots, sp)) return LORA_ERR_WORKSPACE;
  if (addr.num_tokens == 0) {
    // no tokens: counts are zero, no active tokens
    LORA_CUDA(cudaMemsetAsync(counts, 0, (size_t)addr.num_slots * 4, st));
    LORA_CUDA(cudaMemsetAsync(num_active, 0, 4, st));
    return LORA_OK;
  }
  return launch_group(addr, ranks, counts, perm, num_active, sp.header, sp.tiles, st);
}

static lora_status_t schedule(const MultiArgs &m, void *ws, size_t ws_bytes, SchedPtrs &sp, cudaStream_t st) {
  WsCarver c(ws, ws_bytes);
  if (!carve_sched(c, m.addr.num_tokens, m.addr.num_slots, sp)) return LORA_ERR_WORKSPACE;
  return launch_group(m.addr, m.ranks, sp.counts, sp.perm, sp.header, sp.header, sp.tiles, st);
}

lora_status_t shrink(MultiArgs m, void *ws, size_t ws_bytes, cudaStream_t st) {
  LORA_TRY(check_seg(m, true, false));
  SchedPtrs sp;
  LORA_TRY(schedule(m, ws, ws_bytes, sp, st));
  return dispatch_seg<kShrink>(seg_args(m, sp), m.addr.num_tokens, st);
}

lora_status_t expand(MultiArgs m, void *ws, size_t ws_bytes, cudaStream_t st) {
  LORA_TRY(check_seg(m, false, true));
  SchedPtrs sp;
  LORA_TRY(schedule(m, ws, ws_bytes, sp, st));
  return dispatch_seg<kExpand>(seg_args(m, sp), m.addr.num_tokens, st);
}

lora_status_t apply_linear(MultiArgs m, void *ws, size_t ws_bytes, cudaStream_t st) {
  LORA_TRY(check_seg(m, true, true));
  SchedPtrs sp;
  LORA_TRY(schedule(m, ws, ws_bytes, sp, st));
  return dispatch_seg<kApply>(seg_args(m, sp), m.addr.num_tokens, st);
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
