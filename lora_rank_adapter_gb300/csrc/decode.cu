// decode.cu -- the multi-adapter shrink of decode batches (a few tokens per
// adapter slot), on CUDA cores fed by TMA.
//
// Operation (mstar page "mstar.engine.resources.lora.ops", shrink):
//   h[t, i*R + j] = x[t] . a[slot(t)][i*R + j]              (j < rank)
// over the slot-sorted tiles (at most four tokens of one slot) that the
// grouping kernel lists on the device.
//
// A decode batch gives each slot one to a few tokens, so the work is streaming
// the slots' adapter rows: each a element meets one to four x values.  The
// fifth-generation tensor cores do not pay here: a 128-row tcgen05 MMA would
// carry a handful of useful rows, and its issue rate, not memory, would set the
// pace.  Neither do plain FMAs: unpacking and multiplying every element costs
// more instructions than the SM can issue at HBM speed.  The contraction runs
// instead on warp-level mma.sync m16n8k16: A = 16 adapter rows x 16 columns,
// B = the tile's (at most four) token rows, fp32 accumulators in registers; one
// instruction covers 512 bytes of a.
//
// One persistent kernel (one CTA per SM), warp 0 loading, warps 1..8 computing:
//   chunks  (tile, 256 columns of `in`) are split over the grid by cost: a chunk
//           of tile t weighs n * round8(rank) adapter rows + len token rows + a
//           fixed C0, and CTA i takes the chunks whose cost position falls in
//           [W i / G, W (i + 1) / G).  The grouping kernel lists the running sum
//           of round8(rank) per tile, so a CTA finds its first chunk with one
//           parallel pass over the tile list.
//   stages  hold q consecutive chunks of one tile (as many as fit 40 KB), or,
//           for tiles with more than 64 adapter rows, one chunk's rows in blocks
//           of 64.  A chunk's x rows arrive as one 256-column box per token; its
//           a rows as boxes of 8 rows x 4 x 64 columns (a four-dimensional view
//           of the stack whose third dimension steps 64 columns along the row),
//           in the 128-byte swizzle that ldmatrix reads without bank conflicts:
//           exactly round8(rank) rows per slice.  The copies are dealt over the
//           loader's lanes.
//   compute warp w takes the 16-row group w % ngr of the tile's rows and every
//           (8 / ngr)-th 16-column step of each chunk; its fragments accumulate
//           over the CTA's chunks of the tile, and at the tile's end the warps
//           of a row group add theirs through shared memory, in warp order.  A
//           tile cut between CTAs leaves fp32 partial sums that the last CTA of
//           the tile adds in CTA order (deterministic).
#include <algorithm>
#include <cstddef>
#include <cstring>

#include "common.cuh"
#include "decode.h"
#include "host_common.h"
#include "multi.h"
#include "tc_common.cuh"

namespace lora {
namespace dec {

constexpr int CH = 256;                       // columns of a chunk
constexpr int ROWB = CH * 2;                  // bytes of one row of a chunk
constexpr int XB = kDecTokens * ROWB;         // x area of a chunk (four token rows)
constexpr int NCW = 8;                        // compute warps
constexpr int NTHR = 32 * (NCW + 1);          // warp 0 loads
constexpr int STAGE = 40 * 1024;
constexpr int NS = 5;
constexpr int kRing = NS * STAGE;
constexpr int kScr = NCW * 4 * 4 * 32 * 4;    // fragments of the tile-end exchange (four row blocks)
constexpr int kSmem = kRing + kScr;
constexpr int GB = 8 * 4 * 128;               // one 8-row group of a chunk: 8 rows x 4 x 64 columns
constexpr int kMaxQ = 16;                     // chunks per stage
constexpr int RB = 64;                        // adapter rows of a stage at most
constexpr int C0 = 8;                         // fixed cost of a chunk (copy issue, stage hand-offs), in 512-byte rows

// Warp-uniform bounded wait, polled by lane 0.
__device__ __forceinline__ bool wait_lane0(uint64_t *bar, uint32_t parity) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity);
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// The cost split of the chunks over the grid.
struct Split {
  int nk, n, tw, G;           // units per tile, adapter-row weight, token-row weight
  int64_t W;
  // first cost position of tile t (rows8 = its running sum of round8(rank))
  __device__ int64_t base(int t, int start, int rows8) const {
    return (int64_t)nk * ((int64_t)n * rows8 + (int64_t)tw * start + (int64_t)C0 * t);
  }
  // the CTA whose run holds the chunk at cost position cs
  __device__ int owner(int64_t cs) const {
    const int64_t o = cs * G / W;
    return o < G - 1 ? (int)o : G - 1;
  }
  // first cost position of CTA i's run
  __device__ int64_t begin(int i) const { return (W * i + G - 1) / G; }
};

struct Tile {
  int slot, start, len, rank, r8, nrow, nrb, q;
  int64_t base, w;   // first cost position, cost per chunk
};
__device__ __forceinline__ Tile load_tile(const DecArgs &p, const Split &sp, int tile, int ntiles) {
  const int4 td = p.tiles[tile];
  const int rows_next = tile + 1 < ntiles ? p.tiles[tile + 1].w : p.header[2];
  Tile t;
  t.slot = td.x;
  t.start = td.y;
  t.len = td.z;
  t.r8 = rows_next - td.w;
  t.rank = min(p.ranks[t.slot], t.r8);
  t.nrow = p.n * t.r8;
  t.nrb = (t.nrow + RB - 1) / RB;
  t.q = t.nrb == 1 ? max(1, min(kMaxQ, STAGE / (XB + t.nrow * ROWB))) : 1;
  t.base = sp.base(tile, t.start, td.w);
  t.w = (int64_t)t.nrow + t.len + C0;
  return t;
}

// The chunks [kb, ke) of a tile inside the run [u0, u1).
__device__ __forceinline__ void tile_chunks(int64_t tile, int64_t u0, int64_t u1, int nk, int &kb, int &ke) {
  kb = tile == u0 / nk ? (int)(u0 % nk) : 0;
  ke = tile == (u1 - 1) / nk ? (int)((u1 - 1) % nk) + 1 : nk;
}

// Stage si of a tile's run: chunks [k0, k0 + nq), adapter rows [r0, r0 + nr).
struct Stage {
  int k0, nq, r0, nr;
};
__device__ __forceinline__ int num_stages(const Tile &t, int kb, int ke) {
  return t.nrb == 1 ? (ke - kb + t.q - 1) / t.q : (ke - kb) * t.nrb;
}
__device__ __forceinline__ Stage stage_of(const Tile &t, int kb, int ke, int si) {
  Stage s;
  if (t.nrb == 1) {
    s.k0 = kb + si * t.q;
    s.nq = min(t.q, ke - s.k0);
    s.r0 = 0;
    s.nr = t.nrow;
  } else {
    s.k0 = kb + si / t.nrb;
    s.nq = 1;
    s.r0 = (si % t.nrb) * RB;
    s.nr = min(RB, t.nrow - s.r0);
  }
  return s;
}

// ============================================================================= the kernel
// RBK: 64-row blocks of a tile's adapter rows at most (n * round8(R) / 64, rounded up to 1, 2 or 4).
template <int RBK>
__global__ void __launch_bounds__(NTHR, 1)
    shrink_dec_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmA, DecArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *scr = reinterpret_cast<float *>(ring + kRing);
  uint64_t *full = reinterpret_cast<uint64_t *>(ring + kSmem), *empty = full + NS;
  int64_t *s_run = reinterpret_cast<int64_t *>(empty + NS);   // first and end chunk of this CTA's run
  int *s_flag = reinterpret_cast<int *>(s_run + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    fence_barrier_init();
    s_run[0] = s_run[1] = 0;
  }
  __syncthreads();
  pdl_wait();
  // the cost split: W is the total cost; G CTAs take runs of at least the
  // largest chunk cost, so that every run holds a chunk
  const int ntiles = p.header[1];
  Split sp;
  sp.nk = p.nk;
  sp.n = p.n;
  sp.tw = 1;
  sp.W = (int64_t)p.nk * ((int64_t)p.n * p.header[2] + p.header[0] + (int64_t)C0 * ntiles);
  const int64_t wmax = (int64_t)p.n * ((p.R + 7) & ~7) + kDecTokens + C0, gw = sp.W / wmax;
  sp.G = gw < 1 ? 1 : gw < (int64_t)gridDim.x ? (int)gw : (int)gridDim.x;
  const int cta = blockIdx.x;
  const bool active = sp.W > 0 && cta < sp.G;
  if (active) {
    // the chunks at cost positions begin(cta) and begin(cta + 1): each thread
    // checks the tiles threadIdx.x, threadIdx.x + NTHR, ...
    const int64_t a0 = sp.begin(cta), a1 = sp.begin(cta + 1);
    for (int t = threadIdx.x; t < ntiles; t += NTHR) {
      const int4 td = p.tiles[t];
      const int rn = t + 1 < ntiles ? p.tiles[t + 1].w : p.header[2];
      const int64_t base = sp.base(t, td.y, td.w), w = (int64_t)p.n * (rn - td.w) + td.z + C0;
      const int64_t end = base + (int64_t)p.nk * w;
      if (a0 >= base && a0 < end) s_run[0] = (int64_t)t * p.nk + (a0 - base + w - 1) / w;
      if (a1 >= base && a1 < end) s_run[1] = (int64_t)t * p.nk + (a1 - base + w - 1) / w;
    }
    if (threadIdx.x == 0 && a1 >= sp.W) s_run[1] = (int64_t)ntiles * p.nk;
  }
  __syncthreads();
  const int64_t u0 = active ? s_run[0] : 0, u1 = active ? s_run[1] : 0;
  const int nk = p.nk;
  const int64_t tb0 = u0 < u1 ? u0 / nk : 0, tb1 = u0 < u1 ? (u1 - 1) / nk : -1;

  if (warp == 0) {
    // ------------------------------------------------------------------ loader warp
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmA);
    }
    int g = 0;
    bool ok = true;
    for (int64_t tile = tb0; ok && tile <= tb1; ++tile) {
      const Tile t = load_tile(p, sp, (int)tile, ntiles);
      const int aslot = p.a_one_slot ? 0 : t.slot;
      int rows[kDecTokens];
#pragma unroll
      for (int e = 0; e < kDecTokens; ++e) rows[e] = e < t.len ? p.perm[t.start + e] : 0;
      int kb, ke;
      tile_chunks(tile, u0, u1, nk, kb, ke);
      const int nst = num_stages(t, kb, ke);
      for (int si = 0; si < nst; ++si, ++g) {
        const Stage st = stage_of(t, kb, ke, si);
        const int s = g % NS;
        if (g >= NS && !(ok = wait_lane0(&empty[s], ((g / NS) & 1) ^ 1))) break;
        uint8_t *sx = ring + s * STAGE, *sa = sx + st.nq * XB;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(st.nq * (t.len + st.nr) * ROWB));
        __syncwarp();
        // per chunk: len token rows, then nr / 8 adapter boxes; dealt over the lanes
        const int per = t.len + st.nr / 8;
        for (int idx = lane; idx < st.nq * per; idx += 32) {
          const int kq = idx / per, e = idx - kq * per, col = (st.k0 + kq) * CH;
          if (e < t.len) {
            int r = rows[0];
#pragma unroll
            for (int k = 1; k < kDecTokens; ++k)
              if (e == k) r = rows[k];
            tma_load_2d(sx + kq * XB + e * ROWB, &tmX, &full[s], col, r);
          } else {
            const int gi = e - t.len, rr = st.r0 + 8 * gi, sl = rr / t.r8, j = rr - sl * t.r8;
            tma_load_4d(sa + (kq * (st.nr / 8) + gi) * GB, &tmA, &full[s], 0, sl * p.R + j, (st.k0 + kq) * 4, aslot);
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ compute warps
    const int w = warp - 1, tid = threadIdx.x - 32;
    bool ok = true;   // after a timed-out wait: skip the work, keep the barrier sequence
    int g = 0;
    for (int64_t tile = tb0; tile <= tb1; ++tile) {
      const Tile t = load_tile(p, sp, (int)tile, ntiles);
      // row groups of 16 per 64-row block, as a power of two; warp w takes group
      // w % ngp and the 16-column steps ks = w / ngp (mod 8 / ngp)
      const int ngr = t.nrb == 1 ? (t.nrow + 15) / 16 : 4, ngp = ngr <= 1 ? 1 : ngr <= 2 ? 2 : 4;
      const int rg = w % ngp, ph = w / ngp, nph = NCW / ngp;
      float acc[RBK][4];
#pragma unroll
      for (int b = 0; b < RBK; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[b][e] = 0.f;
      int kb, ke;
      tile_chunks(tile, u0, u1, nk, kb, ke);
      const int nst = num_stages(t, kb, ke);
      // B fragments: token n = lane / 4 (zero past the tile's tokens), columns 2 (lane % 4) + {0, 1} (+ 8)
      const int bn = lane >> 2, bk = (lane & 3) << 1;
      for (int si = 0; si < nst; ++si, ++g) {
        const Stage st = stage_of(t, kb, ke, si);
        const int s = g % NS;
        if (ok) ok = wait_lane0(&full[s], (g / NS) & 1);
        if (ok && 16 * rg < st.nr) {
          const uint8_t *sx = ring + s * STAGE;
          const uint32_t sa = smem_u32(sx + st.nq * XB);
          // ldmatrix rows: lane l gives row l % 8 of 8-row group 2 rg + (l / 8) % 2 (past the
          // stage's rows: its last group, whose products are never written out) and the
          // 16-byte column group 2 (ks % 4) + l / 16 of sub-chunk ks / 4, swizzled
          const int gl = min(2 * rg + ((lane >> 3) & 1), st.nr / 8 - 1), lr = lane & 7, hi = lane >> 4;
#pragma unroll
          for (int b = 0; b < RBK; ++b) {
            if (b != st.r0 / RB) continue;
            for (int kq = 0; kq < st.nq; ++kq) {
              const uint32_t ga = sa + (uint32_t)((kq * (st.nr / 8) + gl) * GB + lr * 128);
              const uint8_t *xr = sx + kq * XB + bn * ROWB;
              for (int ks = ph; ks < 16; ks += nph) {
                uint32_t af[4];
                ldsm_x4(ga + (ks >> 2) * 1024 + (((((ks & 3) << 1) | hi) ^ lr) << 4), af[0], af[1], af[2], af[3]);
                const int k0 = 16 * ks + bk;
                const uint32_t b0 = bn < t.len ? *reinterpret_cast<const uint32_t *>(xr + k0 * 2) : 0u;
                const uint32_t b1 = bn < t.len ? *reinterpret_cast<const uint32_t *>(xr + (k0 + 8) * 2) : 0u;
                mma_bf16(acc[b], af, b0, b1);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      // the warps of a row group add their fragments in warp order
#pragma unroll
      for (int b = 0; b < RBK; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e) scr[((w * RBK + b) * 4 + e) * 32 + lane] = acc[b][e];
      named_bar_sync(1, 32 * NCW);
      if (ph == 0) {
#pragma unroll
        for (int b = 0; b < RBK; ++b)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v = 0.f;
            for (int q = 0; q < nph; ++q) v += scr[(((rg + ngp * q) * RBK + b) * 4 + e) * 32 + lane];
            acc[b][e] = v;
          }
      }
      named_bar_sync(1, 32 * NCW);
      const int first = sp.owner(t.base), last_cta = sp.owner(t.base + (int64_t)(nk - 1) * t.w);
      const bool whole = first == last_cta;
      const int ncm = p.n * ((p.R + 7) & ~7);
      float *mypart = p.part + (2 * (int64_t)cta + (tile == tb0 ? 0 : 1)) * kDecTokens * ncm;
      // fragment entry e of lane l: row 16 rg + l / 4 (+ 8 for e >= 2) of block b, token 2 (l % 4) + e % 2
      if (ph == 0) {
#pragma unroll
        for (int b = 0; b < RBK; ++b)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int rr = RB * b + 16 * rg + (lane >> 2) + (e >> 1) * 8, tk = bk + (e & 1);
            if (b >= t.nrb || rr >= t.nrow || tk >= kDecTokens) continue;
            if (whole) {
              const int sl = rr / t.r8, j = rr - sl * t.r8;
              if (tk < t.len && j < t.rank) p.h[(int64_t)p.perm[t.start + tk] * p.ldh + sl * p.R + j] = acc[b][e];
            } else {
              __stcg(mypart + tk * ncm + rr, acc[b][e]);
            }
          }
      }
      if (whole) continue;
      __threadfence();
      named_bar_sync(1, 32 * NCW);
      if (tid == 0) *s_flag = atomicAdd(p.counters + tile, 1) == last_cta - first;
      named_bar_sync(1, 32 * NCW);
      if (*s_flag) {
        __threadfence();
        // the CTA that owns the tile's first chunk keeps it in slot 1 when its
        // run started in an earlier tile (it owns the chunk before the tile too)
        int first_slot = 0;
        if (tile > 0) {
          const int4 tp = p.tiles[tile - 1];
          const int64_t wprev = (int64_t)p.n * (p.tiles[tile].w - tp.w) + tp.z + C0;
          first_slot = sp.owner(t.base - wprev) == first ? 1 : 0;
        }
        for (int q = tid; q < kDecTokens * t.nrow; q += 32 * NCW) {
          const int e = q / t.nrow, rr = q - e * t.nrow;
          float v = 0.f;
          for (int c = first; c <= last_cta; ++c) {
            const int64_t slot = 2 * (int64_t)c + (c == first ? first_slot : 0);
            v += __ldcg(p.part + slot * kDecTokens * ncm + e * ncm + rr);
          }
          const int sl = rr / t.r8, j = rr - sl * t.r8;
          if (e < t.len && j < t.rank) p.h[(int64_t)p.perm[t.start + e] * p.ldh + sl * p.R + j] = v;
        }
        if (tid == 0) p.counters[tile] = 0;   // ready for the next call
      }
      named_bar_sync(1, 32 * NCW);
    }
  }
  pdl_launch_dependents();
}

// ============================================================================= expand
// Units (tile, 256 output columns of slice i) are split over the grid by cost.
// HBM serves whole 128-byte lines, so a unit's 256 rows of b cost the same
// whatever the slot's rank (min(R, 64) entries of each row are fetched): a unit
// weighs that fixed b cost + two token rows of y + C0.  No unit shares an
// output with another, so a CTA's run needs no reduction.  A stage holds up to
// q units of one tile and slice: per unit the tile's y row segments (one
// 256-column box per token, updated in place) and round8(rank) rank entries of
// 256 rows of b as boxes of 64, 32, 16 and 8 entries (one TMA row request per
// box row; swizzled so that the fragment loads hit distinct banks).  Compute
// warp w takes the 8-column groups w, w + 8, w + 16, w + 24 of each unit:
// mma.sync with A = the tile's h rows rounded to bf16 once (relative error
// 2^-9 per term, well inside what the bf16 result of the add holds, as in the
// prefill expand) and B = the b pieces (entries past the rank
// masked: b may hold anything there), then y += scal * D in shared memory;
// after a barrier one thread stores the updated rows with TMA stores.
constexpr int ECB = 256;                     // output columns of a unit
constexpr int EYB = ECB * 2;                 // bytes of a y row segment
constexpr int EYA = kDecTokens * EYB;        // y area of a unit
constexpr int EGB = ECB * 16;                // one box of b: 256 rows x 8 entries

struct ExpTile {
  int slot, start, len, rank, r8, ng, q;
};
__device__ __forceinline__ ExpTile exp_tile(const DecExpArgs &p, int tile, int ntiles) {
  const int4 td = p.tiles[tile];
  const int rows_next = tile + 1 < ntiles ? p.tiles[tile + 1].w : p.header[2];
  ExpTile t;
  t.slot = td.x;
  t.start = td.y;
  t.len = td.z;
  t.r8 = rows_next - td.w;
  t.rank = min(p.ranks[t.slot], t.r8);
  t.ng = t.r8 / 8;
  t.q = max(1, min(kMaxQ, STAGE / (EYA + t.ng * EGB)));
  return t;
}
// Box k of the round8(rank) entries (64, 32, 16 or 8 wide, largest first): its
// width index (0: 8 ... 3: 64) and first entry; at most three boxes since
// round8(rank) <= 72.  A unit's b area holds the boxes in this order, box k at
// byte j0[k] * 512 (256 rows of j0[k] entries before it).
struct ExpBoxes {
  int n, wi[3], j0[3];
};
__device__ __forceinline__ int widest(int v) { return v >= 64 ? 3 : v >= 32 ? 2 : v >= 16 ? 1 : 0; }
__device__ __forceinline__ ExpBoxes exp_boxes(int r8) {
  ExpBoxes b;
  b.wi[0] = widest(r8);
  b.j0[0] = 0;
  const int r1 = r8 - (8 << b.wi[0]);
  b.wi[1] = widest(r1);
  b.j0[1] = 8 << b.wi[0];
  const int r2 = r1 - (r1 > 0 ? 8 << b.wi[1] : 0);
  b.wi[2] = widest(r2);
  b.j0[2] = b.j0[1] + (8 << b.wi[1]);
  b.n = r1 <= 0 ? 1 : r2 <= 0 ? 2 : 3;
  return b;
}
// Byte offset of entries (j, j + 1) of row c in a unit's b area (j even, j < r8),
// written as off + (c / 8) * stride: the swizzle of a row depends on c % 8 only.
__device__ __forceinline__ void exp_boff(const ExpBoxes &bx, int c8, int j, int &off, int &stride) {
  int wi = bx.wi[0], j0 = 0;
  if (bx.n > 1 && j >= bx.j0[1]) {
    wi = bx.wi[1];
    j0 = bx.j0[1];
  }
  if (bx.n > 2 && j >= bx.j0[2]) {
    wi = bx.wi[2];
    j0 = bx.j0[2];
  }
  const int jj = j - j0, ch = jj >> 3;
  // 16-byte chunk ch of a (16 << wi)-byte row, swizzled as the copy wrote it
  const int sw = wi == 3 ? c8 : wi == 2 ? ((c8 >> 1) & 3) : wi == 1 ? ((c8 >> 2) & 1) : 0;
  off = j0 * ECB * 2 + c8 * (16 << wi) + ((ch ^ sw) << 4) + (jj & 7) * 2;
  stride = 8 * (16 << wi);
}
// The slice holding unit u of a tile, and its end.
__device__ __forceinline__ int slice_of(const DecExpArgs &p, int u) {
  int i = 0;
  while (i + 1 < p.n && p.blk0[i + 1] <= u) ++i;
  return i;
}

// Warp 0 loads, warps 1..8 compute, warp 9 stores the updated y rows.  Only
// the loader walks the tile list (it runs stages ahead, so the latency of
// those reads is hidden): before arming a stage it writes the stage's header
// (tile, slice, columns, token rows, scale) and the tile's h rows of the slice
// into shared memory, where the compute and store warps read them.
constexpr int ECW = 8;                       // compute warps of the expand
constexpr int ESW = ECW + 1;
constexpr int NTHR_E = 32 * (ECW + 2);
constexpr int EHR = 80;                      // h entries per token row in a header (round16(72))

// h first: the compute warps read it as float2 pairs (8-byte aligned)
struct __align__(16) ExpHdr {
  float h[kDecTokens][EHR];   // zero past the rank and past the tile's tokens
  int rows[kDecTokens];
  int len, rank, r8, i, c0, nq, last;
  float sc;
};
static_assert(offsetof(ExpHdr, h) == 0 && (EHR * 4) % 16 == 0, "header rows must stay 16-byte aligned");
constexpr int kHdr = (int)((sizeof(ExpHdr) + 127) / 128 * 128);

// KS: 16-entry steps of the rank at most (round16(R) / 16).
template <int KS>
__global__ void __launch_bounds__(NTHR_E, 1)
    expand_dec_kernel(const __grid_constant__ DecExpMaps mp, DecExpArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *hdr_base = ring + kRing;
  uint64_t *full = reinterpret_cast<uint64_t *>(hdr_base + NS * kHdr), *empty = full + NS, *ydone = empty + NS;
  int64_t *s_run = reinterpret_cast<int64_t *>(ydone + NS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&ydone[s], ECW);
    }
    fence_barrier_init();
    s_run[0] = s_run[1] = 0;
  }
  __syncthreads();
  pdl_wait();
  // the cost split: a tile's unit weighs round8(rank) + 2 len + C0
  const int ntiles = p.header[1];
  Split sp;
  sp.nk = p.nbu;
  sp.n = 1;
  sp.tw = 2;
  sp.W = (int64_t)p.nbu * ((int64_t)p.header[2] + 2 * (int64_t)p.header[0] + (int64_t)C0 * ntiles);
  sp.G = (int)gridDim.x;
  const int cta = blockIdx.x;
  const bool active = sp.W > 0;
  if (active) {
    const int64_t a0 = sp.begin(cta), a1 = sp.begin(cta + 1);
    for (int t = threadIdx.x; t < ntiles; t += NTHR_E) {
      const int4 td = p.tiles[t];
      const int rn = t + 1 < ntiles ? p.tiles[t + 1].w : p.header[2];
      const int64_t base = sp.base(t, td.y, td.w), w = (int64_t)(rn - td.w) + 2 * td.z + C0;
      const int64_t end = base + (int64_t)p.nbu * w;
      if (a0 >= base && a0 < end) s_run[0] = (int64_t)t * p.nbu + (a0 - base + w - 1) / w;
      if (a1 >= base && a1 < end) s_run[1] = (int64_t)t * p.nbu + (a1 - base + w - 1) / w;
    }
    // the whole grid takes part, so with W < G the last runs begin at W: empty
    if (threadIdx.x == 0 && a0 >= sp.W) s_run[0] = (int64_t)ntiles * p.nbu;
    if (threadIdx.x == 0 && a1 >= sp.W) s_run[1] = (int64_t)ntiles * p.nbu;
  }
  __syncthreads();
  const int64_t u0 = active ? s_run[0] : 0, u1 = active ? s_run[1] : 0;
  const int nbu = p.nbu;
  const bool any = u0 < u1;
  const int64_t tb0 = any ? u0 / nbu : 0, tb1 = any ? (u1 - 1) / nbu : -1;

  if (warp == 0) {
    // ------------------------------------------------------------------ loader warp
    int g = 0;
    bool ok = true;
    for (int64_t tile = tb0; ok && tile <= tb1; ++tile) {
      const ExpTile t = exp_tile(p, (int)tile, ntiles);
      const ExpBoxes bx = exp_boxes(t.r8);
      const int bslot = p.b_one_slot ? 0 : t.slot;
      const float sc = p.scal[t.slot];
      int rows[kDecTokens];
#pragma unroll
      for (int e = 0; e < kDecTokens; ++e) rows[e] = e < t.len ? p.perm[t.start + e] : 0;
      int kb, ke;
      tile_chunks(tile, u0, u1, nbu, kb, ke);
      int cur_i = -1;
      float hv[kDecTokens * EHR / 32];   // this lane's h entries (e, j) = (idx / EHR, idx % EHR), idx = lane + 32 k
      for (int u = kb; u < ke; ++g) {
        const int i = slice_of(p, u), nq = min(min(t.q, ke - u), p.blk0[i + 1] - u), s = g % NS;
        const int c0 = (u - p.blk0[i]) * ECB;
        if (i != cur_i) {
          cur_i = i;
#pragma unroll
          for (int k = 0; k < kDecTokens * EHR / 32; ++k) {
            const int idx = lane + 32 * k, e = idx / EHR, j = idx - e * EHR;
            int r = rows[0];
#pragma unroll
            for (int q = 1; q < kDecTokens; ++q)
              if (e == q) r = rows[q];
            hv[k] = e < t.len && j < t.rank ? p.h[(int64_t)r * p.ldh + (int64_t)i * p.R + j] : 0.f;
          }
        }
        if (g >= NS && !(ok = wait_lane0(&empty[s], ((g / NS) & 1) ^ 1))) break;
        // the stage's header, then the barrier that publishes it with the copies
        ExpHdr *H = reinterpret_cast<ExpHdr *>(hdr_base + s * kHdr);
#pragma unroll
        for (int k = 0; k < kDecTokens * EHR / 32; ++k) {
          const int idx = lane + 32 * k, e = idx / EHR, j = idx - e * EHR;
          H->h[e][j] = hv[k];
        }
        if (lane == 0) {
          H->len = t.len;
          H->rank = t.rank;
          H->r8 = t.r8;
          H->i = i;
          H->c0 = c0;
          H->nq = nq;
          H->last = tile == tb1 && u + nq >= ke;
          H->sc = sc;
#pragma unroll
          for (int e = 0; e < kDecTokens; ++e) H->rows[e] = rows[e];
        }
        __syncwarp();
        uint8_t *sy = ring + s * STAGE, *sb = sy + nq * EYA;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(nq * (t.len * EYB + t.ng * EGB)));
        __syncwarp();
        const int per = t.len + bx.n;
        for (int idx = lane; idx < nq * per; idx += 32) {
          const int kq = idx / per, e = idx - kq * per, col = c0 + kq * ECB;
          if (e < t.len) {
            int r = rows[0];
#pragma unroll
            for (int k = 1; k < kDecTokens; ++k)
              if (e == k) r = rows[k];
            tma_load_2d(sy + (kq * kDecTokens + e) * EYB, &mp.y[i], &full[s], col, r);
          } else {
            const int k = e - t.len;
            const int wi = k == 0 ? bx.wi[0] : k == 1 ? bx.wi[1] : bx.wi[2];
            const int j0 = k == 0 ? 0 : k == 1 ? bx.j0[1] : bx.j0[2];
            const CUtensorMap *m = wi == 3 ? &mp.b[i][3] : wi == 2 ? &mp.b[i][2] : wi == 1 ? &mp.b[i][1] : &mp.b[i][0];
            tma_load_3d(sb + kq * t.ng * EGB + j0 * ECB * 2, m, &full[s], j0, col, bslot);
          }
        }
        u += nq;
      }
    }
  } else if (warp < ESW) {
    // ------------------------------------------------------------------ compute warps
    const int w = warp - 1;
    const int gm = lane >> 2, gt = (lane & 3) << 1;   // fragment row (token) / column pair
    int cur_r8 = -1, cur_rank = -1;
    int boff[KS][2], bstr[KS][2];
    uint32_t bmsk[KS][2];
    for (int g = 0; any; ++g) {
      const int s = g % NS;
      if (!wait_lane0(&full[s], (g / NS) & 1)) break;
      const ExpHdr *H = reinterpret_cast<const ExpHdr *>(hdr_base + s * kHdr);
      const int len = H->len, rank = H->rank, r8 = H->r8, nq = H->nq, last = H->last;
      const float sc = H->sc;
      if (r8 != cur_r8 || rank != cur_rank) {
        // this lane's B pieces: byte offset (8-column group 0), stride per
        // 8-column group and rank mask of entries 16 ks + 8 hf + gt, gt + 1
        cur_r8 = r8;
        cur_rank = rank;
        const ExpBoxes bx = exp_boxes(r8);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int j = 16 * ks + 8 * hf + gt;
            boff[ks][hf] = 0;
            bstr[ks][hf] = 0;
            if (j < r8) exp_boff(bx, gm, j, boff[ks][hf], bstr[ks][hf]);
            bmsk[ks][hf] = j >= rank ? 0u : j + 1 >= rank ? 0xffffu : 0xffffffffu;
          }
      }
      // A fragments a0 / a2 of the tile's h rows in bf16
      const int kst = (r8 + 15) / 16, ng = r8 / 8;
      uint32_t ahi[KS][2];
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int j = 16 * ks + 8 * hf + gt;   // below 16 kst <= EHR when ks < kst
          float2 v = make_float2(0.f, 0.f);
          if (ks < kst && gm < kDecTokens) v = *reinterpret_cast<const float2 *>(&H->h[gm][j]);
          ahi[ks][hf] = pack_bf16(v.x, v.y);
        }
      uint8_t *sy = ring + s * STAGE;
      const uint8_t *sb = sy + nq * EYA;
      for (int kq = 0; kq < nq; ++kq) {
        const uint8_t *bu = sb + kq * ng * EGB;
#pragma unroll
        for (int q = 0; q < ECB / 8 / ECW; ++q) {
          const int nt = w + q * ECW;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            if (ks >= kst) break;
            uint32_t b[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
              b[hf] = bmsk[ks][hf] ? *reinterpret_cast<const uint32_t *>(bu + boff[ks][hf] + nt * bstr[ks][hf]) &
                                         bmsk[ks][hf]
                                   : 0u;
            const uint32_t ah[4] = {ahi[ks][0], 0u, ahi[ks][1], 0u};
            mma_bf16(acc, ah, b[0], b[1]);
          }
          if (gm < len) {
            uint32_t *yp = reinterpret_cast<uint32_t *>(sy + (kq * kDecTokens + gm) * EYB + (8 * nt + gt) * 2);
            const float2 y = unpack_bf16(*yp);
            *yp = pack_bf16(y.x + sc * acc[0], y.y + sc * acc[1]);
          }
        }
      }
      // the store warp reads the updated rows through the async proxy
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ydone[s]);
      if (last) break;
    }
  } else {
    // ------------------------------------------------------------------ store warp
    // stores stage g's rows once the compute warps are done with it (the copies
    // dealt over the lanes; each lane waits for its own), and frees stage g - 1
    // when its stores have read their shared memory (one group in flight)
    int prev = -1;
    for (int g = 0; any; ++g) {
      const int s = g % NS;
      if (!wait_lane0(&ydone[s], (g / NS) & 1)) break;
      const ExpHdr *H = reinterpret_cast<const ExpHdr *>(hdr_base + s * kHdr);
      const int len = H->len, i = H->i, c0 = H->c0, nq = H->nq, last = H->last;
      const uint8_t *sy = ring + s * STAGE;
      for (int idx = lane; idx < nq * len; idx += 32) {
        const int kq = idx / len, e = idx - kq * len;
        tma_store_2d(&mp.y[i], sy + (kq * kDecTokens + e) * EYB, c0 + kq * ECB, H->rows[e]);
      }
      bulk_commit();
      bulk_wait_read1();
      __syncwarp();
      if (lane == 0 && prev >= 0) mbar_arrive(&empty[prev]);
      prev = s;
      if (last) break;
    }
    bulk_wait_read_all();
    __syncwarp();
    if (lane == 0 && prev >= 0) mbar_arrive(&empty[prev]);
    bulk_wait_all();
  }
  pdl_launch_dependents();
}

template <int KS>
lora_status_t exp_launch(const DecExpMaps &mp, const DecExpArgs &p, cudaStream_t st) {
  const size_t smem = 1024 + kRing + NS * kHdr + 256;
  LORA_CUDA(ensure_smem((const void *)expand_dec_kernel<KS>, smem));
  const int occ = occupancy((const void *)expand_dec_kernel<KS>, NTHR_E, smem);
  const int G = std::max(1, std::min(occ * num_sms(), kMaxDecGrid));
  LORA_CUDA(launch(expand_dec_kernel<KS>, dim3((unsigned)G), dim3(NTHR_E), smem, st, 1, true, mp, p));
  return LORA_OK;
}

int read_clear_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
  return v;
}

template <int RBK>
lora_status_t launch_rbk(const CUtensorMap &tmX, const CUtensorMap &tmA, const DecArgs &p, cudaStream_t st) {
  const size_t smem = 1024 + kSmem + 256;
  LORA_CUDA(ensure_smem((const void *)shrink_dec_kernel<RBK>, smem));
  const int occ = occupancy((const void *)shrink_dec_kernel<RBK>, NTHR, smem);
  const int G = std::max(1, std::min(occ * num_sms(), kMaxDecGrid));
  LORA_CUDA(launch(shrink_dec_kernel<RBK>, dim3((unsigned)G), dim3(NTHR), smem, st, 1, true, tmX, tmA, p));
  return LORA_OK;
}

}  // namespace dec

// ----------------------------------------------------------------------------- host side
size_t dec_part_bytes(int n, int R) {
  return (size_t)2 * kMaxDecGrid * kDecTokens * n * round_up(std::max(R, 1), 8) * 4;
}

lora_status_t shrink_dec_launch(const DecArgs &args, const MultiArgs &m, int64_t T, cudaStream_t st) {
  using namespace dec;
  DecArgs p = args;
  CUtensorMap tmX, tmA;
  memset(&tmX, 0, sizeof(tmX));
  memset(&tmA, 0, sizeof(tmA));
  const int64_t NR = (int64_t)m.n * m.addr.max_rank;
  p.a_one_slot = m.sa_slot == 0 ? 1 : 0;
  const int64_t aS = p.a_one_slot ? 1 : m.addr.num_slots, sslot = p.a_one_slot ? NR * m.sa_row : m.sa_slot;
  {
    // x [T][in]: one 256-column row per copy
    uint64_t dims[2] = {(uint64_t)m.in, (uint64_t)T};
    uint64_t str[1] = {(uint64_t)m.ldx * 2};
    uint32_t box[2] = {CH, 1};
    if (!encode_tmap(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, m.x, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return LORA_ERR_ALIGNMENT;
  }
  {
    // a [S][n R][in] seen as (64 columns, n R rows, in / 64 column blocks, S): a
    // copy takes 8 rows x 4 blocks of 64 columns, 128-byte swizzled
    uint64_t dims[4] = {64, (uint64_t)NR, (uint64_t)(m.in / 64), (uint64_t)aS};
    uint64_t str[3] = {(uint64_t)m.sa_row * 2, 128, (uint64_t)sslot * 2};
    uint32_t box[4] = {64, 8, 4, 1};
    if (!encode_tmap(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, m.a, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return LORA_ERR_ALIGNMENT;
  }
  const int blocks = (int)ceil_div((int64_t)m.n * round_up(m.addr.max_rank, 8), RB);
  if (blocks <= 1) return launch_rbk<1>(tmX, tmA, p, st);
  if (blocks <= 2) return launch_rbk<2>(tmX, tmA, p, st);
  if (blocks <= 4) return launch_rbk<4>(tmX, tmA, p, st);
  return LORA_ERR_UNSUPPORTED;
}

lora_status_t expand_dec_launch(const DecExpArgs &args, const MultiArgs &m, int64_t T, cudaStream_t st) {
  using namespace dec;
  DecExpArgs p = args;
  DecExpMaps mp;
  memset(&mp, 0, sizeof(mp));
  const int R = m.addr.max_rank;
  // one unit (y rows and round8(R) / 8 boxes of b) must fit a stage
  if (EYA + ceil_div(round_up(R, 8), 8) * EGB > STAGE) return LORA_ERR_UNSUPPORTED;
  p.b_one_slot = m.sb_slot == 0 ? 1 : 0;
  int off = 0, nb = 0;
  for (int i = 0; i < m.n; ++i) {
    const int64_t w = m.out_slices[i];
    p.blk0[i] = nb;
    nb += (int)ceil_div(w, ECB);
    {
      // y columns of slice i: one 256-column row segment per copy
      uint64_t dims[2] = {(uint64_t)w, (uint64_t)T};
      uint64_t str[1] = {(uint64_t)m.ldy * 2};
      uint32_t box[2] = {ECB, 1};
      if (!encode_tmap(&mp.y[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (const __nv_bfloat16 *)m.y + off, dims, str,
                       box, CU_TENSOR_MAP_SWIZZLE_NONE))
        return LORA_ERR_ALIGNMENT;
    }
    // b rows of slice i: boxes of 8, 16, 32 or 64 rank entries x 256 rows (the
    // wider ones swizzled over their 32-, 64- or 128-byte rows), no sector promotion
    const int64_t bS = p.b_one_slot ? 1 : m.addr.num_slots;
    const int64_t sslot = p.b_one_slot ? m.O * m.sb_row : m.sb_slot;
    const CUtensorMapSwizzle swz[4] = {CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                                       CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_SWIZZLE_128B};
    for (int wi = 0; wi < 4 && (8 << wi) <= round_up(R, 8); ++wi) {
      uint64_t dims[3] = {(uint64_t)R, (uint64_t)w, (uint64_t)bS};
      uint64_t str[2] = {(uint64_t)m.sb_row * 2, (uint64_t)sslot * 2};
      uint32_t box[3] = {(uint32_t)(8 << wi), ECB, 1};
      if (!encode_tmap(&mp.b[i][wi], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                       (const __nv_bfloat16 *)m.b + (int64_t)off * m.sb_row, dims, str, box, swz[wi],
                       CU_TENSOR_MAP_L2_PROMOTION_NONE))
        return LORA_ERR_ALIGNMENT;
    }
    off += (int)w;
  }
  p.blk0[m.n] = nb;
  p.nbu = nb;
  // bytes HBM serves per b row: the row itself when rows are at most 128 bytes
  // (neighbouring rows share the lines), else whole 128-byte lines; for the
  // 256 rows of a unit, in 512-byte units
  const int64_t r8b = round_up(R, 8) * 2, rowb = r8b <= 128 ? r8b : round_up(r8b, 128);
  p.bw = (int)(ECB * rowb / 512);
  if (nb == 0) return LORA_OK;
  const int ks = (int)ceil_div(round_up(R, 8), 16);
  if (ks <= 1) return exp_launch<1>(mp, p, st);
  if (ks <= 2) return exp_launch<2>(mp, p, st);
  if (ks <= 4) return exp_launch<4>(mp, p, st);
  if (ks <= 8) return exp_launch<8>(mp, p, st);
  return LORA_ERR_UNSUPPORTED;
}

int read_clear_error_decode() { return dec::read_clear_error(); }

}  // namespace lora
