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
#include <cstring>

#include "common.cuh"
#include "decode.h"
#include "host_common.h"
#include "multi.h"

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
  int nk, n, G;
  int64_t W;
  // first cost position of tile t (rows8 = its running sum of round8(rank))
  __device__ int64_t base(int t, int start, int rows8) const {
    return (int64_t)nk * ((int64_t)n * rows8 + start + (int64_t)C0 * t);
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

int read_clear_error_decode() { return dec::read_clear_error(); }

}  // namespace lora
