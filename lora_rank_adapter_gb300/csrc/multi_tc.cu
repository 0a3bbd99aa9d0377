// multi_tc.cu -- the multi-adapter shrink of decode-shaped batches (a few
// tokens per adapter slot) on the fifth-generation tensor cores of sm_103a.
//
// Operation (mstar page "mstar.engine.resources.lora.ops", shrink):
//   h[t, i*R + j] = x[t] . a[slot(t)][i*R + j]              (j < rank)
// over the slot-sorted tiles (at most 128 tokens of one slot) that the grouping
// kernel lists on the device.
//
// One persistent kernel (one CTA per SM):
//   units (tile, 64-column chunk of `in`), split evenly over the grid
//           (stream-K).  x rows arrive as one TMA box when the tile's tokens are
//           consecutive, else as four-row gather copies issued by the lanes of
//           the loader warp; the first rank16 rows of every slice of a[slot]
//           arrive as 3-D boxes.  The MMA computes the 128 x (n * rank16) block
//           into TMEM; a tile cut between CTAs leaves fp32 partial sums that the
//           last CTA of the tile adds in CTA order (deterministic).
// Rows of a past a slot's rank (which may hold anything, NaN included) only
// reach accumulator columns that are never written out.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "host_common.h"
#include "multi.h"
#include "multi_tc.h"
#include "tc_common.cuh"

namespace lora {
namespace mtc {

constexpr int TM = 128;          // tokens per tile (the MMA M)
constexpr int BOXC = 64;         // columns per chunk
constexpr int NTHR = 192;        // warp 0 loads, warp 1 MMA, warps 2..5 epilogue
constexpr int EPI0 = 2;
constexpr int kMaxNC = 256;      // n * rank16 columns of a shrink accumulator
constexpr int kSmem = 200 * 1024;
constexpr int SX = TM * BOXC * 2;                // x or y tile: 16 KB
constexpr int SA = kMaxNC * 128;                 // a rows of a shrink stage: 32 KB
constexpr int STAGE1 = SX + SA;                  // 48 KB
constexpr int NS1 = kSmem / STAGE1;              // 4

__device__ __forceinline__ int round16(int v) { return (v + 15) & ~15; }

// Warp-uniform wait, polled by lane 0.
__device__ __forceinline__ bool wait_lane0(uint64_t *bar, uint32_t parity) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity);
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

struct Tile {
  int slot, start, len, rank, r16;
  bool dense;
  int t0;
};
__device__ __forceinline__ Tile load_tile(const MtArgs &p, int tile) {
  const int4 td = p.tiles[tile];
  Tile t;
  t.slot = td.x;
  t.start = td.y;
  t.len = td.z;
  t.rank = p.ranks[t.slot];
  t.r16 = round16(t.rank);
  t.t0 = p.perm[t.start];
  t.dense = p.perm[t.start + t.len - 1] - t.t0 == t.len - 1;
  return t;
}

// ============================================================================= shrink phase
__device__ void shrink_phase(const MtArgs &p, const CUtensorMap *tmX, const CUtensorMap *tmXd,
                             const CUtensorMap *tmA16, const CUtensorMap *tmA32, const CUtensorMap *tmA64,
                             uint8_t *ring, uint64_t *bar, uint32_t tmem, int *s_flag, int ntiles, uint64_t *mdone) {
  uint64_t *full = bar, *empty = bar + NS1, *afull = bar + 2 * NS1, *aempty = afull + 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = p.nk, i = blockIdx.x;
  const int64_t U = (int64_t)ntiles * nk;
  // the units are dealt to the first min(grid, U) CTAs, so every run holds at
  // least one unit and the CTAs sharing a tile are consecutive
  const int G = (int)(U < (int64_t)gridDim.x ? (U > 0 ? U : 1) : (int64_t)gridDim.x);
  const int64_t u0 = i < G ? sk_begin(U, G, i) : 0, u1 = i < G ? sk_begin(U, G, i + 1) : 0;

  if (warp == 0) {
    // ------------------------------------------------------------------ loader warp
    int cur = -1, aslot = 0;
    Tile t{};
    int rr[4] = {0, 0, 0, 0};
    const CUtensorMap *bmap = nullptr;
    int bdst = 0, brow = 0, ngath = 0;
    uint32_t tx = 0;
    if (lane == 0) {
      prefetch_tmap(tmX);
      prefetch_tmap(tmXd);
      prefetch_tmap(tmA16);
      prefetch_tmap(tmA32);
      prefetch_tmap(tmA64);
    }
    for (int64_t u = u0; u < u1; ++u) {
      const int tile = (int)(u / nk), kc = (int)(u % nk);
      if (tile != cur) {
        cur = tile;
        t = load_tile(p, tile);
        aslot = p.a_one_slot ? 0 : t.slot;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = 4 * lane + e;
          rr[e] = r < t.len ? p.perm[t.start + r] : p.T;   // past the tile: rows read as zeros
        }
        ngath = (t.len + 3) / 4;
        // lane b issues the b-th adapter box (each slice's rank16 rows as boxes of 64, 32 and 16 rows)
        bmap = nullptr;
        int b = 0;
        for (int si = 0; si < p.n && !bmap; ++si)
          for (int j0 = 0; j0 < t.r16;) {
            const int hb = t.r16 - j0 >= 64 ? 64 : t.r16 - j0 >= 32 ? 32 : 16;
            if (b++ == lane) {
              bmap = hb == 64 ? tmA64 : hb == 32 ? tmA32 : tmA16;
              bdst = (si * t.r16 + j0) * 128;
              brow = si * p.R + j0;
              break;
            }
            j0 += hb;
          }
        tx = (uint32_t)((t.dense ? SX : ngath * 512) + p.n * t.r16 * 128);
      }
      const int g = (int)(u - u0), s = g % NS1;
      if (g >= NS1 && !wait_lane0(&empty[s], ((g / NS1) & 1) ^ 1)) break;
      uint8_t *st = ring + s * STAGE1;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], tx);
      __syncwarp();
      if (t.dense) {
        if (lane == 0) tma_load_2d(st, tmXd, &full[s], kc * BOXC, t.t0);
      } else if (lane < ngath) {
        tma_gather4(st + lane * 512, tmX, &full[s], kc * BOXC, rr[0], rr[1], rr[2], rr[3]);
      }
      if (bmap) tma_load_3d(st + SX + bdst, bmap, &full[s], kc * BOXC, brow, aslot);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int seg = 0, cur = -1, ncols = 0;
      uint32_t idesc = 0;
      bool ok = true;
      for (int64_t u = u0; ok && u < u1; ++u) {
        const int tile = (int)(u / nk), kc = (int)(u % nk);
        if (tile != cur) {
          cur = tile;
          const int rank = p.ranks[p.tiles[tile].x];
          ncols = p.n * round16(rank);
          idesc = tc_idesc(TM, ncols, false, false);
        }
        const bool first = u == u0 || kc == 0, last = u == u1 - 1 || kc == nk - 1;
        const int g = (int)(u - u0), s = g % NS1, b = seg & 1;
        if (first && seg >= 2 && !(ok = mbar_wait(&aempty[b], ((seg >> 1) & 1) ^ 1))) break;
        if (!(ok = mbar_wait(&full[s], (g / NS1) & 1))) break;
        tc_fence_after();
        const uint32_t xa = smem_u32(ring + s * STAGE1), aa = xa + SX;
#pragma unroll
        for (int kk = 0; kk < BOXC / 16; ++kk)
          tc_mma_bf16(tmem + b * kMaxNC, tc_desc(xa + kk * 32, 16, 1024, 128), tc_desc(aa + kk * 32, 16, 1024, 128),
                      idesc, (first && kk == 0) ? 0u : 1u);
        tc_commit(&empty[s]);
        if (last) {
          tc_commit(&afull[b]);
          ++seg;
        }
      }
      tc_commit(mdone);
      mbar_wait(mdone, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3, row = 32 * q + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    bool ok = true;   // after a timed-out wait: skip the work, keep the barrier sequence
    int seg = 0;
    const int64_t tb0 = u0 < u1 ? u0 / nk : 0, tb1 = u0 < u1 ? (u1 - 1) / nk : -1;
    for (int64_t tile = tb0; tile <= tb1; ++tile, ++seg) {
      const int b = seg & 1;
      const Tile t = load_tile(p, (int)tile);
      const int ncols = p.n * t.r16;
      const int first = sk_cta(U, G, tile * nk), last_cta = sk_cta(U, G, (tile + 1) * nk - 1);
      const bool whole = first == last_cta;
      float *hrow = row < t.len ? p.h + (int64_t)p.perm[t.start + row] * p.ldh : nullptr;
      // columns c (slice c / r16, j = c % r16) of this thread's row go to h when j < rank
      auto emit = [&](int c0, const float *v) {
        if (!hrow) return;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const int c = c0 + e, si = c / t.r16, j = c - si * t.r16;
          if (c >= ncols) break;
          float *hp = hrow + si * p.R + j;
          if (j + 4 <= t.rank) {
            *reinterpret_cast<float4 *>(hp) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
          } else {
            for (int k = 0; k < 4; ++k)
              if (j + k < t.rank) hp[k] = v[e + k];
          }
        }
      };
      if (ok) ok = wait_warp(&afull[b], (seg >> 1) & 1);
      if (ok) tc_fence_after();
      // partial sums column-major ([column][128 rows]): a warp's accesses of one
      // column are 32 consecutive floats
      float *mypart = p.part + part_slot(U, G, i, tile, nk) * TM * p.ncm + row;
      for (int c0 = 0; c0 < ncols; c0 += 32) {
        float v[32];
        if (ok) {
          tmem_ld32(tl + b * kMaxNC + c0, v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
        }
        if (whole) {
          emit(c0, v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c0 + e < ncols) __stcg(mypart + (int64_t)(c0 + e) * TM, v[e]);
        }
      }
      if (ok) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&aempty[b]);
      }
      if (whole) continue;
      __threadfence();
      named_bar_sync(1, 128);
      if (threadIdx.x == EPI0 * 32) *s_flag = atomicAdd(p.counters + tile, 1) == last_cta - first;
      named_bar_sync(1, 128);
      if (*s_flag) {
        __threadfence();
        // the partials of two CTAs at a time are loaded together (their loads in
        // flight at once), then added in CTA order
        for (int c0 = 0; c0 < ncols; c0 += 32) {
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
          for (int cb = first; cb <= last_cta; cb += 2) {
            float w[2][32];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const float *pp = p.part + part_slot(U, G, min(cb + k, last_cta), tile, nk) * TM * p.ncm + row;
#pragma unroll
              for (int e = 0; e < 32; ++e)
                w[k][e] = cb + k <= last_cta && c0 + e < ncols ? __ldcg(pp + (int64_t)(c0 + e) * TM) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] += w[k][e];
          }
          emit(c0, v);
        }
        if (threadIdx.x == EPI0 * 32) p.counters[tile] = 0;   // ready for the next call
      }
      named_bar_sync(1, 128);
    }
  }
}

// ============================================================================= the kernel
__global__ void __launch_bounds__(NTHR, 1)
    shrink_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXd,
                     const __grid_constant__ CUtensorMap tmA16, const __grid_constant__ CUtensorMap tmA32,
                     const __grid_constant__ CUtensorMap tmA64, MtArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kSmem);   // full, empty [NS1], afull, aempty [2]
  uint64_t *mdone = bar + 2 * NS1 + 4;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mdone + 1);
  int *s_flag = reinterpret_cast<int *>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS1; ++s) {
      mbar_init(&bar[s], 1);
      mbar_init(&bar[NS1 + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar[2 * NS1 + b], 1);
      mbar_init(&bar[2 * NS1 + 2 + b], 4);
    }
    mbar_init(mdone, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  shrink_phase(p, &tmX, &tmXd, &tmA16, &tmA32, &tmA64, smem, bar, tmem, s_flag, p.header[1], mdone);
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int read_clear_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
  return v;
}

}  // namespace mtc

// ----------------------------------------------------------------------------- host side
namespace {

using namespace mtc;

bool map2(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows) {
  uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  uint64_t str[1] = {(uint64_t)ld * 2};
  uint32_t box[2] = {64, box_rows};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// a [S][rows][cols]: boxes of 64 columns x box_rows rows (128-byte swizzle)
bool map_a3(CUtensorMap *m, const void *base, int64_t S, int64_t rows, int64_t cols, int64_t s_slot, int64_t s_row,
            uint32_t box_rows) {
  uint64_t dims[3] = {(uint64_t)cols, (uint64_t)rows, (uint64_t)S};
  uint64_t str[2] = {(uint64_t)s_row * 2, (uint64_t)s_slot * 2};
  uint32_t box[3] = {64, box_rows, 1};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
}  // namespace

size_t multi_tc_part_bytes(int n, int R) {
  const int ncm = n * std::max(16, (int)round_up(R, 16));
  return (size_t)2 * kMaxTcGrid * TM * ncm * 4;
}

lora_status_t shrink_tc_launch(const MtArgs &args, const MultiArgs &m, int64_t T, cudaStream_t st) {
  MtArgs p = args;
  CUtensorMap maps[5];
  memset(maps, 0, sizeof(maps));
  const int64_t NR = (int64_t)m.n * m.addr.max_rank;
  p.a_one_slot = m.sa_slot == 0 ? 1 : 0;
  const int64_t aS = p.a_one_slot ? 1 : m.addr.num_slots, sslot = p.a_one_slot ? NR * m.sa_row : m.sa_slot;
  if (!map2(&maps[0], m.x, T, m.in, m.ldx, 1) || !map2(&maps[1], m.x, T, m.in, m.ldx, TM) ||
      !map_a3(&maps[2], m.a, aS, NR, m.in, sslot, m.sa_row, 16) ||
      !map_a3(&maps[3], m.a, aS, NR, m.in, sslot, m.sa_row, 32) ||
      !map_a3(&maps[4], m.a, aS, NR, m.in, sslot, m.sa_row, 64))
    return LORA_ERR_ALIGNMENT;
  const size_t smem = 1024 + kSmem + 1024;
  LORA_CUDA(ensure_smem((const void *)shrink_tc_kernel, smem));
  const int occ = occupancy((const void *)shrink_tc_kernel, NTHR, smem);
  const int G = std::max(1, std::min(occ * num_sms(), kMaxTcGrid));
  LORA_CUDA(launch(shrink_tc_kernel, dim3((unsigned)G), dim3(NTHR), smem, st, 1, true, maps[0], maps[1], maps[2],
                   maps[3], maps[4], p));
  return LORA_OK;
}

int read_clear_error_multi_tc() { return mtc::read_clear_error(); }

}  // namespace lora
