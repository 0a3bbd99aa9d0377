// single_tc.cu -- single-adapter LoRA kernels (bf16 storage, fp32 accumulation)
// on the fifth-generation tensor cores of sm_103a: tcgen05.mma with the
// accumulators in tensor memory (TMEM), operands staged in shared memory by the
// tensor-memory accelerator (TMA).
//
// Operations ([NeMo lora_kernel] = NeMo AutoModel API page
// "nemo_automodel.components._peft.lora_kernel"), in forward roles X [M,K],
// A [K,r], B [r,L]:
//   forward   Y += s * (X*A)*B       lora_forward_kernel (inner_kernel, block_vector_mul)
//   dyb       dY * B^T                lora_da_dx_kernel (DYB = DY x B)
//   dX, dA    s * dyb*A^T, s * X^T*dyb   lora_da_dx_kernel / lora_da_dx_update_wrapper
//   h, dB     X*A, s * h^T*dY           lora_db_kernel / lora_db_update_wrapper
//
// Three kernels do all of it:
//   rows_kernel    out[m, :] = In[m, :] * W over a contraction of C columns, for
//                  128-row blocks (h = X*A with W = A, dyb = dY*B^T with W = B^T).
//                  The (row block, 128-column chunk) units are split evenly over a
//                  persistent grid (stream-K); a row block cut between CTAs leaves
//                  fp32 partial sums in the workspace and the last CTA to finish
//                  adds them in CTA order (deterministic).  The result goes out as
//                  a "blob": the bf16 hi and lo parts (v ~= hi + lo to ~2^-17) of
//                  the 128 x RP block, already in the swizzled layout the tensor
//                  cores read, and optionally as fp32 rows (the saved h).
//   expand_kernel  Y[m, l] += s * sum_j h[m, j] B[j, l] over (row block, 128-column
//                  chunk of Y) units: h hi/lo from the blob, B^T chunks and Y tiles
//                  by TMA, the product in TMEM, Y read-modify-written once.
//   col_kernel     acc[c, :] = sum over rows m of In[m, c] * blob[m, :] for
//                  128-column blocks of In (dA = X^T*dyb, dB^T = dY^T*h), stream-K
//                  over (column block, 128-row tile) units with the same ordered
//                  reduction; with kDX it also writes, per row tile, the dX tile
//                  s * dyb*A^T (dX is read-modified-written when accumulating).
// Warp roles in every kernel: warp 0 loads (one lane issues TMA), warp 1 issues
// the MMAs (one lane) and owns the TMEM allocation, warps 2..5 drain TMEM (one
// accumulator row per thread; warp w reads TMEM lanes 32 (w % 4) ..).
//
// Operand layouts: every staged tile is rows of 32/64/128 bytes with the
// matching TMA swizzle.  A tile is read K-major (rows = M or N, K along the row)
// or MN-major (rows = K, M or N along the row); the second form lets the
// transposed products (X^T, dY^T, B^T in PEFT layout) use the tiles as TMA
// wrote them.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "host_common.h"
#include "single_common.h"
#include "single_tc.h"
#include "tc_common.cuh"

namespace lora {
namespace tc {

constexpr int TM = 128;        // rows of a tile (the MMA M)
constexpr int BOXC = 64;       // columns of one TMA box (128 bytes of bf16)
constexpr int NTHR = 192;      // six warps
constexpr int EPI0 = 2;        // first epilogue warp
constexpr int kRingBytes = 196 * 1024;

__host__ __device__ constexpr int pw_of(int RP) { return RP < 64 ? RP : 64; }
// bytes of one (hi or lo) 128 x RP bf16 tile of a blob
__host__ __device__ constexpr int blob_tile(int RP) { return TM * RP * 2; }
__host__ __device__ constexpr int tmem_cols(int need) {
  return need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;
}

// Byte offset of (row, col) in a blob tile: panels of PW columns, each [128][PW]
// with a (2 PW)-byte swizzle.
template <int RP>
__device__ __forceinline__ uint32_t blob_off(int row, int col) {
  constexpr int PW = pw_of(RP);
  return (uint32_t)((col / PW) * (TM * PW * 2)) + swz((uint32_t)row, (uint32_t)(col % PW) * 2, PW * 2);
}

// Partial sums are stored column-major ([RP columns][128 rows]): a warp's
// accesses of one column are 32 consecutive floats.  They are stored with an
// L2 evict-last policy (a few MB in all): the CTA that finishes the block reads
// them back, usually at the end of the pass, after the HBM stream has gone by.
template <int RP>
__device__ __forceinline__ void store_partial(float *part, int row, const float *v) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
#pragma unroll
  for (int j = 0; j < RP; ++j)
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(part + j * TM + row), "f"(v[j]), "l"(pol)
                 : "memory");
}
// RP accumulator columns of this thread's TMEM lane.
template <int RP>
__device__ __forceinline__ void tmem_row(uint32_t taddr, float *v) {
  if constexpr (RP == 16) {
    float t[16];
    tmem_ld16(taddr, t);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = t[j];
  } else {
#pragma unroll
    for (int c = 0; c < RP; c += 32) tmem_ld32(taddr + c, v + c);
  }
}

// The epilogue's end of the segment of group g (units [g n, (g + 1) n)) that CTA
// i computed: either the group is all this CTA's (no partial), or the partial
// goes to the workspace and the last CTA of the group to finish adds the
// partials of all its CTAs in CTA order, starting from 0.  Returns true when
// this CTA then holds the group's full sum in v.  Called by the four epilogue
// warps together (`leader` is the first thread of the four).
//
// The group's first CTA reaches the group with the last units of its range, the
// others with their first units, so the first CTA usually finishes it last.  It
// therefore takes its ticket before storing anything: it adds kFirstTicket; if
// every other CTA has already stored (the count it sees is theirs), it is the
// last one, and its own partial, the first term of the sum, never leaves v.
// Otherwise it stores like the others, which add 1 after storing, and the CTA
// whose addition completes kFirstTicket + (number of CTAs) is the last one: by
// then every partial is stored, and it reloads them all, its own included (the
// stored copy holds the same values, so the result does not depend on which
// CTA finishes last).  No CTA waits for another either way.
constexpr int kFirstTicket = 1 << 16;
template <int RP>
__device__ __forceinline__ bool reduce_segment(int64_t U, int G, int i, int64_t g, int64_t n, float *part,
                                               int *counter, int row, float *v, int *s_flag,
                                               int leader = EPI0 * 32) {
  const int first = sk_cta(U, G, g * n), last_cta = sk_cta(U, G, (g + 1) * n - 1);
  if (first == last_cta) return true;
  const int others = last_cta - first;
  bool last;
  if (i == first) {
    if (threadIdx.x == leader) *s_flag = atomicAdd(counter, kFirstTicket) == others;
    named_bar_sync(1, 128);
    last = *s_flag != 0;
    named_bar_sync(1, 128);
    if (last) {
      __threadfence();
#pragma unroll
      for (int j = 0; j < RP; ++j) v[j] = 0.f + v[j];   // as summed from 0 (the sign of a zero included)
      for (int c = first + 1; c <= last_cta; ++c) {
        const float *pc = part + part_slot(U, G, c, g, n) * TM * RP + row;
#pragma unroll
        for (int j = 0; j < RP; ++j) v[j] += __ldcg(pc + j * TM);
      }
      if (threadIdx.x == leader) *counter = 0;
      return true;
    }
  }
  store_partial<RP>(part + part_slot(U, G, i, g, n) * TM * RP, row, v);
  __threadfence();
  named_bar_sync(1, 128);
  if (threadIdx.x == leader) *s_flag = atomicAdd(counter, 1) == kFirstTicket + others;
  named_bar_sync(1, 128);
  last = *s_flag != 0;
  if (last) {
    __threadfence();
#pragma unroll
    for (int j = 0; j < RP; ++j) v[j] = 0.f;
    for (int c = first; c <= last_cta; ++c) {
      const float *pc = part + part_slot(U, G, c, g, n) * TM * RP + row;
#pragma unroll
      for (int j = 0; j < RP; ++j) v[j] += __ldcg(pc + j * TM);
    }
    if (threadIdx.x == leader) *counter = 0;
  }
  named_bar_sync(1, 128);
  return last;
}

// Row `row` of 128-row block `blk` of a saved fp32 h (columns j < r; zero past r
// and past M) into that block's hi / lo blob tiles.
template <int RP>
__device__ __forceinline__ void hrow_to_blob(const float *__restrict__ h, int64_t ldh, int64_t M, int r, int64_t blk,
                                             int row, uint8_t *blob) {
  uint8_t *bhi = blob + blk * (int64_t)(2 * blob_tile(RP)), *blo = bhi + blob_tile(RP);
  const int64_t m = blk * TM + row;
#pragma unroll
  for (int col = 0; col < RP; col += 8) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = m < M && col + k < r ? h[m * ldh + col + k] : 0.f;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) split_bf16(v[2 * k], v[2 * k + 1], hi[k], lo[k]);
    const uint32_t o = blob_off<RP>(row, col);
    *reinterpret_cast<uint4 *>(bhi + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4 *>(blo + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// ============================================================================= rows
// A rows unit covers RUC columns of the contraction: two 64-column In boxes and
// the two matching W chunks (fewer, larger units stream In faster: a column
// pass with 32 KB units reads at 5.3 TB/s, a rows pass with 16 KB units 4.7)
constexpr int RUC = 2 * BOXC;

template <int RP, bool kWMN>
struct RowsCfg {
  static constexpr int PW = pw_of(RP);
  static constexpr int IN_B = TM * RUC * 2;     // 32 KB: two [128][64] boxes
  static constexpr int W_B = 2 * RP * 128;      // two Ac [RP][64] or two B^T [64][RP] chunks
  static constexpr int STAGE = IN_B + W_B;
  static constexpr int NS = kRingBytes / STAGE > 8 ? 8 : kRingBytes / STAGE;
  static constexpr int TMEM = tmem_cols(2 * RP);
  static constexpr int BYTES = 1024 + NS * STAGE + 1024;
};

template <int RP, bool kWMN>
__global__ void __launch_bounds__(NTHR, 1) rows_kernel(const __grid_constant__ CUtensorMap tmIn,
                                                       const __grid_constant__ CUtensorMap tmW, TcRowsArgs p) {
  using C = RowsCfg<RP, kWMN>;
  constexpr int NS = C::NS, PW = C::PW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(ring + NS * C::STAGE);
  uint64_t *empty = full + NS;
  uint64_t *afull = empty + NS;    // [2] accumulator written
  uint64_t *aempty = afull + 2;    // [2] accumulator drained
  uint64_t *mdone = aempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mdone + 1);
  int *s_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x;
  const int64_t u0 = sk_begin(p.U, p.G, i), u1 = sk_begin(p.U, p.G, i + 1);
  const int nc = p.nc;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], 4);
    }
    mbar_init(mdone, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------------------ loader
    if (lane == 0) {
      prefetch_tmap(&tmIn);
      prefetch_tmap(&tmW);
      for (int64_t u = u0; u < u1; ++u) {
        const int g = (int)(u - u0), s = g % NS;
        if (g >= NS && !mbar_wait(&empty[s], ((g / NS) & 1) ^ 1)) break;
        const int rb = (int)(u / nc), c = (int)(u % nc);
        uint8_t *st = ring + s * C::STAGE;
        mbar_arrive_expect_tx(&full[s], C::STAGE);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int c0 = c * RUC + hf * BOXC;
          tma_load_2d(st + hf * (TM * BOXC * 2), &tmIn, &full[s], c0, rb * TM);
          uint8_t *w = st + C::IN_B + hf * (RP * 128);
          if (kWMN) {
#pragma unroll
            for (int pp = 0; pp < RP / PW; ++pp) tma_load_2d(w + pp * (BOXC * PW * 2), &tmW, &full[s], pp * PW, c0);
          } else {
            tma_load_2d(w, &tmW, &full[s], c0, 0);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc_idesc(TM, RP, false, kWMN);
      int seg = 0;
      bool ok = true;
      for (int64_t u = u0; ok && u < u1; ++u) {
        const int g = (int)(u - u0), s = g % NS;
        const int c = (int)(u % nc);
        const bool first = u == u0 || c == 0, last = u == u1 - 1 || c == nc - 1;
        const int b = seg & 1;
        if (first && seg >= 2 && !(ok = mbar_wait(&aempty[b], ((seg >> 1) & 1) ^ 1))) break;
        if (!(ok = mbar_wait(&full[s], (g / NS) & 1))) break;
        tc_fence_after();
        const uint32_t st0 = smem_u32(ring + s * C::STAGE);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t st = st0 + hf * (TM * BOXC * 2), w = st0 + C::IN_B + hf * (RP * 128);
#pragma unroll
          for (int kk = 0; kk < BOXC / 16; ++kk) {
            const uint64_t ad = tc_desc(st + kk * 32, 16, 1024, 128);
            const uint64_t bd = kWMN ? tc_desc(w + kk * 16 * PW * 2, RP > PW ? BOXC * PW * 2 : 16, 8 * PW * 2, PW * 2)
                                     : tc_desc(w + kk * 32, 16, 1024, 128);
            tc_mma_bf16(tmem + b * RP, ad, bd, idesc, (first && hf == 0 && kk == 0) ? 0u : 1u);
          }
        }
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
    float v[RP];
    int seg = 0;
    bool ok = true;   // after a timed-out wait: skip the work, keep the barrier sequence
    const int64_t rb0 = u0 < u1 ? u0 / nc : 0, rb1 = u0 < u1 ? (u1 - 1) / nc : -1;
    if (p.hin != nullptr) {
      // the saved h as a blob for a later pass: the epilogue is idle until its
      // first block's accumulator is complete
      const int64_t nrb = ((int64_t)p.M + TM - 1) / TM;
      for (int64_t blk = i; blk < nrb; blk += gridDim.x) hrow_to_blob<RP>(p.hin, p.ldhin, p.M, p.r, blk, row, p.hblob);
    }
    for (int64_t rb = rb0; rb <= rb1; ++rb, ++seg) {
      const int b = seg & 1;
      if (ok) ok = wait_warp(&afull[b], (seg >> 1) & 1);
#pragma unroll
      for (int j = 0; j < RP; ++j) v[j] = 0.f;
      if (ok) {
        tc_fence_after();
        tmem_row<RP>(tl + b * RP, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&aempty[b]);
      }
      if (!reduce_segment<RP>(p.U, p.G, i, rb, nc, p.part, p.counters + rb, row, v, s_flag)) continue;
      // the block's full sum: the hi / lo blob, and the fp32 rows when asked for
      uint8_t *bhi = p.blob + rb * (int64_t)(2 * blob_tile(RP)), *blo = bhi + blob_tile(RP);
#pragma unroll
      for (int j = 0; j < RP; j += 8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_bf16(v[j + 2 * e], v[j + 2 * e + 1], hi[e], lo[e]);
        const uint32_t o = blob_off<RP>(row, j);
        *reinterpret_cast<uint4 *>(bhi + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(blo + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      const int64_t grow = rb * TM + row;
      if (p.hout != nullptr && grow < p.M) {
        float *hr = p.hout + grow * p.ldh;
        if (p.h_vec4) {
          // 16-byte stores: a quarter of the store instructions (each lane writes its own row)
#pragma unroll
          for (int j = 0; j < RP; j += 4)
            if (j < p.r) *reinterpret_cast<float4 *>(hr + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < RP; ++j)
            if (j < p.r) hr[j] = v[j];
        }
      }
    }
  }
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM);
  }
}

// ============================================================================= expand
// Y[m, l] += s * (h_hi + h_lo)[m, :] . B^T[l, :]; four TMEM accumulators of 64
// columns let the epilogue of one chunk overlap the MMAs of the next.
// An expand unit covers EUC columns of Y: two 64-column Y boxes, a 128-row B^T
// chunk, one N = 128 MMA per K step (fewer, larger units, as in the rows pass).
constexpr int EUC = 2 * BOXC;

template <int RP>
struct ExpCfg {
  static constexpr int PW = pw_of(RP);
  static constexpr int Y_B = TM * EUC * 2;       // 32 KB: two [128][64] boxes
  static constexpr int B_B = EUC * RP * 2;       // B^T chunk: RP / PW panels of [128 l][PW]
  static constexpr int HB = 2 * blob_tile(RP);   // hi + lo of one row block
  // blob buffers: a row block covers L / 128 units, so at r = 64 one buffer
  // (a short stall when the row block changes) buys the ring more Y stages
  static constexpr int NB = RP >= 64 ? 1 : 2;
  // Y tiles and B^T chunks have rings of their own: a Y stage is held until its
  // tile has been stored, a B^T stage only until the MMAs have read it, and the
  // MMAs never wait for a Y tile.  The loader issues both in unit order, so it
  // runs at most NBB + ND units ahead of the epilogue (not fewer than NS here).
  static constexpr int ND = 4;                   // accumulators of 128 TMEM columns
  static constexpr int NBB = 2;
  static constexpr int NS0 = (kRingBytes + 28 * 1024 - NB * HB - NBB * B_B) / Y_B;
  static constexpr int NS = NS0 > 12 ? 12 : NS0;
  static_assert(NS <= NBB + ND, "the loader must be able to fill the Y ring");
  static constexpr int TMEM = 512;
  static constexpr int BYTES = 1024 + NB * HB + NS * Y_B + NBB * B_B + 1024;
  static_assert(BYTES <= 227 * 1024, "expand shared memory");
};

template <int RP>
__global__ void __launch_bounds__(NTHR, 1) expand_kernel(const __grid_constant__ CUtensorMap tmY,
                                                         const __grid_constant__ CUtensorMap tmYs,
                                                         const __grid_constant__ CUtensorMap tmB, TcExpArgs p) {
  using C = ExpCfg<RP>;
  constexpr int NS = C::NS, PW = C::PW, ND = C::ND, NB = C::NB, NBB = C::NBB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *hbuf = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = hbuf + NB * C::HB;     // Y tiles
  uint8_t *bring = ring + NS * C::Y_B;   // B^T chunks
  uint64_t *full = reinterpret_cast<uint64_t *>(bring + NBB * C::B_B);
  uint64_t *empty = full + NS;
  uint64_t *bfull = empty + NS;    // [NBB]
  uint64_t *bempty = bfull + NBB;
  uint64_t *hfull = bempty + NBB;  // [2]
  uint64_t *hempty = hfull + 2;    // [2]
  uint64_t *dfull = hempty + 2;    // [ND]
  uint64_t *dempty = dfull + ND;   // [ND]
  uint64_t *mdone = dempty + ND;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mdone + 1);
  // the unit of the g-th stage of this CTA's sequence, written by the loader
  // before it arrives on the stage's barriers (the MMA warp reads it after its
  // B^T wait, the epilogue after its Y wait); -1 ends the sequence
  int64_t *s_u = reinterpret_cast<int64_t *>(tmem_slot + 2);
  constexpr int kQ = 16;   // more than the loader can run ahead of the epilogue

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the first Us units are dealt evenly (stream-K), the rest CH at a time to
  // whichever CTA asks first: SMs stream at rates some percent apart, and the
  // shared tail lets the fast ones take more
  const int64_t u0 = sk_begin(p.Us, p.G, blockIdx.x), u1 = sk_begin(p.Us, p.G, blockIdx.x + 1);
  const int nl = p.nl;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    for (int s = 0; s < NBB; ++s) {
      mbar_init(&bfull[s], 1);
      mbar_init(&bempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&hfull[b], 1);
      mbar_init(&hempty[b], 1);
    }
    for (int b = 0; b < ND; ++b) {
      mbar_init(&dfull[b], 1);
      mbar_init(&dempty[b], 4);
    }
    mbar_init(mdone, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmY);
      prefetch_tmap(&tmB);
      int64_t prev = -1;
      int hidx = 0, g = 0;
      // unit u into the stages of sequence number g; false after a timed-out wait
      auto issue = [&](int64_t u) -> bool {
        const int64_t rb = u / nl;
        const int lc = (int)(u % nl);
        const int s = g % NS, sb = g % NBB;
        if (g >= NS && !mbar_wait(&empty[s], ((g / NS) & 1) ^ 1)) return false;
        s_u[g % kQ] = u;
        mbar_arrive_expect_tx(&full[s], C::Y_B);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_load_2d(ring + s * C::Y_B + hf * (TM * BOXC * 2), &tmY, &full[s], lc * EUC + hf * BOXC, (int)(rb * TM));
        if (g >= NBB && !mbar_wait(&bempty[sb], ((g / NBB) & 1) ^ 1)) return false;
        uint8_t *bt = bring + sb * C::B_B;
        mbar_arrive_expect_tx(&bfull[sb], C::B_B);
#pragma unroll
        for (int pp = 0; pp < RP / PW; ++pp)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_2d(bt + pp * (EUC * PW * 2) + hf * (BOXC * PW * 2), &tmB, &bfull[sb], pp * PW,
                        lc * EUC + hf * BOXC);
        // the row block's blob after the unit's stage (which does not need it), so
        // that a buffer still read by the previous block's MMAs delays no Y copy
        if (rb != prev) {
          const int hb = hidx % NB;
          if (hidx >= NB && !mbar_wait(&hempty[hb], ((hidx / NB) & 1) ^ 1)) return false;
          mbar_arrive_expect_tx(&hfull[hb], C::HB);
          bulk_load(hbuf + hb * C::HB, p.blob + rb * (int64_t)C::HB, C::HB, &hfull[hb]);
          prev = rb;
          ++hidx;
        }
        ++g;
        return true;
      };
      bool ok = true;
      for (int64_t u = u0; ok && u < u1; ++u) ok = issue(u);
      while (ok && p.next != nullptr) {
        const int64_t a0 = p.Us + (int64_t)atomicAdd(p.next, 1) * p.CH;
        if (a0 >= p.U) break;
        const int64_t a1 = a0 + p.CH < p.U ? a0 + p.CH : p.U;
        for (int64_t u = a0; ok && u < a1; ++u) ok = issue(u);
      }
      if (ok) {
        // the end of the sequence, through the barriers the MMA warp and the
        // epilogue wait on next
        const int s = g % NS, sb = g % NBB;
        if (g < NS || mbar_wait(&empty[s], ((g / NS) & 1) ^ 1)) {
          s_u[g % kQ] = -1;
          mbar_arrive(&full[s]);
          if (g < NBB || mbar_wait(&bempty[sb], ((g / NBB) & 1) ^ 1)) mbar_arrive(&bfull[sb]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc_idesc(TM, EUC, false, false);
      int64_t prev = -1;
      int hidx = 0, hb = 0, g = 0;
      bool ok = mbar_wait(&bfull[0], 0);
      int64_t u = ok ? s_u[0] : -1;
      while (ok && u >= 0) {
        const int64_t rb = u / nl;
        if (rb != prev) {
          hb = hidx % NB;
          if (!(ok = mbar_wait(&hfull[hb], (hidx / NB) & 1))) break;
          prev = rb;
          ++hidx;
        }
        const int sb = g % NBB, b = g % ND;
        if (g >= ND && !(ok = mbar_wait(&dempty[b], ((g / ND) & 1) ^ 1))) break;
        tc_fence_after();
        const uint32_t hh = smem_u32(hbuf + hb * C::HB), bb = smem_u32(bring + sb * C::B_B);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int qk = 0; qk < RP / 16; ++qk) {
            const int pan = (qk * 16) / PW, in = ((qk * 16) % PW) * 2;
            const uint64_t ad = tc_desc(hh + part * blob_tile(RP) + pan * (TM * PW * 2) + in, 16, 8 * PW * 2, PW * 2);
            const uint64_t bd = tc_desc(bb + pan * (EUC * PW * 2) + in, 16, 8 * PW * 2, PW * 2);
            tc_mma_bf16(tmem + b * EUC, ad, bd, idesc, (part == 0 && qk == 0) ? 0u : 1u);
          }
        tc_commit(&dfull[b]);
        tc_commit(&bempty[sb]);
        ++g;
        // the next unit (or the end) tells whether this row block's blob is still read
        if (!(ok = mbar_wait(&bfull[g % NBB], (g / NBB) & 1))) break;
        const int64_t un = s_u[g % kQ];
        if (un < 0 || un / nl != rb) tc_commit(&hempty[hb]);
        u = un;
      }
      if (ok) {
        // the end of the sequence for the epilogue
        const int b = g % ND;
        if (g < ND || mbar_wait(&dempty[b], ((g / ND) & 1) ^ 1)) mbar_arrive(&dfull[b]);
      }
      tc_commit(mdone);
      mbar_wait(mdone, 0);
    }
    __syncwarp();
  } else {
    // Each warp owns the 32 rows of its TMEM lane quarter: it adds s * acc into
    // them in the staged Y tile and writes them back with one TMA store (rows
    // past M and columns past L are clipped by the store).  A stage is released
    // to the loader once the store of the next unit has been issued and this
    // store has finished reading the stage.
    const int q = warp & 3, row = 32 * q + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    const float scale = p.scale;
    int pend = -1;   // stage whose store may still be reading it
    if (lane == 0) prefetch_tmap(&tmYs);
    for (int g = 0;; ++g) {
      const int s = g % NS, b = g % ND;
      if (!wait_warp(&dfull[b], (g / ND) & 1) || !wait_warp(&full[s], (g / NS) & 1)) break;
      const int64_t u = s_u[g % kQ];
      if (u < 0) break;
      tc_fence_after();
      uint8_t *ys = ring + s * C::Y_B;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float acc[64];
        tmem_ld32(tl + b * EUC + hf * BOXC, acc);
        tmem_ld32(tl + b * EUC + hf * BOXC + 32, acc + 32);
        uint8_t *yt = ys + hf * (TM * BOXC * 2);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 *yp = reinterpret_cast<uint4 *>(yt + swz(row, c * 16, 128));
          const uint4 yv = *yp;
          const uint32_t w[4] = {yv.x, yv.y, yv.z, yv.w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 y = unpack_bf16(w[e]);
            o[e] = pack_bf16(y.x + scale * acc[8 * c + 2 * e], y.y + scale * acc[8 * c + 2 * e + 1]);
          }
          *yp = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();   // the TMA stores read what this warp wrote
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&dempty[b]);
        const int64_t rb = u / nl;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_store_2d(&tmYs, ys + hf * (TM * BOXC * 2) + q * 32 * 128, (int)(u % nl) * EUC + hf * BOXC,
                       (int)(rb * TM) + 32 * q);
        bulk_commit();
        if (pend >= 0) {
          bulk_wait_read1();
          mbar_arrive(&empty[pend]);
        }
        pend = s;
      }
    }
    if (lane == 0) {
      bulk_wait_read_all();
      if (pend >= 0) mbar_arrive(&empty[pend]);
      bulk_wait_all();
    }
  }
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM);
  }
}

// ============================================================================= column pass
template <int RP, bool kDX>
struct ColCfg {
  static constexpr int PW = pw_of(RP);
  static constexpr int IN_B = 2 * TM * BOXC * 2;   // two 64-column boxes: 32 KB
  static constexpr int BL_B = 2 * blob_tile(RP);   // hi + lo
  // A^T of one column block for dX: two [RP][64] boxes.  At RP <= 64 two such
  // buffers, so that the next column block's A^T loads while the MMAs still read
  // the current one and the In stream goes on (the ring keeps its stages); at
  // RP = 128 one (a second would cost an In stage): there the loader waits at a
  // column block's start for the MMAs of the one before.
  static constexpr int AC1 = 2 * RP * 128;
  static constexpr int NAC = kDX ? (RP <= 64 ? 2 : 1) : 0;
  static constexpr int AC_B = NAC * AC1;
  static constexpr int SPACE = kRingBytes + 28 * 1024 - AC_B;
  // In tiles and blobs have rings of their own.  With dX an In stage is held
  // until the dX tile written over it has been stored, a blob stage only until
  // the MMAs have read it: two blob stages, the rest of the space In stages.
  // Without dX both are released by the MMAs: as many blob stages as In stages.
  static constexpr int NX0 = kDX ? (SPACE - 2 * BL_B) / IN_B : SPACE / (IN_B + BL_B);
  static constexpr int NX = NX0 > 6 ? 6 : NX0;
  static constexpr int NBL = kDX ? 2 : NX;
  // The blob's hi and lo tiles lie one after the other, as two column panels of
  // one [128][2 RP] operand: at RP <= 64 one MMA of N = 2 RP takes both (half
  // the MMA issues; the accumulator's two halves are added when read out)
  static constexpr bool HL = RP <= 64;
  static constexpr int AW = HL ? 2 * RP : RP;      // TMEM columns of one accumulator
  static constexpr int TMEM = tmem_cols(2 * AW + (kDX ? 2 * TM : 0));
  static constexpr int ACC0 = kDX ? 2 * TM : 0;   // first TMEM column of the accumulators
  static constexpr int BYTES = 1024 + NX * IN_B + NBL * BL_B + AC_B + 1024;
  static_assert(BYTES <= 227 * 1024, "column pass shared memory");
  // With dX at RP <= 64 the accumulators have four epilogue warps of their own
  // (warps 6-9, the same TMEM lane quarters as warps 2-5): the read-out, the
  // partial-sum stores and the fences of a column block's end then never hold
  // the dX tiles, which warps 2-5 drain.  (A fence waits behind the SM's loads
  // in flight: microseconds in the middle of the stream.)  At RP = 128 the
  // accumulator row takes the registers that ten warps would not leave.
  static constexpr bool SPLIT = kDX && RP <= 64;
  static constexpr int NT = SPLIT ? 320 : NTHR;
  static_assert(2 * AW + (kDX ? 2 * TM : 0) <= 512, "column pass tensor memory");
};

template <int RP, bool kDX, bool kAccX>
__global__ void __launch_bounds__(ColCfg<RP, kDX>::NT, 1) col_kernel(const __grid_constant__ CUtensorMap tmIn,
                                                      const __grid_constant__ CUtensorMap tmAc,
                                                      const __grid_constant__ CUtensorMap tmDX, TcColArgs p) {
  using C = ColCfg<RP, kDX>;
  constexpr int NS = C::NX, NBL = C::NBL, PW = C::PW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *bring = ring + NS * C::IN_B;   // blob stages
  uint8_t *acbuf = bring + NBL * C::BL_B;
  uint64_t *full = reinterpret_cast<uint64_t *>(acbuf + C::AC_B);
  uint64_t *empty = full + NS;
  uint64_t *bfull = empty + NS;    // [NBL] blob stages
  uint64_t *bempty = bfull + NBL;
  uint64_t *afull = bempty + NBL;  // [2] accumulators
  uint64_t *aempty = afull + 2;
  uint64_t *dfull = aempty + 2;    // [2] dX tiles
  uint64_t *dempty = dfull + 2;
  uint64_t *acfull = dempty + 2;   // [2] A^T buffer loaded
  uint64_t *acempty = acfull + 2;  // [2] A^T buffer no longer read
  uint64_t *mdone = acempty + 2;
  uint64_t *xfree = mdone + 1;     // [NS] the MMAs no longer read the stage's In tile
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(xfree + NS);
  int *s_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x;
  const int64_t u0 = sk_begin(p.U, p.G, i), u1 = sk_begin(p.U, p.G, i + 1);
  const int nt = p.nt;
  if (threadIdx.x == 0) {
    // with dX, a stage is released by the four epilogue warps once the dX tile
    // they wrote over its In tile has been stored; else by the MMAs' completion
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDX ? 4 : 1);
      mbar_init(&xfree[s], 1);
    }
    for (int s = 0; s < NBL; ++s) {
      mbar_init(&bfull[s], 1);
      mbar_init(&bempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], 4);
      mbar_init(&dfull[b], 1);
      mbar_init(&dempty[b], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acfull[b], 1);
      mbar_init(&acempty[b], 1);
    }
    mbar_init(mdone, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The dB pass of lora_backward needs nothing from the dX pass before it (its
  // dY and h blob were complete before that pass got past its own wait): it
  // starts while the dX pass's last CTAs finish and waits for that pass only
  // before exiting, so that it still completes after it.
  if (p.wait_first) pdl_wait();
  if (kDX) pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmIn);
      if (kDX) {
        prefetch_tmap(&tmAc);
        prefetch_tmap(&tmDX);
      }
      int seg = 0;
      for (int64_t u = u0; u < u1; ++u) {
        const int cb = (int)(u / nt), t = (int)(u % nt);
        if (kDX && (u == u0 || t == 0)) {
          // column block `seg` of the range uses A^T buffer seg % NAC
          const int ab = C::NAC == 2 ? (seg & 1) : 0, use = C::NAC == 2 ? seg >> 1 : seg;
          if (use >= 1 && !mbar_wait(&acempty[ab], (use - 1) & 1)) break;
          uint8_t *ac = acbuf + ab * C::AC1;
          mbar_arrive_expect_tx(&acfull[ab], C::AC1);
          tma_load_2d(ac, &tmAc, &acfull[ab], cb * 2 * BOXC, 0);
          tma_load_2d(ac + RP * 128, &tmAc, &acfull[ab], cb * 2 * BOXC + BOXC, 0);
          ++seg;
        }
        const int g = (int)(u - u0), s = g % NS, sb = g % NBL;
        if (g >= NS && !mbar_wait(&empty[s], ((g / NS) & 1) ^ 1)) break;
        uint8_t *st = ring + s * C::IN_B;
        mbar_arrive_expect_tx(&full[s], C::IN_B);
        tma_load_2d(st, &tmIn, &full[s], cb * 2 * BOXC, t * TM);
        tma_load_2d(st + TM * BOXC * 2, &tmIn, &full[s], cb * 2 * BOXC + BOXC, t * TM);
        if (g >= NBL && !mbar_wait(&bempty[sb], ((g / NBL) & 1) ^ 1)) break;
        mbar_arrive_expect_tx(&bfull[sb], C::BL_B);
        bulk_load(bring + sb * C::BL_B, p.blob + (int64_t)t * C::BL_B, C::BL_B, &bfull[sb]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_acc = tc_idesc(TM, C::AW, true, true);
      const uint32_t id_dx = tc_idesc(TM, 2 * BOXC, false, true);
      int seg = 0;
      bool ok = true;
      for (int64_t u = u0; ok && u < u1; ++u) {
        const int g = (int)(u - u0), s = g % NS, sb = g % NBL;
        const int t = (int)(u % nt);
        const bool first = u == u0 || t == 0, last = u == u1 - 1 || t == nt - 1;
        const int ab = seg & 1;
        if (first) {
          if (seg >= 2 && !(ok = mbar_wait(&aempty[ab], ((seg >> 1) & 1) ^ 1))) break;
          if (kDX && !(ok = mbar_wait(&acfull[C::NAC == 2 ? (seg & 1) : 0], (C::NAC == 2 ? seg >> 1 : seg) & 1)))
            break;
        }
        if (!(ok = mbar_wait(&full[s], (g / NS) & 1))) break;
        if (!(ok = mbar_wait(&bfull[sb], (g / NBL) & 1))) break;
        const int db = g & 1;
        if (kDX && g >= 2 && !(ok = mbar_wait(&dempty[db], ((g >> 1) & 1) ^ 1))) break;
        tc_fence_after();
        const uint32_t st = smem_u32(ring + s * C::IN_B), bl = smem_u32(bring + sb * C::BL_B);
        if (kDX) {
          // dX tile [128 rows][128 columns] = (dyb_hi + dyb_lo) * A^T
          const uint32_t ac = smem_u32(acbuf + (C::NAC == 2 ? (seg & 1) : 0) * C::AC1);
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int qk = 0; qk < RP / 16; ++qk) {
              const int pan = (qk * 16) / PW, in = ((qk * 16) % PW) * 2;
              const uint64_t ad =
                  tc_desc(bl + part * blob_tile(RP) + pan * (TM * PW * 2) + in, 16, 8 * PW * 2, PW * 2);
              const uint64_t bd = tc_desc(ac + qk * 2048, RP * 128, 1024, 128);
              tc_mma_bf16(tmem + db * TM, ad, bd, id_dx, (part == 0 && qk == 0) ? 0u : 1u);
            }
          tc_commit(&dfull[db]);
        }
        // acc[c][j] += sum over the tile's 128 rows of In[row][c] * blob[row][j]
        // (with HL: acc[c][j] from hi, acc[c][RP + j] from lo, in the same MMAs)
#pragma unroll
        for (int part = 0; part < (C::HL ? 1 : 2); ++part)
#pragma unroll
          for (int kk = 0; kk < TM / 16; ++kk) {
            const uint64_t ad = tc_desc(st + kk * 2048, TM * BOXC * 2, 1024, 128);
            const uint64_t bd = tc_desc(bl + part * blob_tile(RP) + kk * 16 * PW * 2,
                                        (C::HL || RP > PW) ? TM * PW * 2 : 16, 8 * PW * 2, PW * 2);
            tc_mma_bf16(tmem + C::ACC0 + ab * C::AW, ad, bd, id_acc, (first && part == 0 && kk == 0) ? 0u : 1u);
          }
        tc_commit(&bempty[sb]);
        tc_commit(kDX ? &xfree[s] : &empty[s]);
        if (last) {
          tc_commit(&afull[ab]);
          if (kDX) tc_commit(&acempty[C::NAC == 2 ? (seg & 1) : 0]);
          ++seg;
        }
      }
      tc_commit(mdone);
      mbar_wait(mdone, 0);
    }
    __syncwarp();
  } else {
    const int q = warp & 3, row = 32 * q + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    // with SPLIT warps 2-5 drain the dX tiles and warps 6-9 the accumulators
    const bool dxw = kDX && (!C::SPLIT || warp < 6);
    const int leader = C::SPLIT ? 6 * 32 : EPI0 * 32;
    int seg = 0;
    bool ok = true;   // after a timed-out wait: skip the work, keep the barrier sequence
    int pend = -1;    // stage whose dX store may still be reading it
    float v[RP];
    // unit u's dX tile (kDX)
    auto dx_unit = [&](int g, int cb, int t) {
      if (ok) ok = wait_warp(&dfull[g & 1], (g >> 1) & 1);
      if (ok) ok = wait_warp(&xfree[g % NS], (g / NS) & 1);
      if (ok) {
        // the dX tile: scaled (and added to the old dX), rounded to bf16 and
        // written over the stage's In tile (same swizzled layout), then each
        // warp stores its 32 rows with TMA (rows past M and columns past K are
        // clipped by the store)
        const int db = g & 1, s = g % NS;
        uint8_t *st = ring + s * C::IN_B;
        tc_fence_after();
        const int64_t grow = (int64_t)t * TM + row;
        const __nv_bfloat16 *dxr = p.dX + grow * p.lddx;
        const float sc = p.scale;
#pragma unroll 1
        for (int c0 = 0; c0 < 2 * BOXC; c0 += 32) {
          float d[32];
          tmem_ld32(tl + db * TM + c0, d);
#pragma unroll
          for (int c8 = 0; c8 < 32; c8 += 8) {
            const int cc = c0 + c8, col = cb * 2 * BOXC + cc;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = sc * d[c8 + e];
            if (kAccX && grow < p.M && col < p.C) {
              if (col + 8 <= p.C) {
                const uint4 o = *reinterpret_cast<const uint4 *>(dxr + col);
                const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 f = unpack_bf16(w[e]);
                  x[2 * e] += f.x;
                  x[2 * e + 1] += f.y;
                }
              } else {
                for (int e = 0; e < 8 && col + e < p.C; ++e) x[e] += __bfloat162float(dxr[col + e]);
              }
            }
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = pack_bf16(x[2 * e], x[2 * e + 1]);
            *reinterpret_cast<uint4 *>(st + (cc / BOXC) * (TM * BOXC * 2) + swz(row, (cc % BOXC) * 2, 128)) =
                make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&dempty[db]);
          tma_store_2d(&tmDX, st + q * 32 * 128, cb * 2 * BOXC, t * TM + 32 * q);
          tma_store_2d(&tmDX, st + TM * BOXC * 2 + q * 32 * 128, cb * 2 * BOXC + BOXC, t * TM + 32 * q);
          bulk_commit();
          if (pend >= 0) {
            bulk_wait_read1();
            mbar_arrive(&empty[pend]);
          }
          pend = s;
        }
      }
    };
    // the end of column block cb: its accumulator, the block reduction, the output rows
    auto acc_end = [&](int cb) {
      const int ab = seg & 1;
      if (ok) ok = wait_warp(&afull[ab], (seg >> 1) & 1);
#pragma unroll
      for (int j = 0; j < RP; ++j) v[j] = 0.f;
      if (ok) {
        tc_fence_after();
        tmem_row<RP>(tl + C::ACC0 + ab * C::AW, v);
        if constexpr (C::HL) {
          // the lo half, added in 16- or 32-column pieces
          if constexpr (RP == 16) {
            float w[16];
            tmem_ld16(tl + C::ACC0 + ab * C::AW + RP, w);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] += w[j];
          } else {
#pragma unroll
            for (int c = 0; c < RP; c += 32) {
              float w[32];
              tmem_ld32(tl + C::ACC0 + ab * C::AW + RP + c, w);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[c + j] += w[j];
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&aempty[ab]);
      }
      ++seg;
      if (!reduce_segment<RP>(p.U, p.G, i, cb, nt, p.part, p.counters + cb, row, v, s_flag, leader)) return;
      const int64_t c = (int64_t)cb * TM + row;
      if (c < p.C && p.out_vec4) {
        // fp32 rows of the output contiguous and 16-byte aligned: 16-byte stores
        float *orow = reinterpret_cast<float *>(p.out) + c * p.out_sc;
#pragma unroll
        for (int j = 0; j < RP; j += 4)
          if (j < p.r)
            *reinterpret_cast<float4 *>(orow + j) = make_float4(p.out_scale * v[j], p.out_scale * v[j + 1],
                                                                p.out_scale * v[j + 2], p.out_scale * v[j + 3]);
      } else if (c < p.C) {
#pragma unroll
        for (int j = 0; j < RP; ++j) {
          if (j >= p.r) break;
          const int64_t o = c * p.out_sc + (int64_t)j * p.out_sj;
          if (p.out_bf16) reinterpret_cast<__nv_bfloat16 *>(p.out)[o] = __float2bfloat16_rn(p.out_scale * v[j]);
          else reinterpret_cast<float *>(p.out)[o] = p.out_scale * v[j];
        }
      }
    };
    if (C::SPLIT) {
      for (int64_t u = u0; u < u1; ++u) {
        const int g = (int)(u - u0);
        const int cb = (int)(u / nt), t = (int)(u % nt);
        if (dxw) dx_unit(g, cb, t);
        else if (u == u1 - 1 || t == nt - 1) acc_end(cb);
      }
    } else {
      for (int64_t u = u0; u < u1; ++u) {
        const int g = (int)(u - u0);
        const int cb = (int)(u / nt), t = (int)(u % nt);
        if (kDX) dx_unit(g, cb, t);
        if (u == u1 - 1 || t == nt - 1) acc_end(cb);
      }
    }
    if (dxw && lane == 0) {
      bulk_wait_read_all();
      if (pend >= 0) mbar_arrive(&empty[pend]);
      bulk_wait_all();
    }
  }
  if (!p.wait_first) pdl_wait();
  if (!kDX) pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM);
  }
}

}  // namespace tc

// ----------------------------------------------------------------------------- host side
namespace {

using namespace tc;

// Big row-major bf16 operand [rows][cols] with row stride ld: boxes of 64 columns x box_rows rows.
bool map_rows_box(CUtensorMap *m, const void *p, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows) {
  uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  uint64_t str[1] = {(uint64_t)ld * 2};
  uint32_t box[2] = {64, box_rows};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
bool map_big128(CUtensorMap *m, const void *p, int64_t rows, int64_t cols, int64_t ld) {
  return map_rows_box(m, p, rows, cols, ld, 128);
}
// Ac [r][K] (k contiguous, row stride lda): boxes of 64 k x RP rows.
bool map_ac_tc(CUtensorMap *m, const void *p, int64_t K, int r, int64_t lda, int RP) {
  uint64_t dims[2] = {(uint64_t)K, (uint64_t)r};
  uint64_t str[1] = {(uint64_t)lda * 2};
  uint32_t box[2] = {64, (uint32_t)RP};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// Bc [L][r] (j contiguous, row stride ldb): boxes of PW j x 64 rows.
bool map_bc_tc(CUtensorMap *m, const void *p, int64_t L, int r, int64_t ldb, int RP) {
  const int PW = RP < 64 ? RP : 64;
  uint64_t dims[2] = {(uint64_t)r, (uint64_t)L};
  uint64_t str[1] = {(uint64_t)ldb * 2};
  uint32_t box[2] = {(uint32_t)PW, 64};
  const CUtensorMapSwizzle sw = PW >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : PW == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                           : CU_TENSOR_MAP_SWIZZLE_32B;
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p, dims, str, box, sw);
}

// Persistent grid: every SM holds one CTA of these kernels (their shared memory
// allows no more).  Stream-K passes give every CTA at least min_units units
// (kMinUnits: fewer CTAs on small problems, and a bound on the partial sums), at
// most kMaxGrid CTAs (one per SM; more than any GB300 has), so that workspace
// sizes depend on the arguments only.
constexpr int kMinUnits = 8;
constexpr int kMaxGrid = 160;
int grid_for(int64_t units, const void *kern, size_t smem, int min_units, int threads = NTHR) {
  const int occ = occupancy(kern, threads, smem);
  return (int)std::max<int64_t>(
      1, std::min<int64_t>({ceil_div(units, min_units), (int64_t)occ * num_sms(), (int64_t)kMaxGrid}));
}
// partial-sum slots (two per CTA) of a stream-K pass over U units
int64_t part_slots(int64_t U) { return 2 * std::max<int64_t>(1, std::min<int64_t>(ceil_div(U, kMinUnits), kMaxGrid)); }

// workspace of one rows pass (partials, blob) and one column pass (partials);
// the counters are counted by the caller
template <int RP>
size_t ws_rows(int64_t M, int64_t C) {
  const int64_t nrb = ceil_div(M, TM), nc = ceil_div(C, RUC);
  return ws_round((size_t)part_slots(nrb * nc) * TM * RP * 4) + ws_round((size_t)nrb * 2 * blob_tile(RP));
}
template <int RP>
size_t ws_col(int64_t M, int64_t C) {
  const int64_t nt = ceil_div(M, TM), ncb = ceil_div(C, TM);
  return ws_round((size_t)part_slots(ncb * nt) * TM * RP * 4);
}

// h = In * W (W = A: K-major, kWMN = false; W = B^T from B in PEFT layout: kWMN = true)
// into the blob (and fp32 rows into hout when given); with hin, the saved fp32 h
// [M][ldhin] is also converted into the blob hblob.
template <int RP, bool kWMN>
lora_status_t launch_rows(const void *in, int64_t ld_in, int64_t M, int64_t Cdim, int r, const CUtensorMap &tW,
                          int *counters, WsCarver &ws, uint8_t **blob_out, float *hout, int64_t ldh, cudaStream_t st,
                          const float *hin = nullptr, int64_t ldhin = 0, uint8_t *hblob = nullptr) {
  using Cf = RowsCfg<RP, kWMN>;
  auto kern = rows_kernel<RP, kWMN>;
  LORA_CUDA(ensure_smem((const void *)kern, Cf::BYTES));
  const int64_t nrb = ceil_div(M, TM), nc = ceil_div(Cdim, RUC);
  const int G = grid_for(nrb * nc, (const void *)kern, Cf::BYTES, kMinUnits);
  float *part = (float *)ws.take((size_t)2 * G * TM * RP * 4);
  uint8_t *blob = (uint8_t *)ws.take((size_t)nrb * 2 * blob_tile(RP));
  if (!part || !blob) return LORA_ERR_WORKSPACE;
  CUtensorMap tIn;
  if (!map_big128(&tIn, in, M, Cdim, ld_in)) return LORA_ERR_ALIGNMENT;
  TcRowsArgs p{};
  p.M = (int)M;
  p.C = (int)Cdim;
  p.r = r;
  p.nc = (int)nc;
  p.U = nrb * nc;
  p.G = G;
  p.part = part;
  p.counters = counters;
  p.blob = blob;
  p.hout = hout;
  p.ldh = ldh;
  p.h_vec4 = hout != nullptr && (reinterpret_cast<uintptr_t>(hout) & 15) == 0 && ldh % 4 == 0 && r % 4 == 0;
  p.hin = hin;
  p.ldhin = ldhin;
  p.hblob = hblob;
  LORA_CUDA(launch(kern, dim3((unsigned)G), dim3(NTHR), Cf::BYTES, st, 1, true, tIn, tW, p));
  *blob_out = blob;
  return LORA_OK;
}

// acc = In^T * blob over 128-column blocks of In (dA or dB^T), with the dX tiles when kDX.
template <int RP, bool kDX>
lora_status_t launch_col(const void *in, int64_t ld_in, int64_t M, int64_t Cdim, int r, const uint8_t *blob,
                         const CUtensorMap *tAc, float scale, void *out, int64_t out_sc, int64_t out_sj, bool out_bf16,
                         void *dX, int64_t lddx, bool dx_acc, int *counters, WsCarver &ws, cudaStream_t st,
                         bool wait_first = true) {
  using Cf = ColCfg<RP, kDX>;
  auto kern = kDX ? (dx_acc ? col_kernel<RP, true, true> : col_kernel<RP, true, false>) : col_kernel<RP, false, false>;
  LORA_CUDA(ensure_smem((const void *)kern, Cf::BYTES));
  const int64_t nt = ceil_div(M, TM), ncb = ceil_div(Cdim, TM);
  const int G = grid_for(ncb * nt, (const void *)kern, Cf::BYTES, kMinUnits, Cf::NT);
  float *part = (float *)ws.take((size_t)2 * G * TM * RP * 4);
  if (!part) return LORA_ERR_WORKSPACE;
  CUtensorMap tIn, tDX;
  if (!map_big128(&tIn, in, M, Cdim, ld_in)) return LORA_ERR_ALIGNMENT;
  if (kDX && !map_rows_box(&tDX, dX, M, Cdim, lddx, 32)) return LORA_ERR_ALIGNMENT;
  TcColArgs p{};
  p.M = (int)M;
  p.C = (int)Cdim;
  p.r = r;
  p.nt = (int)nt;
  p.U = ncb * nt;
  p.G = G;
  p.part = part;
  p.counters = counters;
  p.blob = blob;
  p.scale = scale;
  p.out_scale = scale;
  p.out = out;
  p.out_sc = out_sc;
  p.out_sj = out_sj;
  p.out_bf16 = out_bf16 ? 1 : 0;
  p.out_vec4 = !out_bf16 && out_sj == 1 && out_sc % 4 == 0 && r % 4 == 0 &&
               (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  p.dX = (__nv_bfloat16 *)dX;
  p.lddx = lddx;
  p.wait_first = wait_first ? 1 : 0;
  LORA_CUDA(launch(kern, dim3((unsigned)G), dim3(Cf::NT), Cf::BYTES, st, 1, true, tIn, kDX ? *tAc : tIn, kDX ? tDX : tIn,
                   p));
  return LORA_OK;
}

template <int RP>
lora_status_t launch_expand(const uint8_t *blob, const SingleArgs &a, const CUtensorMap &tB, int *next,
                            cudaStream_t st) {
  using Cf = ExpCfg<RP>;
  auto kern = expand_kernel<RP>;
  LORA_CUDA(ensure_smem((const void *)kern, Cf::BYTES));
  const int64_t nrb = ceil_div(a.M, TM), nl = ceil_div(a.L, EUC);
  const int G = grid_for(nrb * nl, (const void *)kern, Cf::BYTES, 1);
  CUtensorMap tY, tYs;
  if (!map_big128(&tY, a.Y, a.M, a.L, a.ldy) || !map_rows_box(&tYs, a.Y, a.M, a.L, a.ldy, 32))
    return LORA_ERR_ALIGNMENT;
  TcExpArgs p{};
  p.M = (int)a.M;
  p.L = (int)a.L;
  p.nl = (int)nl;
  p.U = nrb * nl;
  p.G = G;
  // the last eighth of the units (in chunks of about a thirtieth of a CTA's
  // share) go to whichever CTA is free first
  const bool tail = next != nullptr && p.U >= 4 * (int64_t)G;
  p.CH = tail ? (int)std::max<int64_t>(1, std::min<int64_t>(4, p.U / (32 * (int64_t)G))) : 1;
  p.Us = p.U - (tail ? p.U / 8 / p.CH * p.CH : 0);
  p.next = tail ? next : nullptr;
  p.blob = blob;
  p.Y = (__nv_bfloat16 *)a.Y;
  p.ldy = a.ldy;
  p.scale = a.scale;
  LORA_CUDA(launch(kern, dim3((unsigned)G), dim3(NTHR), Cf::BYTES, st, 1, true, tY, tYs, tB, p));
  return LORA_OK;
}

lora_status_t pack_tc(const SingleArgs &a, const SingleLayout &lay, WsCarver &ws, const void **Ac, const void **Bc,
                      cudaStream_t st) {
  if (lay.pack_A) {
    void *d = ws.take((size_t)a.r * lay.lda * 2);
    if (!d) return LORA_ERR_WORKSPACE;
    LORA_TRY(pack_bf16_2d(a.A, a.sA_r, a.sA_k, a.r, a.K, d, lay.lda, st));
    *Ac = d;
  } else if (Ac) {
    *Ac = a.A;
  }
  if (lay.pack_B) {
    void *d = ws.take((size_t)a.L * lay.ldb * 2);
    if (!d) return LORA_ERR_WORKSPACE;
    LORA_TRY(pack_bf16_2d(a.B, a.sB_l, a.sB_r, a.L, a.r, d, lay.ldb, st));
    *Bc = d;
  } else if (Bc) {
    *Bc = a.B;
  }
  return LORA_OK;
}

// Ticket counters of every stream-K pass of one op, zeroed by one memset.
int *take_counters(WsCarver &ws, int64_t n, cudaStream_t st, lora_status_t *err) {
  int *c = (int *)ws.take((size_t)n * 4);
  if (!c) {
    *err = LORA_ERR_WORKSPACE;
    return nullptr;
  }
  *err = cudaMemsetAsync(c, 0, (size_t)n * 4, st) == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
  return c;
}

template <int RP>
lora_status_t forward_rp(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  SingleLayout lay = plan_layout(a, true, a.L > 0);
  WsCarver carver(ws, ws_bytes);
  const void *Ac = nullptr, *Bc = nullptr;
  lora_status_t e;
  // the rows pass's tickets and the expand's claim counter
  int *cnt = take_counters(carver, ceil_div(a.M, TM) + 1, st, &e);
  LORA_TRY(e);
  LORA_TRY(pack_tc(a, lay, carver, &Ac, &Bc, st));
  CUtensorMap tA, tB;
  if (!map_ac_tc(&tA, Ac, a.K, a.r, lay.lda, RP)) return LORA_ERR_ALIGNMENT;
  uint8_t *blob = nullptr;
  LORA_TRY((launch_rows<RP, false>(a.X, a.ldx, a.M, a.K, a.r, tA, cnt, carver, &blob, a.h, a.ldh, st)));
  if (a.L == 0) return LORA_OK;
  if (!map_bc_tc(&tB, Bc, a.L, a.r, lay.ldb, RP)) return LORA_ERR_ALIGNMENT;
  return launch_expand<RP>(blob, a, tB, cnt + ceil_div(a.M, TM), st);
}

// dyb blob, then dX and dA; cnt holds ceil(M/128) + ceil(K/128) counters.  With
// hblob, the dyb pass also writes the blob of the saved h (a.h) there.
template <int RP>
lora_status_t dxda_rp(const SingleArgs &a, int *cnt, WsCarver &carver, cudaStream_t st, uint8_t *hblob = nullptr) {
  SingleLayout lay = plan_layout(a, true, true);
  const void *Ac = nullptr, *Bc = nullptr;
  LORA_TRY(pack_tc(a, lay, carver, &Ac, &Bc, st));
  CUtensorMap tA, tB;
  if (!map_ac_tc(&tA, Ac, a.K, a.r, lay.lda, RP) || !map_bc_tc(&tB, Bc, a.L, a.r, lay.ldb, RP))
    return LORA_ERR_ALIGNMENT;
  uint8_t *blob = nullptr;
  LORA_TRY((launch_rows<RP, true>(a.dY, a.lddy, a.M, a.L, a.r, tB, cnt, carver, &blob, nullptr, 0, st,
                                   hblob ? (const float *)a.h : nullptr, a.ldh, hblob)));
  return launch_col<RP, true>(a.X, a.ldx, a.M, a.K, a.r, blob, &tA, a.scale, a.dA, a.sdA_k, a.sdA_r, a.grad_lo != 0,
                              a.dX, a.lddx, a.dx_acc != 0, cnt + ceil_div(a.M, TM), carver, st);
}

// dB from a blob of h; cnt holds ceil(L/128) counters.  wait_first = false when
// the previous launch neither writes the blob nor dY (the dX pass of lora_backward).
template <int RP>
lora_status_t db_from_blob(const SingleArgs &a, const uint8_t *hblob, int *cnt, WsCarver &carver, cudaStream_t st,
                           bool wait_first = true) {
  return launch_col<RP, false>(a.dY, a.lddy, a.M, a.L, a.r, hblob, nullptr, a.scale, a.dB, a.sdB_l, a.sdB_r,
                               a.grad_lo != 0, nullptr, 0, false, cnt, carver, st, wait_first);
}

template <int RP>
lora_status_t dxda_op(const SingleArgs &a, WsCarver &carver, cudaStream_t st) {
  lora_status_t e;
  int *cnt = take_counters(carver, ceil_div(a.M, TM) + ceil_div(a.K, TM), st, &e);
  LORA_TRY(e);
  return dxda_rp<RP>(a, cnt, carver, st);
}

template <int RP>
lora_status_t db_op(const SingleArgs &a, WsCarver &carver, cudaStream_t st) {
  lora_status_t e;
  const int64_t nrb = ceil_div(a.M, TM);
  int *cnt = take_counters(carver, nrb + ceil_div(a.L, TM), st, &e);
  LORA_TRY(e);
  SingleLayout lay = plan_layout(a, true, false);
  const void *Ac = nullptr;
  LORA_TRY(pack_tc(a, lay, carver, &Ac, nullptr, st));
  CUtensorMap tA;
  if (!map_ac_tc(&tA, Ac, a.K, a.r, lay.lda, RP)) return LORA_ERR_ALIGNMENT;
  uint8_t *blob = nullptr;
  LORA_TRY((launch_rows<RP, false>(a.X, a.ldx, a.M, a.K, a.r, tA, cnt, carver, &blob, nullptr, 0, st)));
  return db_from_blob<RP>(a, blob, cnt + nrb, carver, st);
}

template <int RP>
lora_status_t backward_op(const SingleArgs &a, WsCarver &carver, cudaStream_t st) {
  lora_status_t e;
  const int64_t nrb = ceil_div(a.M, TM), nkb = ceil_div(a.K, TM);
  int *cnt = take_counters(carver, nrb + nkb + ceil_div(a.L, TM), st, &e);
  LORA_TRY(e);
  uint8_t *hb = (uint8_t *)carver.take((size_t)nrb * 2 * blob_tile(RP));
  if (!hb) return LORA_ERR_WORKSPACE;
  LORA_TRY(dxda_rp<RP>(a, cnt, carver, st, hb));
  return db_from_blob<RP>(a, hb, cnt + nrb + nkb, carver, st, false);
}

template <typename F>
auto by_rank(int r, F f) -> decltype(f(std::integral_constant<int, 16>())) {
  switch (rank_bucket(r)) {
    case 16: return f(std::integral_constant<int, 16>());
    case 32: return f(std::integral_constant<int, 32>());
    case 64: return f(std::integral_constant<int, 64>());
    default: return f(std::integral_constant<int, 128>());
  }
}

}  // namespace

size_t tc_ws_bytes(int op, int64_t M, int64_t K, int64_t L, int r) {
  if (M <= 0 || K < 0 || L < 0 || r <= 0) return 0;
  const size_t packA = ws_round((size_t)r * round_up(K, 8) * 2);
  const size_t packB = ws_round((size_t)L * round_up(r, 8) * 2);
  const int64_t nrb = ceil_div(M, TM), nkb = ceil_div(K, TM), nlb = ceil_div(L, TM);
  return by_rank(r, [&](auto rp) -> size_t {
    constexpr int RP = decltype(rp)::value;
    const size_t hb = ws_round((size_t)nrb * 2 * blob_tile(RP));
    if (op == LORA_OP_FORWARD) return ws_round((size_t)(nrb + 1) * 4) + packA + packB + ws_rows<RP>(M, K);
    if (op == LORA_OP_BACKWARD_DX_DA)
      return ws_round((size_t)(nrb + nkb) * 4) + packA + packB + ws_rows<RP>(M, L) + ws_col<RP>(M, K);
    if (op == LORA_OP_BACKWARD_DB)
      return ws_round((size_t)(nrb + nlb) * 4) + packA + ws_rows<RP>(M, K) + ws_col<RP>(M, L);
    if (op == LORA_OP_BACKWARD)
      return ws_round((size_t)(nrb + nkb + nlb) * 4) + packA + packB + ws_rows<RP>(M, L) + ws_col<RP>(M, K) + hb +
             ws_col<RP>(M, L);
    return (size_t)0;
  });
}

lora_status_t forward_tc(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  return by_rank(a.r, [&](auto rp) { return forward_rp<decltype(rp)::value>(a, ws, ws_bytes, st); });
}
lora_status_t backward_dx_da_tc(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  WsCarver c(ws, ws_bytes);
  return by_rank(a.r, [&](auto rp) { return dxda_op<decltype(rp)::value>(a, c, st); });
}
lora_status_t backward_db_tc(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  WsCarver c(ws, ws_bytes);
  return by_rank(a.r, [&](auto rp) { return db_op<decltype(rp)::value>(a, c, st); });
}
lora_status_t backward_tc(const SingleArgs &a, void *ws, size_t ws_bytes, cudaStream_t st) {
  WsCarver c(ws, ws_bytes);
  return by_rank(a.r, [&](auto rp) { return backward_op<decltype(rp)::value>(a, c, st); });
}

int read_clear_error_single_tc() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
  return v;
}

}  // namespace lora
