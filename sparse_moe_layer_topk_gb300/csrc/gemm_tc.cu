// Persistent tcgen05 GEMM engine for sm_103a.
//
// One CTA per SM walks a tile list (dense, ragged-M grouped, or ragged-K
// grouped). Warp roles:
//   warp 0      TMA producer: 128 x 64 A tile and BN x 64 B tile per stage,
//               128-byte swizzled, K-major or MN-major per operand.
//   warp 1      TMEM allocation + MMA issue: one elected lane issues
//               tcgen05.mma (M=128, N=BN, K=16) x 4 per stage into a
//               double-buffered fp32 accumulator in tensor memory.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, fused elementwise
//   (or 2..9)   work (SwiGLU, routing-weight scale, SwiGLU backward), stores.
//   2 more      gathering launches only: copy the gathered operand's rows
//               (cp.async) into the stage while TMA loads the other operand.
// The accumulator double buffer lets the epilogue of tile i overlap the
// mainloop of tile i+1. Ragged expert segments are handled on the device:
// grouped-M tiles come from the per-expert tile schedule, grouped-K tiles mask
// the rows past the segment end in shared memory before the MMA reads them.
//
// Source of the operation: the Grouped GEMM over per-expert token batches of
// the "昇腾实现Kimi K3.1 Pro模型LoRA训练适配" page, section
// "MoE(Mixture of Experts):算子融合与通信协同", run over all local experts
// through one compute view as in the "TorchTitan Ascend开源" page, section
// "权重预取与梯度归约".
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "timing.h"

namespace moe {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int CHUNK_BYTES = 64 * 128;  // one 64-row x 128-byte swizzled block
constexpr int MISC_BYTES = 768;  // barriers (256 B) + spare (512 B)
// Warps that copy a gathered operand's rows (cp.async) in gathering launches.
constexpr int kGatherWarps = 2;

// BN: tile width (UMMA N); EW: epilogue warps (4, or 8 for heavy epilogues:
// two warps per TMEM lane quadrant, splitting the tile's column chunks).
// PAIR: the CTA is one of a pair computing 256-row tiles with cta_group::2 MMAs
// (each CTA holds its 128 rows of A and half of B's columns).
// SBWD: the SwiGLU-backward epilogue with TMA-staged inputs (4 warps, each
// with a ring of SLOTS 6 KB slots for a chunk's g, u and h blocks: four where
// the stages leave room (32 KB stages), else three).
template <int BN, int EW, bool CW16 = false, bool PAIR = false, bool SBWD = false>
struct Cfg {
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES =
      SBWD ? ((BN == 256 && !PAIR) ? 3 : 4)
           : PAIR ? ((EW == 8 && !CW16) ? 5 : 6)
                  : ((BN == 256) ? ((EW == 8 && !CW16) ? 3 : 4) : ((EW == 8 && !CW16) ? 5 : 6));
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int THREADS = 64 + 32 * EW;
  // Per-warp output staging, a ring of slots of one chunk's output each (4 KB
  // fp32 or 2 KB bf16 for a 32-column block; SwiGLU chunks hold two or three
  // blocks), so that a chunk's bulk store may still be reading its slot while
  // the next chunks are staged: one fp32 / three bf16 slots with 4 epilogue
  // warps (a whole tile table of a ragged-K weight gradient measured faster
  // than a second fp32 slot), one SwiGLU chunk with 8.
  static constexpr int SLOTS = (PAIR || BN == 128) ? 4 : 3;
  static constexpr int STG = SBWD ? SLOTS * 6144 : (CW16 ? 3072 : (EW == 8 ? 6144 : 7168));
  // The rest of the 227 KB (after 1 KB alignment slack and the barriers) holds
  // the CTA's table of decoded grouped tiles, 16 bytes per tile.
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int TT_FIT =
      (SMEM_LIMIT - 1024 - MISC_BYTES - STAGES * STAGE_BYTES - EW * STG) / 16 * 16;
  static constexpr int TT_BYTES = TT_FIT > 16384 ? 16384 : TT_FIT;
  static constexpr int TT_CAP = TT_BYTES / 16;
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + EW * STG + 1024 + MISC_BYTES + TT_BYTES;
  static_assert(TT_CAP >= 64, "tile table");
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
};

struct Params {
  int sched, M, N, K, G;
  const int* offsets;
  const int* tile_sched;
  const int* expert_order;  // grouped-M: position -> group (nullptr: identity)
  int a_mn, b_mn, b_rank3;
  // MN-major operand read through a chunked map ([batch][cols/64][rows][64]):
  // all of a tile's 64-column chunks in one copy instead of one copy per chunk
  int a_chunked, b_chunked;
  int b_batch_mode, n_tiles_per_batch, k_per_batch;
  int swiglu_b, f;
  int mt, nt;         // m tiles (dense / grouped-K), n tiles
  int splitk, kslice; // dense: K split into `splitk` slices of `kslice` (multiple of 64)
  int kcat;           // dense: K index where A/B switch to the second operand pair (0: none)
  int ncat;           // dense pairs: output column where B / C switch to B2 / C2 (0: none)
  int c2_bf16;        // C2 holds bf16 (else fp32)
  int total_static;   // tile count when it does not depend on device data
  int epi;
  void* C;
  long long ldc, c_batch_stride;
  int c_batch_n, c_bf16, accumulate;
  const float* row_w;
  bf16* gu;
  long long ldgu;
  // FP8 cache of g|u (instead of gu): E4M3 bytes [R][ldgu] and one fp32 scale
  // per row and 64-feature block, gu_scale[row * ld_scale + block] (the f / 64
  // g blocks, then the u blocks)
  uint8_t* gu8;
  float* gu_scale;
  int ld_scale;
  bf16* h;
  long long ldh;
  bf16* aux;
  long long ldaux;
  float* dw_part;
  int dw_nparts;
  int* err_flag;
  int c0_rank3;  // the C store map is 3-D (grouped-K groups or column batches)
  // Row gather: permuted row r of the gathered operand is row gather_idx[r] of its
  // (unpermuted) source tensor, copied by the gather warps (cp.async).
  const int* gather_idx;
  int gather_a, gather_b;
  const bf16* gsrc;  // the gathered operand's source tensor [rows][gwidth], gld apart
  long long gld;
  int gwidth;
  int tt_cap;  // tiles of a CTA held in its shared-memory table (the rest are decoded inline)
  int m64;     // grouped-M: tiles of at most 64 rows run M = 64 MMAs (see quad_rows)
  int pair;  // 1: CTA pairs (cluster of 2) own 256-row tiles (dense schedule)
  int mt2;   // pair rows of tiles: ceil(mt / 2)
};

struct Tile {
  int g;       // group (grouped schedules)
  int m0;      // first output row (and A row / A column coordinate)
  int rows;    // valid output rows
  int n_blk;   // n tile index
  int nb0;     // first B column/row coordinate of the tile (within its batch)
  int batch;   // B batch coordinate (BATCH_GROUP / BATCH_FROM_N)
  int k0;      // first K coordinate
  int krows;   // valid K rows (grouped-K), else K
  int nk;      // number of 64-wide K blocks
};

// Rows of the accumulator in each tensor-memory lane quadrant. An M = 128 MMA
// puts row r in lane r (32 rows per quadrant); an M = 64 MMA (grouped-M tiles
// of at most 64 rows when p.m64) puts rows 16q .. 16q+15 in lanes 32q ..
// 32q+15 of quadrant q. The epilogue warp of quadrant q reads its 32 lanes and
// uses the first quad_rows of them.
__device__ __forceinline__ int quad_rows(const Params& p, int rows) {
  return (p.m64 && p.sched == SCHED_GROUPED_M && rows <= 64) ? 16 : 32;
}

__device__ __forceinline__ int total_tiles(const Params& p) {
  if (p.sched == SCHED_GROUPED_M) return __ldg(p.tile_sched + p.G) * p.nt;
  return p.total_static;
}

// A CTA (or a CTA pair) walks tiles tile_begin + i * tile_step.
template <bool PAIR>
__device__ __forceinline__ int tile_begin() {
  return static_cast<int>(blockIdx.x) >> (PAIR ? 1 : 0);
}
template <bool PAIR>
__device__ __forceinline__ int tile_step() {
  return static_cast<int>(gridDim.x) >> (PAIR ? 1 : 0);
}

template <int BN, bool PAIR = false>
__device__ __forceinline__ Tile decode(const Params& p, int t) {
  Tile ti;
  const int bn_eff = p.swiglu_b ? BN / 2 : BN;
  if (p.sched == SCHED_GROUPED_M) {
    int lo = 0, hi = p.G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.tile_sched + mid) * p.nt <= t) lo = mid; else hi = mid;
    }
    const int pos = lo;
    const int g = p.expert_order ? __ldg(p.expert_order + pos) : pos;
    const int ts0 = __ldg(p.tile_sched + pos);
    const int mtg = __ldg(p.tile_sched + pos + 1) - ts0;
    const int local = t - ts0 * p.nt;
    ti.g = g;
    ti.n_blk = local / mtg;
    const int m_blk = local - ti.n_blk * mtg;
    const int seg0 = __ldg(p.offsets + g), seg1 = __ldg(p.offsets + g + 1);
    ti.m0 = seg0 + m_blk * BM;
    ti.rows = min(BM, seg1 - ti.m0);
    ti.nb0 = ti.n_blk * bn_eff;
    ti.batch = g;
    ti.k0 = 0;
    ti.krows = p.K;
    ti.nk = (p.K + BK - 1) / BK;
  } else if (p.sched == SCHED_GROUPED_K) {
    const int per = p.mt * p.nt;
    const int g = t / per;
    const int local = t - g * per;
    ti.g = g;
    ti.n_blk = local / p.mt;
    const int m_blk = local - ti.n_blk * p.mt;
    ti.m0 = m_blk * BM;
    ti.rows = min(BM, p.M - ti.m0);
    ti.nb0 = ti.n_blk * bn_eff;
    ti.batch = 0;
    const int seg0 = __ldg(p.offsets + g), seg1 = __ldg(p.offsets + g + 1);
    ti.k0 = seg0;
    ti.krows = seg1 - seg0;
    ti.nk = (ti.krows + BK - 1) / BK;
  } else {
    // split-K: the slice index is the outer tile index and takes the role of g;
    // a CTA pair's tile is two 128-row blocks, the CTA's rank picking its block
    // (the second block of a last odd pair has no rows: rows <= 0)
    const int mtx = PAIR ? p.mt2 : p.mt;
    const int per = mtx * p.nt;
    ti.g = t / per;
    t -= ti.g * per;
    // n fastest: the n tiles of one row block run side by side, so an A larger
    // than L2 (read by each of them) comes from DRAM once
    int m_blk = t / p.nt;
    ti.n_blk = t - m_blk * p.nt;
    if (PAIR) m_blk = 2 * m_blk + static_cast<int>(cluster_ctarank());
    ti.m0 = m_blk * BM;
    ti.rows = min(BM, p.M - ti.m0);
    if (p.b_batch_mode == BATCH_FROM_N) {
      ti.batch = ti.n_blk / p.n_tiles_per_batch;
      ti.nb0 = (ti.n_blk - ti.batch * p.n_tiles_per_batch) * bn_eff;
    } else {
      ti.batch = 0;
      ti.nb0 = ti.n_blk * bn_eff;
    }
    ti.k0 = ti.g * p.kslice;
    ti.krows = min(p.kslice, p.K - ti.k0);
    ti.nk = (ti.krows + BK - 1) / BK;
  }
  return ti;
}

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, int* err_flag) {
  *abort_flag = 1;
  set_flag(err_flag, MOE_FLAG_TIMEOUT);
}

// Table entry of a grouped tile: grouped-M {g, m0, rows, n_blk}; grouped-K
// {g, n_blk << 16 | m_blk, k0, krows}.
template <int BN>
__device__ __forceinline__ int4 pack_tile(const Params& p, const Tile& ti) {
  if (p.sched == SCHED_GROUPED_M) return make_int4(ti.g, ti.m0, ti.rows, ti.n_blk);
  return make_int4(ti.g, (ti.n_blk << 16) | (ti.m0 / BM), ti.k0, ti.krows);
}

// The i-th tile (t = blockIdx.x + i * gridDim.x) of this CTA: from the table when
// it holds it (the first `cap` tiles), else decoded from the schedule.
template <int BN, bool PAIR = false>
__device__ __forceinline__ Tile tile_of(const Params& p, const int4* ttab, int i, int t) {
  if (p.sched == SCHED_DENSE || i >= p.tt_cap) return decode<BN, PAIR>(p, t);
  const int4 e = ttab[i];
  const int bn_eff = p.swiglu_b ? BN / 2 : BN;
  Tile ti;
  ti.g = e.x;
  if (p.sched == SCHED_GROUPED_M) {
    ti.m0 = e.y;
    ti.rows = e.z;
    ti.n_blk = e.w;
    ti.batch = e.x;
    ti.k0 = 0;
    ti.krows = p.K;
    ti.nk = (p.K + BK - 1) / BK;
  } else {
    ti.n_blk = e.y >> 16;
    ti.m0 = (e.y & 0xFFFF) * BM;
    ti.rows = min(BM, p.M - ti.m0);
    ti.batch = 0;
    ti.k0 = e.z;
    ti.krows = e.w;
    ti.nk = (e.w + BK - 1) / BK;
  }
  ti.nb0 = ti.n_blk * bn_eff;
  return ti;
}

// ------------------------------------------------------------------ producer

template <int BN, int EW, bool CW16, bool PAIR, int GW, bool SBWD>
__device__ void producer_loop(const Params& p, const CUtensorMap* mapA, const CUtensorMap* mapB,
                              const CUtensorMap* mapA2, const CUtensorMap* mapB2,
                              uint8_t* smem, uint64_t* full, uint64_t* empty, const int4* ttab,
                              volatile int* abort_flag) {
  // Run by one lane. PAIR: the CTA loads its own 128 rows of A and its half of
  // the tile's B columns. A gathered operand (p.gather_a / p.gather_b) is copied
  // by the gather warps instead; the stage's expected bytes are then the other
  // operand's alone.
  using C = Cfg<BN, EW, CW16, PAIR, SBWD>;
  const int half_n = PAIR ? static_cast<int>(cluster_ctarank()) * (BN / 2) : 0;
  int stage = 0;
  uint32_t phase = 0;
  long long issued = 0;
  const int total = total_tiles(p);
  const bool gather_a = GW > 0 && p.gather_a, gather_b = GW > 0 && p.gather_b;
  const uint32_t tx_bytes =
      C::STAGE_BYTES - (gather_a ? A_BYTES : 0) - (gather_b ? C::B_BYTES : 0);
  bool ok = true;
  int it = 0;
  for (int t = tile_begin<PAIR>(); t < total && ok; t += tile_step<PAIR>(), ++it) {
    const Tile ti = tile_of<BN, PAIR>(p, ttab, it, t);
    for (int kb = 0; kb < ti.nk; ++kb) {
      // (pairs: the stage is freed by the first CTA's MMA completion, a tcgen05
      // commit multicast to both CTAs)
      if (!mbar_wait<PAIR>(&empty[stage], phase ^ 1u, abort_flag)) {
        raise_abort(abort_flag, p.err_flag);
        ok = false;
        break;
      }
      const int k = ti.k0 + kb * BK;
      const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
      const uint32_t sB = sA + A_BYTES;
      int kb_coord = k, batch = ti.batch;
      if (p.b_batch_mode == BATCH_FROM_K) {
        batch = k / p.k_per_batch;
        kb_coord = k - batch * p.k_per_batch;
      }
      if (PAIR) {
        // Both CTAs' copies of the stage count on the first CTA's full barrier,
        // whose producer posts the bytes of both.
        const uint32_t fb = half_n == 0 ? smem_u32(&full[stage])
                                        : cluster_map(smem_u32(&full[stage]), 0);
        if (half_n == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
        if (p.kcat > 0 && k >= p.kcat) {
          tma_load_2d_pair(sA, mapA2, fb, k - p.kcat, ti.m0);
          tma_load_2d_pair(sB, mapB2, fb, k - p.kcat, ti.nb0 + half_n);
        } else {
          if (!p.a_mn) {
            tma_load_2d_pair(sA, mapA, fb, k, ti.m0);
          } else if (p.a_chunked) {
            tma_load_3d_pair(sA, mapA, fb, 0, k, ti.m0 >> 6);
          } else {
            tma_load_2d_pair(sA, mapA, fb, ti.m0, k);
            tma_load_2d_pair(sA + CHUNK_BYTES, mapA, fb, ti.m0 + 64, k);
          }
          if (!p.b_mn) {
            if (p.b_rank3) tma_load_3d_pair(sB, mapB, fb, kb_coord, ti.nb0 + half_n, batch);
            else tma_load_2d_pair(sB, mapB, fb, kb_coord, ti.nb0 + half_n);
          } else {
            // chunked map (required for pairs): the CTA's BN/128 chunks, its half
            // of the tile (SwiGLU pair: the gate half in CTA 0, the up half in CTA 1)
            const int c0 =
                (p.swiglu_b ? (half_n == 0 ? ti.nb0 : p.f + ti.nb0) : ti.nb0 + half_n) >> 6;
            if (p.b_rank3) tma_load_4d_pair(sB, mapB, fb, 0, kb_coord, c0, batch);
            else if (p.ncat > 0 && c0 * 64 >= p.ncat)  // this half's columns are B2's
              tma_load_3d_pair(sB, mapB2, fb, 0, kb_coord, c0 - p.ncat / 64);
            else tma_load_3d_pair(sB, mapB, fb, 0, kb_coord, c0);
          }
        }
      } else {
        mbar_arrive_expect_tx(&full[stage], tx_bytes);
        if (p.kcat > 0 && k >= p.kcat) {
          // second K segment: [A | A2] @ [B ; B2] (both K-major, dense)
          tma_load_2d(sA, mapA2, &full[stage], k - p.kcat, ti.m0);
          tma_load_2d(sB, mapB2, &full[stage], k - p.kcat, ti.nb0);
        } else {
          // A
          if (gather_a) {
            // copied by the gather warps
          } else if (!p.a_mn) {
            tma_load_2d(sA, mapA, &full[stage], k, ti.m0);
          } else if (p.a_chunked) {
            tma_load_3d(sA, mapA, &full[stage], 0, k, ti.m0 >> 6);
          } else {
            tma_load_2d(sA, mapA, &full[stage], ti.m0, k);
            tma_load_2d(sA + CHUNK_BYTES, mapA, &full[stage], ti.m0 + 64, k);
          }
          // B
          if (gather_b) {
            // copied by the gather warps
          } else if (!p.b_mn) {
            if (p.b_rank3) tma_load_3d(sB, mapB, &full[stage], kb_coord, ti.nb0, batch);
            else tma_load_2d(sB, mapB, &full[stage], kb_coord, ti.nb0);
          } else if (p.b_chunked) {
            // one copy per run of consecutive chunks: the whole tile, or its gate
            // and up halves (columns nb0 and f + nb0) for the SwiGLU pair
            const int nruns = p.swiglu_b ? 2 : 1;
            for (int r = 0; r < nruns; ++r) {
              const int c0 = (r == 0 ? ti.nb0 : p.f + ti.nb0) >> 6;
              const uint32_t dst = sB + r * (BN / 2) * 128;
              if (p.b_rank3) tma_load_4d(dst, mapB, &full[stage], 0, kb_coord, c0, batch);
              else tma_load_3d(dst, mapB, &full[stage], 0, kb_coord, c0);
            }
          } else {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c) {
              int ncoord;
              if (p.swiglu_b) {
                ncoord = (c < BN / 128) ? ti.nb0 + 64 * c : p.f + ti.nb0 + 64 * (c - BN / 128);
              } else {
                ncoord = ti.nb0 + 64 * c;
              }
              if (p.b_rank3) {
                tma_load_3d(sB + c * CHUNK_BYTES, mapB, &full[stage], ncoord, kb_coord, batch);
              } else {
                tma_load_2d(sB + c * CHUNK_BYTES, mapB, &full[stage], ncoord, kb_coord);
              }
            }
          }
        }
      }
      ++issued;
      if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
    }
  }
  if (ok) {
    // Tail: wait until the MMA warp released every stage, so that no
    // tcgen05.commit arrival reaches this CTA's barriers after it exits.
    for (int i = 0; i < C::STAGES; ++i) {
      if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
        raise_abort(abort_flag, p.err_flag);
        break;
      }
      if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
    }
  } else if (!(PAIR && half_n != 0)) {
    // Wait (bounded, ignoring the abort flag) for the copies still in flight so
    // that none lands in shared memory after the CTA exits. (The second CTA of
    // a pair cannot see its copies complete: they count on the first CTA's
    // barriers, whose producer waits for them, and the pair leaves together.)
    int s = stage;
    uint32_t ph = phase;
    volatile int never = 0;
    for (long long i = 0; i < issued && i < C::STAGES; ++i) {
      if (--s < 0) { s = C::STAGES - 1; ph ^= 1u; }
      mbar_wait(&full[s], ph, &never);
    }
  }
}

// ------------------------------------------------------------------ gather warps
//
// A gathered operand's row i is row gather_idx[i] of an unpermuted source
// tensor [rows][gwidth] (row-major bf16, gld elements between rows). GW warps
// copy each stage's part of it with 16-byte cp.async copies straight into the
// 128-byte-swizzled layout the MMA reads, and each of their threads arrives on
// the stage's full barrier once its copies landed. A stage holds ROWS source
// rows of NCH 64-element chunks each:
//   grouped-M, K-major A: the tile's 128 rows x one 64-wide K block (NCH = 1);
//   grouped-K, MN-major A or B: 64 K rows x the tile's 128 (A) or BN (B)
//   columns, chunk c at c * CHUNK_BYTES (NCH = 2 or BN / 64).
// Rows past an expert's segment: grouped-M repeats its last row (those rows'
// results are never stored); grouped-K fills zeros. Chunks past the source
// width are zero-filled as well.
template <int GW, int NCH, int ROWS>
__device__ __forceinline__ void gather_stage(const Params& p, uint32_t dst_base, int gw, int lane,
                                             const int (&idx)[ROWS / GW / 32 > 0 ? ROWS / GW / 32 : 1],
                                             int row0_valid_end, int col0, uint64_t pol) {
  constexpr int PIECES = 8 * NCH;         // 16-byte pieces per row
  constexpr int RPI = 32 / PIECES;        // rows per warp instruction
  constexpr int RPW = ROWS / GW;          // rows per warp
  const int piece = lane % PIECES;
  const int sub = lane / PIECES;
  const int c = piece >> 3, q = piece & 7;
  const bool col_ok = col0 + 64 * c < p.gwidth;
  const char* src = reinterpret_cast<const char*>(p.gsrc);
#pragma unroll
  for (int i = 0; i < RPW / RPI; ++i) {
    const int ri = RPI * i + sub;               // row within this warp's rows
    const int r = gw * RPW + ri;                // row within the stage
    const int srow = __shfl_sync(0xFFFFFFFFu, idx[(RPI * i) >> 5], (RPI * i + sub) & 31);
    const bool ok = col_ok && r < row0_valid_end;
    // (a zero-filled piece reads nothing; its address still points into the source)
    const char* g = src + (static_cast<long long>(srow) * p.gld + (ok ? col0 + 8 * piece : 0)) * 2;
    const uint32_t d = dst_base + c * CHUNK_BYTES + r * 128 + ((q ^ (r & 7)) << 4);
    cp_async_16(d, g, ok ? 16u : 0u, pol);
  }
}

template <int BN, int EW, bool CW16, int GW, bool SBWD>
__device__ void gather_loop(const Params& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                            const int4* ttab, volatile int* abort_flag) {
  using C = Cfg<BN, EW, CW16, false, SBWD>;
  const int gw = (static_cast<int>(threadIdx.x) >> 5) - 2 - EW;
  const int lane = static_cast<int>(lane_id());
  const int total = total_tiles(p);
  const bool gm = p.sched == SCHED_GROUPED_M;
  // the gathered source (a few tens of MB, each row read by several experts'
  // tiles) stays in L2 while the weights and outputs stream past it
  const uint64_t pol = l2_policy_evict_last();
  // Source-row indices are fetched one step ahead: grouped-M, the next tile's
  // rows (this warp's 64 of its 128: lane j holds rows j and 32 + j) while the
  // current tile is copied; grouped-K, the next K block's 64 rows (this warp's
  // 32: lane j holds row j) while the current block is copied. Rows past a
  // segment repeat its last row (grouped-K zero-fills them in the copy).
  auto rows_m = [&](const Tile& ti, int (&out)[2]) {
    const int last = ti.m0 + ti.rows - 1;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      out[h] = __ldg(p.gather_idx + min(ti.m0 + gw * (BM / GW) + 32 * h + lane, last));
  };
  auto rows_k = [&](const Tile& ti, int kb) {
    const int last = ti.k0 + ti.krows - 1;
    return __ldg(p.gather_idx + min(ti.k0 + kb * BK + gw * (BK / GW) + lane, last));
  };
  int stage = 0;
  uint32_t phase = 0;
  int it = 0;
  int t = tile_begin<false>();
  Tile ti = tile_of<BN>(p, ttab, 0, t);
  int idx_m[2] = {0, 0}, nidx_m[2] = {0, 0};
  int idx_k[1] = {0};
  if (t < total) {
    if (gm) rows_m(ti, idx_m);
    else if (ti.nk > 0) idx_k[0] = rows_k(ti, 0);
  }
  bool ok = true;
  while (t < total && ok) {
    const int tn = t + tile_step<false>();
    Tile nt = ti;  // (unused when this is the last tile)
    if (tn < total) {
      nt = tile_of<BN>(p, ttab, it + 1, tn);
      if (gm) rows_m(nt, nidx_m);
    }
    for (int kb = 0; kb < ti.nk; ++kb) {
      int okw = 1;
      if (lane == 0) okw = mbar_wait(&empty[stage], phase ^ 1u, abort_flag) ? 1 : 0;
      okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
      if (!okw) {
        if (lane == 0) raise_abort(abort_flag, p.err_flag);
        ok = false;
        break;
      }
      const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
      if (gm) {
        // K-major A rows: the tile's 128 rows, K block kb (all rows copied)
        gather_stage<GW, 1, BM>(p, sA, gw, lane, idx_m, BM, ti.k0 + kb * BK, pol);
      } else {
        // grouped-K: this block's 64 K rows; the next block's (or the next
        // tile's first block's) indices are fetched before these copies issue
        int nk_idx = 0;
        if (kb + 1 < ti.nk) nk_idx = rows_k(ti, kb + 1);
        else if (tn < total && nt.nk > 0) nk_idx = rows_k(nt, 0);
        const int valid = ti.krows - kb * BK;
        if (p.gather_a)
          gather_stage<GW, BM / 64, BK>(p, sA, gw, lane, idx_k, valid, ti.m0, pol);
        else
          gather_stage<GW, BN / 64, BK>(p, sA + A_BYTES, gw, lane, idx_k, valid, ti.nb0, pol);
        idx_k[0] = nk_idx;
      }
      cp_async_arrive_noinc(&full[stage]);
      if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    if (!gm && ti.nk == 0 && tn < total && nt.nk > 0) idx_k[0] = rows_k(nt, 0);
    ti = nt;
    idx_m[0] = nidx_m[0];
    idx_m[1] = nidx_m[1];
    t = tn;
    ++it;
  }
  // nothing may land in shared memory after the CTA exits
  cp_async_wait_all();
}

// ------------------------------------------------------------------ MMA

template <int BN, int EW, bool CW16, int GW, bool SBWD>
__device__ void mma_loop(const Params& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                         uint64_t* tfull, uint64_t* tempty, uint64_t* drain, uint32_t tmem_base,
                         const int4* ttab, volatile int* abort_flag) {
  using C = Cfg<BN, EW, CW16, false, SBWD>;
  const uint32_t lane = lane_id();
  const uint32_t idesc128 = make_idesc_bf16(BM, BN, p.a_mn, p.b_mn);
  const uint32_t idesc64 = make_idesc_bf16(64, BN, p.a_mn, p.b_mn);
  const uint32_t a_lbo = p.a_mn ? CHUNK_BYTES : 16, b_lbo = p.b_mn ? CHUNK_BYTES : 16;
  const uint32_t a_kstep = p.a_mn ? 2048 : 32, b_kstep = p.b_mn ? 2048 : 32;
  int stage = 0;
  uint32_t phase = 0;
  bool issued_any = false;
  const int total = total_tiles(p);
  int it = 0;
  bool ok = true;
  for (int t = tile_begin<false>(); t < total && ok; t += tile_step<false>(), ++it) {
    const Tile ti = tile_of<BN>(p, ttab, it, t);
    const uint32_t idesc = quad_rows(p, ti.rows) == 16 ? idesc64 : idesc128;
    const int buf = it & 1;
    const uint32_t use = static_cast<uint32_t>(it >> 1);
    if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag)) {
      raise_abort(abort_flag, p.err_flag);
      break;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
    for (int kb = 0; kb < ti.nk; ++kb) {
      if (!mbar_wait(&full[stage], phase, abort_flag)) {
        raise_abort(abort_flag, p.err_flag);
        ok = false;
        break;
      }
      tc_fence_after();
      // rows the gather warps copied (generic proxy) are read by the MMA (async proxy)
      if constexpr (GW > 0) fence_proxy_async_smem();
      uint8_t* sA = smem + stage * C::STAGE_BYTES;
      int nkk = BK / 16;  // K=16 MMAs of this block
      if (p.sched == SCHED_GROUPED_K) {
        const int valid = ti.krows - kb * BK;
        if (valid < BK) {
          // Rows past this expert's segment belong to the next expert (or are
          // repeats of its last row, or zero fill past the tensor). The MMAs
          // wholly past the segment are skipped; in the last one the rows past
          // it are zeroed in A's two 64-wide chunks (rows are whole 128-byte
          // lines), so that they add 0 * (finite B row) = 0.
          nkk = (valid + 15) >> 4;
          const int nz = nkk * 16 - valid;
          if (nz > 0) {
            const int n16 = nz * 8;  // 16-byte pieces per chunk
            const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int c = 0; c < BM / 64; ++c) {
              uint8_t* base = sA + c * CHUNK_BYTES + valid * 128;
              for (int i = lane; i < n16; i += 32)
                *reinterpret_cast<uint4*>(base + (i >> 3) * 128 + (i & 7) * 16) = zero;
            }
            fence_proxy_async_smem();
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        const uint32_t a0 = smem_u32(sA), b0 = a0 + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          if (kk < nkk) {
            const uint64_t ad = make_sdesc(a0 + kk * a_kstep, a_lbo, 1024);
            const uint64_t bd = make_sdesc(b0 + kk * b_kstep, b_lbo, 1024);
            mma_bf16_ss(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
        }
        mma_commit(&empty[stage]);
      }
      issued_any = true;
      __syncwarp();
      if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    if (lane == 0) {
      if (ti.nk > 0) mma_commit(&tfull[buf]);
      else mbar_arrive(&tfull[buf]);
    }
    __syncwarp();
  }
  if (*abort_flag && issued_any) {
    // Let every issued MMA finish before tensor memory is released.
    if (lane == 0) mma_commit(drain);
    __syncwarp();
    volatile int never = 0;
    mbar_wait(drain, 0, &never);
  }
}

// CTA pair, first CTA: the MMA warp. A stage is full once both CTAs' copies
// landed (both count on this CTA's full barrier); the MMAs' completion frees
// the stage in both CTAs and, per tile, fills both CTAs' accumulators
// (multicast commits). The accumulator buffer is free once the epilogue warps
// of both CTAs released it (tempty, 2 * EW arrivals).
template <int BN, int EW, bool CW16, bool SBWD>
__device__ void mma_loop_pair(const Params& p, uint8_t* smem, uint64_t* full, uint64_t* empty, uint64_t* tfull, uint64_t* tempty, uint64_t* drain,
                              uint32_t tmem_base, volatile int* abort_flag) {
  using C = Cfg<BN, EW, CW16, true, SBWD>;
  const uint32_t lane = lane_id();
  const uint32_t idesc = make_idesc_bf16(2 * BM, BN, p.a_mn, p.b_mn);
  const uint32_t a_lbo = p.a_mn ? CHUNK_BYTES : 16, b_lbo = p.b_mn ? CHUNK_BYTES : 16;
  const uint32_t a_kstep = p.a_mn ? 2048 : 32, b_kstep = p.b_mn ? 2048 : 32;
  int stage = 0;
  uint32_t phase = 0;
  bool issued_any = false;
  const int total = total_tiles(p);
  int it = 0;
  bool ok = true;
  for (int t = tile_begin<true>(); t < total && ok; t += tile_step<true>(), ++it) {
    const Tile ti = decode<BN, true>(p, t);
    const int buf = it & 1;
    const uint32_t use = static_cast<uint32_t>(it >> 1);
    if (!mbar_wait<true>(&tempty[buf], (use & 1u) ^ 1u, abort_flag)) {
      raise_abort(abort_flag, p.err_flag);
      break;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
    for (int kb = 0; kb < ti.nk; ++kb) {
      if (!mbar_wait(&full[stage], phase, abort_flag)) {
        raise_abort(abort_flag, p.err_flag);
        ok = false;
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t a0 = smem_u32(smem + stage * C::STAGE_BYTES), b0 = a0 + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = make_sdesc(a0 + kk * a_kstep, a_lbo, 1024);
          const uint64_t bd = make_sdesc(b0 + kk * b_kstep, b_lbo, 1024);
          mma_bf16_ss_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
        }
        mma_commit_pair(&empty[stage], 0x3);
      }
      issued_any = true;
      __syncwarp();
      if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    if (lane == 0) mma_commit_pair(&tfull[buf], 0x3);  // nk > 0 on the dense schedule
    __syncwarp();
  }
  if (*abort_flag && issued_any) {
    // Let every issued MMA finish before tensor memory is released.
    if (lane == 0) mma_commit_pair(drain, 0x1);
    __syncwarp();
    volatile int never = 0;
    mbar_wait(drain, 0, &never);
  }
}

// ------------------------------------------------------------------ epilogue
//
// Each epilogue warp owns 32 accumulator rows (its TMEM lane quadrant) and
// walks the tile in 32-column chunks. Full 32x32 output blocks are written to
// the warp's swizzled staging area in shared memory and stored by one TMA
// tensor store per block (64-byte swizzle for bf16 rows, 128-byte for fp32);
// the staging area is reused once the previous chunk's stores have read it.
// TMA clips rows and columns outside the output tensor; the only blocks that
// take per-thread stores are the last, partial 32-row blocks of an expert
// segment (rows past it belong to the next expert) and read-modify-write
// accumulation.


__device__ __forceinline__ void store16(void* dst, uint4 v) { *reinterpret_cast<uint4*>(dst) = v; }

// Row `row` (= lane) of a 32x32 bf16 block: 64-byte rows, 64-byte TMA swizzle.
__device__ __forceinline__ void stage_bf16(uint8_t* blk, int row, const float* v) {
  uint8_t* rp = blk + row * 64;
  const int sw = (row >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(rp + ((c ^ sw) << 4)) =
        make_uint4(pack_bf16(v[8 * c], v[8 * c + 1]), pack_bf16(v[8 * c + 2], v[8 * c + 3]),
                   pack_bf16(v[8 * c + 4], v[8 * c + 5]), pack_bf16(v[8 * c + 6], v[8 * c + 7]));
}

// Row `row` of a 32x32 fp32 block: 128-byte rows, 128-byte TMA swizzle.
__device__ __forceinline__ void stage_f32(uint8_t* blk, int row, const float* v) {
  uint8_t* rp = blk + row * 128;
  const int sw = row & 7;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(rp + ((c ^ sw) << 4)) =
        make_uint4(__float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                   __float_as_uint(v[4 * c + 2]), __float_as_uint(v[4 * c + 3]));
}

// Row `row` of a 32x16 bf16 block: 32-byte rows, 32-byte TMA swizzle.
__device__ __forceinline__ void stage_bf16_16(uint8_t* blk, int row, const float* v) {
  uint8_t* rp = blk + row * 32;
  const int sw = (row >> 2) & 1;
#pragma unroll
  for (int c = 0; c < 2; ++c)
    *reinterpret_cast<uint4*>(rp + ((c ^ sw) << 4)) =
        make_uint4(pack_bf16(v[8 * c], v[8 * c + 1]), pack_bf16(v[8 * c + 2], v[8 * c + 3]),
                   pack_bf16(v[8 * c + 4], v[8 * c + 5]), pack_bf16(v[8 * c + 6], v[8 * c + 7]));
}

__device__ __forceinline__ void store_bf16_row16(bf16* dst, const float* v) {
#pragma unroll
  for (int c = 0; c < 2; ++c)
    store16(dst + 8 * c,
            make_uint4(pack_bf16(v[8 * c], v[8 * c + 1]), pack_bf16(v[8 * c + 2], v[8 * c + 3]),
                       pack_bf16(v[8 * c + 4], v[8 * c + 5]), pack_bf16(v[8 * c + 6], v[8 * c + 7])));
}

__device__ __forceinline__ void ld_chunk16(uint32_t taddr, float* v) {
  uint32_t r[16];
  tmem_ld_32x32b_x16(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void store_bf16_row(bf16* dst, const float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    store16(dst + 8 * c,
            make_uint4(pack_bf16(v[8 * c], v[8 * c + 1]), pack_bf16(v[8 * c + 2], v[8 * c + 3]),
                       pack_bf16(v[8 * c + 4], v[8 * c + 5]), pack_bf16(v[8 * c + 6], v[8 * c + 7])));
}

__device__ __forceinline__ void store_f32_row(float* dst, const float* v) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    store16(dst + 4 * c, make_uint4(__float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                                    __float_as_uint(v[4 * c + 2]), __float_as_uint(v[4 * c + 3])));
}

__device__ __forceinline__ void ld_chunk(uint32_t taddr, float* v) {
  uint32_t r[32];
  tmem_ld_32x32b_x32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

struct StoreMaps {
  const CUtensorMap* c0;  // C / h / dgu
  const CUtensorMap* c1;  // gu (SwiGLU) / w*h (SwiGLU backward)
  int c0_rank3;
  const CUtensorMap* ld_gu;  // SwiGLU backward: load maps of the saved g|u and h
  const CUtensorMap* ld_h;
};

// SwiGLU-backward element math for eight columns: dh = w * acc,
// dg = dh * u * s(g) * (1 + g (1 - s(g))), du = dh * silu(g), the routing-weight
// dot acc . h, and w * h (the dW2 operand); bf16 in and out, fp32 math.
__device__ __forceinline__ void swiglu_bwd8f(const float* a, const float* G, const float* U,
                                             uint4 H, float w, float& dot, uint4& DG, uint4& DU,
                                             uint4& HW) {
  const uint32_t Hw[4] = {H.x, H.y, H.z, H.w};
  uint32_t pdg[4], pdu[4], phw[4];
#pragma unroll
  for (int e2 = 0; e2 < 4; ++e2) {
    float dgv[2], duv[2], hwv[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float av = a[2 * e2 + hh];
      const float gg = G[2 * e2 + hh];
      const float uu = U[2 * e2 + hh];
      const float hv = hh ? bf16_hi(Hw[e2]) : bf16_lo(Hw[e2]);
      const float sg = sigmoidf_(gg);
      const float dh = w * av;
      dgv[hh] = dh * uu * sg * (1.0f + gg * (1.0f - sg));
      duv[hh] = dh * gg * sg;
      dot = fmaf(av, hv, dot);
      hwv[hh] = w * hv;
    }
    pdg[e2] = pack_bf16(dgv[0], dgv[1]);
    pdu[e2] = pack_bf16(duv[0], duv[1]);
    phw[e2] = pack_bf16(hwv[0], hwv[1]);
  }
  DG = make_uint4(pdg[0], pdg[1], pdg[2], pdg[3]);
  DU = make_uint4(pdu[0], pdu[1], pdu[2], pdu[3]);
  HW = make_uint4(phw[0], phw[1], phw[2], phw[3]);
}

// The same with g and u as bf16 (eight each, packed in pairs).
__device__ __forceinline__ void swiglu_bwd8(const float* a, uint4 G, uint4 U, uint4 H, float w,
                                            float& dot, uint4& DG, uint4& DU, uint4& HW) {
  const uint32_t Gw[4] = {G.x, G.y, G.z, G.w};
  const uint32_t Uw[4] = {U.x, U.y, U.z, U.w};
  float gf[8], uf[8];
#pragma unroll
  for (int e2 = 0; e2 < 4; ++e2) {
    gf[2 * e2] = bf16_lo(Gw[e2]);
    gf[2 * e2 + 1] = bf16_hi(Gw[e2]);
    uf[2 * e2] = bf16_lo(Uw[e2]);
    uf[2 * e2 + 1] = bf16_hi(Uw[e2]);
  }
  swiglu_bwd8f(a, gf, uf, H, w, dot, DG, DU, HW);
}

// SwiGLU-backward epilogue with TMA-staged inputs. Each of the 4 epilogue
// warps owns the 32 accumulator rows of its tensor-memory lane quadrant and a
// ring of 6 KB slots in shared memory (Cfg::SLOTS); a slot holds the g, u and h blocks
// (32 rows x 32 columns, bf16, 64-byte rows with 64-byte swizzle) of one
// 32-column chunk. Lane 0 loads them by TMA SLOTS - 1 chunks ahead of the chunk being
// computed (across tile boundaries too). The chunk's dg, du and w*h overwrite g,
// u and h in place and leave by TMA store from the same slot. With the FP8 cache
// the slot holds g and u as 32-byte rows of E4M3 (read by every lane before any
// writes its outputs) and the row scales come with the tile. (Loading the
// inputs lane by lane instead makes every load instruction touch 32 rows, so
// the L1's request rate, not DRAM, sets the pace.)
template <int BN, bool PAIR>
__device__ void epilogue_loop_sbwd(const Params& p, const StoreMaps& sm, uint8_t* staging,
                                   uint64_t* lbar, uint64_t* tfull, uint64_t* tempty,
                                   uint32_t tmem_base, const int4* ttab, volatile int* abort_flag) {
  using C = Cfg<BN, 4, false, PAIR, true>;
  constexpr int SLOT = 6144;
  constexpr int NS = C::SLOTS;  // ring depth; inputs are requested NS - 1 chunks ahead
  constexpr int NCH = BN / 32;
  const int warp = static_cast<int>(threadIdx.x) >> 5;
  const int q = warp & 3;
  const int ew = warp - 2;
  const uint32_t lane = lane_id();
  uint8_t* const slots = staging + ew * C::STG;
  uint64_t* const lb = lbar + NS * ew;
  const int total = total_tiles(p);
  const int sw = (static_cast<int>(lane) >> 1) & 3;  // 64-byte swizzle of this lane's row

  // The jobs (tile, chunk) this warp computes, in order, walked ahead of the
  // computation to request their inputs: tiles with rows in this warp's
  // quadrant, chunks inside N.
  int a_it = 0, a_t = tile_begin<PAIR>(), a_c = 0;
  Tile a_ti;
  bool a_have = false;
  auto a_seek = [&]() -> bool {
    while (a_t < total) {
      if (!a_have) {
        a_ti = tile_of<BN, PAIR>(p, ttab, a_it, a_t);
        a_have = true;
      }
      if (a_ti.rows - q * quad_rows(p, a_ti.rows) > 0 && a_c < NCH && a_ti.nb0 + 32 * a_c < p.N)
        return true;
      a_c = 0;
      a_t += tile_step<PAIR>();
      ++a_it;
      a_have = false;
    }
    return false;
  };
  long long issued = 0;  // jobs whose inputs were requested
  auto issue = [&]() {
    const int n = a_ti.nb0 + 32 * a_c;
    const int sx = n / p.f;
    const int gcol = sx * 2 * p.f + (n - sx * p.f);
    const int row0 = a_ti.m0 + q * quad_rows(p, a_ti.rows);
    const int slot = static_cast<int>(issued % NS);
    if (lane == 0) {
      const uint32_t d = smem_u32(slots + slot * SLOT);
      if (p.gu8) {
        // FP8 cache: 64-byte rows of the chunk's interleaved g and u bytes (16 g, 16 u,
        // 16 g, 16 u; byte column = gcol + the feature offset within the batch) at 0,
        // h at 4096
        mbar_arrive_expect_tx(&lb[slot], 2048 + 2048);
        tma_load_2d(d, sm.ld_gu, &lb[slot], gcol + (n - sx * p.f), row0);
      } else {
        mbar_arrive_expect_tx(&lb[slot], SLOT);
        tma_load_2d(d, sm.ld_gu, &lb[slot], gcol, row0);
        tma_load_2d(d + 2048, sm.ld_gu, &lb[slot], gcol + p.f, row0);
      }
      tma_load_2d(d + 4096, sm.ld_h, &lb[slot], n, row0);
    }
    ++issued;
    ++a_c;
  };
  for (int i = 0; i < NS - 1 && a_seek(); ++i) issue();

  long long done = 0;  // jobs computed
  bool ok = true;
  int it = 0;
  for (int t = tile_begin<PAIR>(); t < total && ok; t += tile_step<PAIR>(), ++it) {
    const Tile ti = tile_of<BN, PAIR>(p, ttab, it, t);
    const int buf = it & 1;
    const uint32_t use = static_cast<uint32_t>(it >> 1);
    // FP8 cache: the lane's row scales for the tile's 64-column blocks, requested
    // before the accumulator wait so that they arrive while it lasts
    static_assert(BN / 64 <= 4, "four scale blocks per tile at most");
    float4 sgq = make_float4(1.0f, 1.0f, 1.0f, 1.0f), suq = sgq;
    if (p.gu8) {
      const int qr0 = quad_rows(p, ti.rows);
      const int rl = q * qr0 + static_cast<int>(lane);
      const bool rok = static_cast<int>(lane) < qr0 && rl < ti.rows;
      const float* const sc =
          p.gu_scale + static_cast<long long>(ti.m0 + rl) * p.ld_scale + ti.nb0 / 64;
      auto ld = [&](int i, int off) {
        return (rok && ti.nb0 + 64 * i < p.N) ? __ldg(sc + off + i) : 1.0f;
      };
      const int uo = p.ld_scale / 2;
      sgq.x = ld(0, 0);
      suq.x = ld(0, uo);
      sgq.y = ld(1, 0);
      suq.y = ld(1, uo);
      if (BN / 64 > 2) {
        sgq.z = ld(2, 0);
        suq.z = ld(2, uo);
        sgq.w = ld(3, 0);
        suq.w = ld(3, uo);
      }
    }
    if (!mbar_wait<PAIR>(&tfull[buf], use & 1u, abort_flag)) {
      raise_abort(abort_flag, p.err_flag);
      break;
    }
    tc_fence_after();
    const int qr = quad_rows(p, ti.rows);
    const int blk_rows = ti.rows - q * qr;
    const int r_loc = q * qr + static_cast<int>(lane);
    const bool row_ok = static_cast<int>(lane) < qr && r_loc < ti.rows;
    const long long grow = static_cast<long long>(ti.m0) + r_loc;
    const int row0 = ti.m0 + q * qr;
    const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(buf * BN);
    // TMA clips outside the tensor; inside it (grouped-M) only full 32-row blocks may use it
    const bool use_tma = qr == 32 && (blk_rows >= 32 || p.sched != SCHED_GROUPED_M);
    if (blk_rows > 0) {
      const float w = (row_ok && p.row_w) ? __ldg(p.row_w + grow) : 1.0f;
      float dot = 0.0f;
      for (int c = 0; c < NCH; ++c) {
        const int n = ti.nb0 + c * 32;
        if (n >= p.N) break;
        const int slot = static_cast<int>(done % NS);
        int okw = 1;
        if (lane == 0)
          okw = mbar_wait(&lb[slot], static_cast<uint32_t>((done / NS) & 1), abort_flag) ? 1 : 0;
        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
        if (!okw) {
          if (lane == 0) raise_abort(abort_flag, p.err_flag);
          ok = false;
          break;
        }
        float a[32];
        ld_chunk(trow + c * 32, a);
        const int sx = n / p.f;
        const int gcol = sx * 2 * p.f + (n - sx * p.f);
        uint8_t* const sl = slots + slot * SLOT;
        uint8_t* const rowp = sl + lane * 64;
        bf16* dgdst = reinterpret_cast<bf16*>(p.C) + grow * p.ldc + gcol;
        // FP8 cache: the lane's 32 g and 32 u bytes (one 64-byte row, 64-byte
        // swizzle: 16-byte pieces g, u, g, u) are read before any lane writes its
        // outputs over them; block scales per row
        uint32_t g8[8], u8[8];
        float sgl = 1.0f, sul = 1.0f;
        if (p.gu8) {
          const uint8_t* const rp8 = sl + lane * 64;
          const uint4 g0 = *reinterpret_cast<const uint4*>(rp8 + ((0 ^ sw) << 4));
          const uint4 u0 = *reinterpret_cast<const uint4*>(rp8 + ((1 ^ sw) << 4));
          const uint4 g1 = *reinterpret_cast<const uint4*>(rp8 + ((2 ^ sw) << 4));
          const uint4 u1 = *reinterpret_cast<const uint4*>(rp8 + ((3 ^ sw) << 4));
          g8[0] = g0.x; g8[1] = g0.y; g8[2] = g0.z; g8[3] = g0.w;
          g8[4] = g1.x; g8[5] = g1.y; g8[6] = g1.z; g8[7] = g1.w;
          u8[0] = u0.x; u8[1] = u0.y; u8[2] = u0.z; u8[3] = u0.w;
          u8[4] = u1.x; u8[5] = u1.y; u8[6] = u1.z; u8[7] = u1.w;
          const int bi = c >> 1;  // the chunk's 64-column block within the tile
          sgl = bi == 0 ? sgq.x : bi == 1 ? sgq.y : bi == 2 ? sgq.z : sgq.w;
          sul = bi == 0 ? suq.x : bi == 1 ? suq.y : bi == 2 ? suq.z : suq.w;
          __syncwarp();
        }
#pragma unroll
        for (int vv = 0; vv < 4; ++vv) {
          const int off = (vv ^ sw) << 4;
          uint4 DG, DU, HW;
          if (p.gu8) {
            float gf[8], uf[8];
            e4m3x4_to_f32(g8[2 * vv], gf);
            e4m3x4_to_f32(g8[2 * vv + 1], gf + 4);
            e4m3x4_to_f32(u8[2 * vv], uf);
            e4m3x4_to_f32(u8[2 * vv + 1], uf + 4);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              gf[i] *= sgl;
              uf[i] *= sul;
            }
            swiglu_bwd8f(a + 8 * vv, gf, uf, *reinterpret_cast<const uint4*>(rowp + 4096 + off),
                         w, dot, DG, DU, HW);
          } else {
            swiglu_bwd8(a + 8 * vv, *reinterpret_cast<const uint4*>(rowp + off),
                        *reinterpret_cast<const uint4*>(rowp + 2048 + off),
                        *reinterpret_cast<const uint4*>(rowp + 4096 + off), w, dot, DG, DU, HW);
          }
          if (use_tma) {
            *reinterpret_cast<uint4*>(rowp + off) = DG;
            *reinterpret_cast<uint4*>(rowp + 2048 + off) = DU;
            *reinterpret_cast<uint4*>(rowp + 4096 + off) = HW;
          } else if (row_ok) {
            store16(dgdst + vv * 8, DG);
            store16(dgdst + p.f + vv * 8, DU);
            if (p.aux) store16(p.aux + grow * p.ldaux + n + vv * 8, HW);
          }
        }
        if (use_tma) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const uint32_t src = smem_u32(sl);
            tma_store_2d(sm.c0, src, gcol, row0);
            tma_store_2d(sm.c0, src + 2048, gcol + p.f, row0);
            if (p.aux) tma_store_2d(sm.c1, src + 4096, n, row0);
            bulk_commit();
          }
        }
        ++done;
        // the next request reuses the slot of the job before this one: its
        // stores (committed before this job's) must have read it
        if (a_seek()) {
          __syncwarp();
          if (lane == 0) bulk_wait_read_max(use_tma ? 1 : 0);
          __syncwarp();
          issue();
        }
      }
      if (ok && row_ok && p.dw_part) p.dw_part[grow * p.dw_nparts + ti.n_blk] = dot;
    }
    tc_fence_before();
    if (PAIR) {
      // one arrival per warp on the pair's first CTA (it issues the MMAs)
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_map(smem_u32(&tempty[buf]), 0));
    } else {
      mbar_arrive(&tempty[buf]);
    }
  }
  // inputs requested but never computed (after an abort) land before the CTA exits
  if (lane == 0) {
    volatile int never = 0;
    for (long long j = done; j < issued; ++j)
      mbar_wait(&lb[j % NS], static_cast<uint32_t>((j / NS) & 1), &never);
    bulk_wait_all();
  }
  __syncwarp();
}

template <int BN, int EW, bool CW16, bool PAIR>
__device__ void epilogue_loop(const Params& p, const StoreMaps& sm, uint8_t* staging,
                              uint64_t* tfull, uint64_t* tempty, uint32_t tmem_base,
                              const int4* ttab, volatile int* abort_flag) {
  constexpr int NG = EW / 4;  // warps per TMEM lane quadrant; they split the column chunks
  const int warp = threadIdx.x >> 5;
  const int q = warp & 3;  // tensor-memory lane quadrant this warp may read
  const int grp = (warp - 2) / 4;
  const uint32_t lane = lane_id();
  uint8_t* const stg0 = staging + (warp - 2) * Cfg<BN, EW, CW16, PAIR>::STG;
  // slot of one chunk (1 KB multiples keep every swizzle span aligned)
  int slot_bytes;
  if (p.epi == EPI_STORE) slot_bytes = (p.c_bf16 && (p.ncat == 0 || p.c2_bf16)) ? 2048 : 4096;
  else if (p.epi == EPI_ROWSCALE) slot_bytes = 2048;
  else if (p.gu8) slot_bytes = 2048;  // EPI_SWIGLU, FP8 cache: h, g and u of 16 columns
  else slot_bytes = (CW16 ? 1024 : 2048) * (p.gu ? 3 : 1);  // EPI_SWIGLU
  int nslots = Cfg<BN, EW, CW16, PAIR>::STG / slot_bytes;
  if (nslots > 4) nslots = 4;
  int slot = 0;
  uint8_t* stg = stg0;  // the current chunk's slot (set by stage_begin)
  uint32_t stg_s = smem_u32(stg0);
  const int total = total_tiles(p);
  bool pending = false;  // a bulk store of this warp may still read a slot
  auto stage_begin = [&]() {
    stg = stg0 + slot * slot_bytes;
    stg_s = smem_u32(stg);
    if (++slot == nslots) slot = 0;
    if (pending) {
      // the store that last used this slot was committed nslots groups ago
      if (lane == 0) bulk_wait_read_max(nslots - 1);
      __syncwarp();
    }
  };
  auto stage_end = [&]() {
    fence_proxy_async_smem();
    __syncwarp();
  };
  int it = 0;
  for (int t = tile_begin<PAIR>(); t < total; t += tile_step<PAIR>(), ++it) {
    const Tile ti = tile_of<BN, PAIR>(p, ttab, it, t);
    const int buf = it & 1;
    const uint32_t use = static_cast<uint32_t>(it >> 1);
    if (!mbar_wait<PAIR>(&tfull[buf], use & 1u, abort_flag)) {
      raise_abort(abort_flag, p.err_flag);
      break;
    }
    tc_fence_after();
    const int qr = quad_rows(p, ti.rows);  // accumulator rows in this warp's quadrant
    const int r_loc = q * qr + static_cast<int>(lane);
    const int blk_rows = ti.rows - q * qr;  // valid rows of this warp's block
    const bool row_ok = static_cast<int>(lane) < qr && r_loc < ti.rows;
    const long long grow = static_cast<long long>(ti.m0) + r_loc;
    const int row0 = ti.m0 + q * qr;
    const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(buf * BN);
    const bool has_acc = ti.nk > 0;
    // TMA clips outside the tensor; inside it (grouped-M) only full 32-row blocks may use it.
    const bool use_tma = qr == 32 && (blk_rows >= 32 || p.sched != SCHED_GROUPED_M);

    if (blk_rows > 0) {
      if (p.epi == EPI_STORE && p.ncat > 0) {
        // N-concatenated outputs (dense CTA pairs; TMA stores, which clip the rows
        // past M): columns below ncat go to C, the others to C2 at n - ncat. A loop
        // of its own keeps the plain stores' loop below as it is.
#pragma unroll 1
        for (int c = grp; c < BN / 32; c += NG) {
          const int n = ti.nb0 + c * 32;
          if (n >= p.N) break;
          float v[32];
          ld_chunk(trow + c * 32, v);
          const bool second = n >= p.ncat;
          stage_begin();
          if (second ? p.c2_bf16 : p.c_bf16) stage_bf16(stg, lane, v); else stage_f32(stg, lane, v);
          stage_end();
          if (lane == 0) {
            if (second) tma_store_2d(sm.c1, stg_s, n - p.ncat, row0);
            else tma_store_2d(sm.c0, stg_s, n, row0);
            bulk_commit();
          }
          pending = true;
        }
      } else if (p.epi == EPI_STORE) {
#pragma unroll 1
        for (int c = grp; c < BN / 32; c += NG) {
          const int n = ti.nb0 + c * 32;
          if (n >= p.N) break;  // warp-uniform N tail
          float v[32];
          if (has_acc) {
            ld_chunk(trow + c * 32, v);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
          }
          int ncol = n, cb = 0;
          if (p.sched == SCHED_GROUPED_K || p.splitk > 1) {
            cb = ti.g;  // expert (grouped-K) or K slice (split-K partials)
          } else if (p.c_batch_n > 0) {
            cb = n / p.c_batch_n;
            ncol = n - cb * p.c_batch_n;
          }
          if (use_tma && !p.accumulate) {
            stage_begin();
            if (p.c_bf16) stage_bf16(stg, lane, v); else stage_f32(stg, lane, v);
            stage_end();
            if (lane == 0) {
              // weight gradients (grouped-K) are not read again in the step
              if (p.sched == SCHED_GROUPED_K)
                tma_store_3d_hint(sm.c0, stg_s, ncol, row0, cb, l2_policy_evict_first());
              else if (sm.c0_rank3) tma_store_3d(sm.c0, stg_s, ncol, row0, cb);
              else tma_store_2d(sm.c0, stg_s, ncol, row0);
              bulk_commit();
            }
            pending = true;
          } else if (row_ok) {
            const long long off = static_cast<long long>(cb) * p.c_batch_stride + grow * p.ldc + ncol;
            if (p.c_bf16) {
              bf16* dst = reinterpret_cast<bf16*>(p.C) + off;
              if (p.accumulate) {
#pragma unroll
                for (int vv = 0; vv < 4; ++vv) {
                  const uint4 old = *reinterpret_cast<const uint4*>(dst + vv * 8);
                  const uint32_t o[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    v[vv * 8 + 2 * e] += bf16_lo(o[e]);
                    v[vv * 8 + 2 * e + 1] += bf16_hi(o[e]);
                  }
                }
              }
              store_bf16_row(dst, v);
            } else {
              store_f32_row(reinterpret_cast<float*>(p.C) + off, v);
            }
          }
        }
      } else if (p.epi == EPI_SWIGLU) {
        if constexpr (CW16) {
        // TMEM columns [0, BN/2) hold the gate, [BN/2, BN) the up projection;
        // 16-column chunks, the two warps of a lane quadrant taking turns.
        const int out_batch = (p.b_batch_mode == BATCH_FROM_N) ? ti.batch : 0;
        // FP8 cache: each warp takes a contiguous half of the tile's features
        // (a 64-feature block of g and one of u per row) so that it alone sees
        // the block's largest |g| and |u|; one scale per row and block.
        const int c_lo = p.gu8 ? grp * (BN / 32 / NG) : grp;
        const int c_hi = p.gu8 ? c_lo + BN / 32 / NG : BN / 32;
        const int c_step = p.gu8 ? 1 : NG;
        float inv_g = 1.0f, inv_u = 1.0f;
        if (p.gu8) {
          float ag = 0.0f, au = 0.0f;
#pragma unroll 1
          for (int c = c_lo; c < c_hi; ++c) {
            float g[16], u[16];
            ld_chunk16(trow + c * 16, g);
            ld_chunk16(trow + BN / 2 + c * 16, u);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              ag = fmaxf(ag, fabsf(g[i]));
              au = fmaxf(au, fabsf(u[i]));
            }
          }
          float sg, su;
          fp8_block_scale(ag, sg, inv_g);
          fp8_block_scale(au, su, inv_u);
          if (row_ok) {
            float* const sc = p.gu_scale + grow * p.ld_scale + (ti.nb0 + c_lo * 16) / 64;
            sc[0] = sg;
            sc[p.ld_scale / 2] = su;
          }
        }
#pragma unroll 1
        for (int c = c_lo; c < c_hi; c += c_step) {
          float g[16], u[16], hv[16];
          ld_chunk16(trow + c * 16, g);
          ld_chunk16(trow + BN / 2 + c * 16, u);
#pragma unroll
          for (int i = 0; i < 16; ++i) hv[i] = g[i] * sigmoidf_(g[i]) * u[i];
          const int j = ti.nb0 + c * 16;
          const int hcol = out_batch * p.f + j;
          const int gcol = out_batch * 2 * p.f + j;
          if (use_tma) {
            stage_begin();
            stage_bf16_16(stg, lane, hv);
            if (p.gu8) {
              // one 32-byte row per lane: the 16 g bytes, then the 16 u bytes (32-byte swizzle)
              const int sw = (static_cast<int>(lane) >> 2) & 1;
              uint8_t* const rp = stg + 1024 + lane * 32;
              *reinterpret_cast<uint4*>(rp + (sw << 4)) = f32x16_to_e4m3(g, inv_g);
              *reinterpret_cast<uint4*>(rp + ((1 ^ sw) << 4)) = f32x16_to_e4m3(u, inv_u);
            } else if (p.gu) {
              stage_bf16_16(stg + 1024, lane, g);
              stage_bf16_16(stg + 2048, lane, u);
            }
            stage_end();
            if (lane == 0) {
              tma_store_2d(sm.c0, stg_s, hcol, row0);
              // the g|u cache is read by the backward only
              const uint64_t pol = l2_policy_evict_first();
              if (p.gu8) {
                // byte column of feature j: 32 bytes per 16 features (g, then u)
                tma_store_2d_hint(sm.c1, stg_s + 1024, gcol + j, row0, pol);
              } else if (p.gu) {
                tma_store_2d_hint(sm.c1, stg_s + 1024, gcol, row0, pol);
                tma_store_2d_hint(sm.c1, stg_s + 2048, gcol + p.f, row0, pol);
              }
              bulk_commit();
            }
            pending = true;
          } else if (row_ok) {
            store_bf16_row16(p.h + grow * p.ldh + hcol, hv);
            if (p.gu8) {
              store16(p.gu8 + grow * p.ldgu + gcol + j, f32x16_to_e4m3(g, inv_g));
              store16(p.gu8 + grow * p.ldgu + gcol + j + 16, f32x16_to_e4m3(u, inv_u));
            } else if (p.gu) {
              store_bf16_row16(p.gu + grow * p.ldgu + gcol, g);
              store_bf16_row16(p.gu + grow * p.ldgu + gcol + p.f, u);
            }
          }
        }
        } else {
        // TMEM columns [0, BN/2) hold the gate, [BN/2, BN) the up projection.
        const int out_batch = (p.b_batch_mode == BATCH_FROM_N) ? ti.batch : 0;
#pragma unroll 1
        for (int c = grp; c < BN / 64; c += NG) {
          float g[32], u[32], hv[32];
          ld_chunk(trow + c * 32, g);
          ld_chunk(trow + BN / 2 + c * 32, u);
#pragma unroll
          for (int i = 0; i < 32; ++i) hv[i] = g[i] * sigmoidf_(g[i]) * u[i];
          const int j = ti.nb0 + c * 32;
          const int hcol = out_batch * p.f + j;
          const int gcol = out_batch * 2 * p.f + j;
          if (use_tma) {
            stage_begin();
            stage_bf16(stg, lane, hv);
            if (p.gu) {
              stage_bf16(stg + 2048, lane, g);
              stage_bf16(stg + 4096, lane, u);
            }
            stage_end();
            if (lane == 0) {
              tma_store_2d(sm.c0, stg_s, hcol, row0);
              if (p.gu) {  // the g|u cache is read by the backward only
                const uint64_t pol = l2_policy_evict_first();
                tma_store_2d_hint(sm.c1, stg_s + 2048, gcol, row0, pol);
                tma_store_2d_hint(sm.c1, stg_s + 4096, gcol + p.f, row0, pol);
              }
              bulk_commit();
            }
            pending = true;
          } else if (row_ok) {
            store_bf16_row(p.h + grow * p.ldh + hcol, hv);
            if (p.gu) {
              store_bf16_row(p.gu + grow * p.ldgu + gcol, g);
              store_bf16_row(p.gu + grow * p.ldgu + gcol + p.f, u);
            }
          }
        }
        }
      } else if (p.epi == EPI_ROWSCALE) {
        const float w = (row_ok && p.row_w) ? __ldg(p.row_w + grow) : 1.0f;
#pragma unroll 1
        for (int c = grp; c < BN / 32; c += NG) {
          const int n = ti.nb0 + c * 32;
          if (n >= p.N) break;
          float v[32];
          ld_chunk(trow + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= w;
          if (use_tma) {
            stage_begin();
            stage_bf16(stg, lane, v);
            stage_end();
            if (lane == 0) {
              tma_store_2d(sm.c0, stg_s, n, row0);
              bulk_commit();
            }
            pending = true;
          } else if (row_ok) {
            store_bf16_row(reinterpret_cast<bf16*>(p.C) + grow * p.ldc + n, v);
          }
        }
      }
    }
    tc_fence_before();
    if (PAIR) {
      // one arrival per warp on the pair's first CTA (it issues the MMAs)
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_map(smem_u32(&tempty[buf]), 0));
    } else {
      mbar_arrive(&tempty[buf]);
    }
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

template <int BN, int EW, bool CW16, bool PAIR, int GW, bool SBWD>
__global__ void __launch_bounds__(64 + 32 * (EW + GW), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA,
                   const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapC0,
                   const __grid_constant__ CUtensorMap mapC1,
                   const __grid_constant__ CUtensorMap mapA2,
                   const __grid_constant__ CUtensorMap mapB2, const Params p) {
  using C = Cfg<BN, EW, CW16, PAIR, SBWD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* staging = smem + C::STAGES * C::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + EW * C::STG);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // SwiGLU-backward epilogue: three input-slot barriers per epilogue warp
  uint64_t* lbar = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(full) + 256);
  int4* ttab = reinterpret_cast<int4*>(reinterpret_cast<uint8_t*>(full) + MISC_BYTES);
  const int warp = threadIdx.x >> 5;
  if (p.sched != SCHED_DENSE && warp >= 2 && warp < 2 + EW) {
    // the epilogue warps decode this CTA's first TT_CAP tiles in parallel
    const int total = total_tiles(p);
    const int mine = total > static_cast<int>(blockIdx.x)
                         ? (total - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x
                         : 0;
    const int n = mine < p.tt_cap ? mine : p.tt_cap;
    for (int i = threadIdx.x - 64; i < n; i += 32 * EW)
      ttab[i] = pack_tile<BN>(p, decode<BN>(p, blockIdx.x + i * gridDim.x));
  }

  if (threadIdx.x == 0) {
    // a stage is full once the producer posted its TMA bytes (one arrival) and,
    // in gathering launches, every gather thread's copies landed
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1 + 32 * GW);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], PAIR ? 2 * EW : 32 * EW);  // pairs: one arrival per warp of both CTAs
    }
    mbar_init(drain, 1);
    if (SBWD)
      for (int i = 0; i < C::SLOTS * EW; ++i) mbar_init(&lbar[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (PAIR) cluster_sync_all();  // the other CTA's barriers are initialised too
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane_id() == 0)
      producer_loop<BN, EW, CW16, PAIR, GW, SBWD>(p, &mapA, &mapB, &mapA2, &mapB2, smem, full, empty,
                                            ttab, abort_flag);
  } else if (warp == 1) {
    if constexpr (!PAIR) {
      mma_loop<BN, EW, CW16, GW, SBWD>(p, smem, full, empty, tfull, tempty, drain, tmem_base, ttab,
                                 abort_flag);
    } else {
      if (cluster_ctarank() == 0)  // the second CTA's MMA warp has nothing to do
        mma_loop_pair<BN, EW, CW16, SBWD>(p, smem, full, empty, tfull, tempty, drain, tmem_base,
                                    abort_flag);
    }
  } else if (warp < 2 + EW) {
    const StoreMaps sm{&mapC0, &mapC1, p.c0_rank3, &mapA2, &mapB2};
    if constexpr (SBWD)
      epilogue_loop_sbwd<BN, PAIR>(p, sm, staging, lbar, tfull, tempty, tmem_base, ttab,
                                   abort_flag);
    else
      epilogue_loop<BN, EW, CW16, PAIR>(p, sm, staging, tfull, tempty, tmem_base, ttab,
                                        abort_flag);
  } else {
    if constexpr (GW > 0 && !PAIR) gather_loop<BN, EW, CW16, GW, SBWD>(p, smem, full, empty, ttab,
                                                                 abort_flag);
  }
  tc_fence_before();
  if (PAIR) cluster_sync_all();  // no CTA frees tensor memory the pair's MMAs may still use
  else __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, []() {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// Tensor map over a bf16 [batch][rows][cols] view with box {64, box_rows(, 1)}.
bool make_map(CUtensorMap* map, const MatView& v, int box_rows, bool force3d) {
  const bool rank3 = force3d || v.batch > 1;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(v.cols), static_cast<cuuint64_t>(v.rows),
                        static_cast<cuuint64_t>(v.batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(v.ld) * 2,
                           static_cast<cuuint64_t>(v.batch_stride) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank3 ? 3 : 2,
                        const_cast<void*>(v.ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Chunked map of an MN-major bf16 operand [batch][rows][cols] (cols a multiple
// of 64): dimensions {64, rows, cols/64 (, batch)}, box {64, 64, nchunks (, 1)}.
// One copy lands `nchunks` 64-column blocks at 8 KB strides in shared memory,
// the layout that `nchunks` separate {64, 64} boxes of the plain map give.
bool make_map_chunked(CUtensorMap* map, const MatView& v, int nchunks, bool force4d) {
  if (v.cols % 64 != 0) return false;
  const bool rank4 = force4d || v.batch > 1;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(v.rows), static_cast<cuuint64_t>(v.cols / 64),
                        static_cast<cuuint64_t>(v.batch)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(v.ld) * 2, 128,
                           static_cast<cuuint64_t>(v.batch_stride) * 2};
  cuuint32_t box[4] = {64, 64, static_cast<cuuint32_t>(nchunks), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank4 ? 4 : 3,
                        const_cast<void*>(v.ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map of an output tensor [d2][d1][d0] (d0 contiguous) for 32x32-element
// TMA stores: bf16 rows of 64 bytes with 64-byte swizzle, fp32 rows of 128 bytes
// with 128-byte swizzle (the layouts stage_bf16 / stage_f32 write).
bool make_store_map(CUtensorMap* map, void* ptr, bool f32, bool rank3, long long d0, long long d1,
                    long long d2, long long ld, long long batch_stride, int box_cols = 32) {
  const long long es = f32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d0), static_cast<cuuint64_t>(d1),
                        static_cast<cuuint64_t>(d2)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * es),
                           static_cast<cuuint64_t>(batch_stride * es)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  // the swizzle span equals the staged row: 128 B (fp32 x 32), 64 B (bf16 x 32), 32 B (bf16 x 16)
  const long long row_bytes = box_cols * es;
  const CUtensorMapSwizzle sw = row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = g_encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        rank3 ? 3 : 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map of a byte matrix [d1][d0] (ld bytes between rows) for 32-row boxes
// of box_cols bytes (32 or 64), swizzled over the box's row width: the FP8
// cache's blocks (rows of interleaved 16-byte g and u groups).
bool make_u8_map(CUtensorMap* map, void* ptr, long long d0, long long d1, long long ld,
                 int box_cols) {
  if (box_cols != 32 && box_cols != 64) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d0), static_cast<cuuint64_t>(d1)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int EW, bool CW16, bool PAIR, int GW = 0, bool SBWD = false>
int launch_bn(const GemmLaunch& L, cudaStream_t stream) {
  using C = Cfg<BN, EW, CW16, PAIR, SBWD>;
  if (SBWD != (L.epi == EPI_SWIGLU_BWD)) return MOE_ERR_UNSUPPORTED;
  constexpr int THREADS = C::THREADS + 32 * GW;
  Params p{};
  p.tt_cap = C::TT_CAP;
  p.m64 = (L.m64 && L.sched == SCHED_GROUPED_M) ? 1 : 0;
  p.pair = PAIR ? 1 : 0;
  p.sched = L.sched;
  p.M = L.M;
  p.N = L.N;
  p.K = L.K;
  p.G = L.G;
  p.offsets = L.offsets;
  p.tile_sched = L.tile_sched;
  p.expert_order = L.expert_order;
  p.a_mn = L.a_mn;
  p.b_mn = L.b_mn;
  const bool b3 = L.b_batch_mode != BATCH_NONE || L.B.batch > 1;
  p.b_rank3 = b3 ? 1 : 0;
  p.b_batch_mode = L.b_batch_mode;
  p.n_tiles_per_batch = L.n_tiles_per_batch;
  p.k_per_batch = L.k_per_batch;
  p.swiglu_b = L.swiglu_b;
  p.f = L.f;
  const int bn_eff = L.swiglu_b ? BN / 2 : BN;
  p.nt = L.n_tiles > 0 ? L.n_tiles : (L.N + bn_eff - 1) / bn_eff;
  p.mt = (L.M + BM - 1) / BM;
  long long upper;
  if (L.sched == SCHED_DENSE) {
    p.splitk = L.splitk > 1 ? L.splitk : 1;
    p.kslice = ((L.K + p.splitk - 1) / p.splitk + BK - 1) / BK * BK;
    p.splitk = (L.K + p.kslice - 1) / p.kslice;
    p.mt2 = (p.mt + 1) / 2;
    p.total_static = (PAIR ? p.mt2 : p.mt) * p.nt * p.splitk;
    upper = p.total_static;
  } else if (L.sched == SCHED_GROUPED_K) {
    p.total_static = L.G * p.mt * p.nt;
    upper = p.total_static;
  } else {
    p.mt = 0;
    p.total_static = 0;
    upper = (static_cast<long long>(L.R_cap + BM - 1) / BM + L.G) * p.nt;
  }
  p.epi = L.epi;
  p.C = L.C;
  p.ldc = L.ldc;
  p.c_batch_stride = L.c_batch_stride;
  p.c_batch_n = L.c_batch_n;
  p.c_bf16 = L.c_bf16;
  p.accumulate = L.accumulate;
  p.row_w = L.row_w;
  p.gu = reinterpret_cast<bf16*>(L.gu);
  p.ldgu = L.ldgu;
  p.gu8 = static_cast<uint8_t*>(L.gu8);
  p.gu_scale = L.gu_scale;
  p.ld_scale = L.ld_scale;
  if (L.gu8) {
    // one scale per 64 features: a forward epilogue warp holds 64 of a 256-wide tile's
    if (!L.gu_scale || L.ld_scale <= 0 || L.gu ||
        (L.epi == EPI_SWIGLU && !(BN == 256 && EW == 8 && CW16)) ||
        (L.epi != EPI_SWIGLU && L.epi != EPI_SWIGLU_BWD))
      return MOE_ERR_UNSUPPORTED;
  }
  p.h = reinterpret_cast<bf16*>(L.h);
  p.ldh = L.ldh;
  p.aux = reinterpret_cast<bf16*>(L.aux);
  p.ldaux = L.ldaux;
  p.dw_part = L.dw_part;
  p.dw_nparts = L.dw_nparts;
  p.err_flag = L.err_flag;
  p.gather_idx = L.gather_idx;
  p.gather_a = L.gather_a;
  p.gather_b = L.gather_b;
  if ((L.gather_a || L.gather_b) != (GW > 0)) return MOE_ERR_UNSUPPORTED;
  if (L.gather_a || L.gather_b) {
    const MatView& g = L.gather_a ? L.A : L.B;
    p.gsrc = reinterpret_cast<const bf16*>(g.ptr);
    p.gld = g.ld;
    p.gwidth = static_cast<int>(g.cols);
  }
  if (L.gather_a || L.gather_b) {
    // supported: K-major A of a grouped-M GEMM, MN-major A or B of a grouped-K GEMM
    const bool okm = L.sched == SCHED_GROUPED_M && L.gather_a && !L.gather_b && !L.a_mn;
    const bool okk = L.sched == SCHED_GROUPED_K && (L.gather_a ? L.a_mn : 1) &&
                     (L.gather_b ? L.b_mn : 1) && !(L.gather_a && L.gather_b);
    if (!L.gather_idx || !(okm || okk) || (L.gather_b && (b3 || L.swiglu_b)))
      return MOE_ERR_UNSUPPORTED;
  }
  if (upper <= 0) return MOE_OK;

  if (!get_encoder()) return MOE_ERR_CUDA;
  CUtensorMap mapA, mapB, mapC0, mapC1, mapA2, mapB2;
  memset(&mapC0, 0, sizeof(mapC0));
  memset(&mapC1, 0, sizeof(mapC1));
  memset(&mapA2, 0, sizeof(mapA2));
  memset(&mapB2, 0, sizeof(mapB2));
  p.kcat = 0;
  if (L.kcat > 0) {
    // K-concatenated second operand pair: dense, both K-major, segment boundary on a K block
    if (L.sched != SCHED_DENSE || L.a_mn || L.b_mn || L.b_batch_mode != BATCH_NONE ||
        L.kcat % BK != 0 || L.splitk > 1 || L.gather_a || L.gather_b)
      return MOE_ERR_UNSUPPORTED;
    if (!make_map(&mapA2, L.A2, BM, false) || !make_map(&mapB2, L.B2, PAIR ? BN / 2 : BN, false))
      return MOE_ERR_ARG;
    p.kcat = L.kcat;
  }
  p.ncat = 0;
  p.c2_bf16 = L.c2_bf16;
  if (L.ncat > 0) {
    // N-concatenated second operand: dense CTA pairs, MN-major B and B2, plain stores
    if (!PAIR || L.sched != SCHED_DENSE || L.epi != EPI_STORE || L.accumulate ||
        p.splitk > 1 || L.kcat > 0 || !L.b_mn || L.b_batch_mode != BATCH_NONE ||
        L.swiglu_b || L.gather_a || L.gather_b || L.c_batch_n > 0 || L.ncat % 128 != 0 ||
        L.ncat >= L.N || !L.C2 || L.ldc2 < L.N - L.ncat)
      return MOE_ERR_UNSUPPORTED;
    if (!make_map_chunked(&mapB2, L.B2, BN / 128, false)) return MOE_ERR_ARG;
    p.ncat = L.ncat;
  }
  // (a gathered operand is copied by the gather warps, not by TMA: its map is
  // encoded only so that every map the kernel receives is a valid one.) Other
  // MN-major operands are read through a chunked map when their columns allow
  // (else one copy per 64-column chunk)
  // (the chunk coordinate is m0 / 64: grouped-M row starts are not 64-aligned)
  p.a_chunked = L.a_mn && !L.gather_a && L.sched != SCHED_GROUPED_M &&
                make_map_chunked(&mapA, L.A, BM / 64, false);
  // (a CTA of a pair loads half of the tile's B columns: BN/128 chunks)
  p.b_chunked = L.b_mn && !L.gather_b &&
                make_map_chunked(&mapB, L.B, (PAIR || L.swiglu_b) ? BN / 128 : BN / 64, b3);
  if (PAIR && L.b_mn && !p.b_chunked) return MOE_ERR_UNSUPPORTED;
  if (!p.a_chunked && !make_map(&mapA, L.A, L.gather_a ? 1 : (L.a_mn ? 64 : BM), false))
    return MOE_ERR_ARG;
  if (!p.b_chunked &&
      !make_map(&mapB, L.B, L.gather_b ? 1 : (L.b_mn ? 64 : (PAIR ? BN / 2 : BN)), b3))
    return MOE_ERR_ARG;
  // output (store) maps
  const long long rows_out = (L.sched == SCHED_GROUPED_M) ? L.R_cap : L.M;
  bool ok = true;
  p.c0_rank3 = 0;
  if (L.epi == EPI_STORE) {
    if (!L.accumulate) {
      const bool f32 = !L.c_bf16;
      if (L.sched == SCHED_GROUPED_K) {
        p.c0_rank3 = 1;
        ok = make_store_map(&mapC0, L.C, f32, true, L.N, L.M, L.G, L.ldc, L.c_batch_stride);
      } else if (p.splitk > 1) {
        // fp32 partial sums per K slice into the caller's split workspace [splitk][M][N]
        if (!L.splitk_ws) return MOE_ERR_WORKSPACE;
        p.c0_rank3 = 1;
        p.c_bf16 = 0;
        ok = make_store_map(&mapC0, L.splitk_ws, true, true, L.N, L.M, p.splitk, L.N,
                            static_cast<long long>(L.M) * L.N);
      } else if (L.c_batch_n > 0) {
        p.c0_rank3 = 1;
        ok = make_store_map(&mapC0, L.C, f32, true, L.c_batch_n, L.M, L.N / L.c_batch_n, L.ldc,
                            L.c_batch_stride);
      } else if (L.ncat > 0) {
        ok = make_store_map(&mapC0, L.C, f32, false, L.ncat, rows_out, 1, L.ldc, 0) &&
             make_store_map(&mapC1, L.C2, !L.c2_bf16, false, L.N - L.ncat, rows_out, 1, L.ldc2, 0);
      } else {
        ok = make_store_map(&mapC0, L.C, f32, false, L.N, rows_out, 1, L.ldc, 0);
      }
    }
  } else if (L.epi == EPI_SWIGLU) {  // 16-column blocks
    ok = make_store_map(&mapC0, L.h, false, false, L.ldh, rows_out, 1, L.ldh, 0, 16);
    if (ok && L.gu)
      ok = make_store_map(&mapC1, L.gu, false, false, L.ldgu, rows_out, 1, L.ldgu, 0, 16);
    if (ok && L.gu8) ok = make_u8_map(&mapC1, L.gu8, L.ldgu, rows_out, L.ldgu, 32);
  } else if (L.epi == EPI_ROWSCALE) {
    ok = make_store_map(&mapC0, L.C, false, false, L.N, rows_out, 1, L.ldc, 0);
  } else {  // EPI_SWIGLU_BWD (32-column blocks)
    ok = make_store_map(&mapC0, L.C, false, false, L.ldc, rows_out, 1, L.ldc, 0);
    if (ok && L.aux)
      ok = make_store_map(&mapC1, L.aux, false, false, L.ldaux, rows_out, 1, L.ldaux, 0);
    // the epilogue's inputs g|u (or their FP8 cache) and h, in the same 32 x 32 blocks
    if (ok && L.gu8) ok = make_u8_map(&mapA2, L.gu8, L.ldgu, rows_out, L.ldgu, 64);
    else if (ok) ok = make_store_map(&mapA2, L.gu, false, false, L.ldgu, rows_out, 1, L.ldgu, 0);
    if (ok) ok = make_store_map(&mapB2, L.h, false, false, L.ldh, rows_out, 1, L.ldh, 0);
  }
  if (!ok) return MOE_ERR_ARG;

  static bool attr_set[64] = {};  // one flag per device and template instance
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, EW, CW16, PAIR, GW, SBWD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    attr_set[dev] = true;
  }
  cudaError_t e;
  if (PAIR) {
    // clusters of two CTAs, one pair tile each at a time
    const long long pairs = num_sms() / 2;
    const int grid = 2 * static_cast<int>(upper < pairs ? upper : pairs);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    LaunchTimer lt(L.name, stream);
    e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, EW, CW16, PAIR, GW, SBWD>, mapA, mapB, mapC0, mapC1,
                           mapA2, mapB2, p);
  } else {
    const int grid = static_cast<int>(upper < num_sms() ? upper : num_sms());
    LaunchTimer lt(L.name, stream);
    gemm_tc_kernel<BN, EW, CW16, PAIR, GW, SBWD><<<grid, THREADS, C::SMEM_BYTES, stream>>>(
        mapA, mapB, mapC0, mapC1, mapA2, mapB2, p);
    e = cudaSuccess;
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace

// out (fp32 or bf16, layout of the GEMM's C) = sum over K slices of the fp32
// partials ws[s][m][n]; four columns per thread, slices summed in order.
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, int splitk, int M, int N,
                                     void* __restrict__ out, int out_bf16, long long ldc,
                                     int c_batch_n, long long c_batch_stride) {
  const long long n4 = static_cast<long long>(M) * (N / 4);
  const long long MN = static_cast<long long>(M) * N;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long m = i / (N / 4);
    const int n = static_cast<int>(i - m * (N / 4)) * 4;
    float4 acc = *reinterpret_cast<const float4*>(ws + m * N + n);
    for (int sl = 1; sl < splitk; ++sl) {
      const float4 v = *reinterpret_cast<const float4*>(ws + sl * MN + m * N + n);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    int col = n;
    long long base = 0;
    if (c_batch_n > 0) {
      const int cb = n / c_batch_n;
      col = n - cb * c_batch_n;
      base = cb * c_batch_stride;
    }
    const long long o = base + m * ldc + col;
    if (out_bf16) {
      uint2 pk = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
      *reinterpret_cast<uint2*>(reinterpret_cast<bf16*>(out) + o) = pk;
    } else {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o) = acc;
    }
  }
}

int gemm_epilogue_warps(const GemmLaunch& L) {
  // The fused SwiGLU epilogues do enough arithmetic and loads per element
  // that one warp per TMEM lane quadrant cannot hide their latency: they get
  // 8 warps (and one pipeline stage less). Plain stores keep 4 warps and the
  // deeper pipeline.
  return L.epi == EPI_SWIGLU ? 8 : 4;
}

int gemm_launch(const GemmLaunch& L, cudaStream_t stream) {
  const int ew = gemm_epilogue_warps(L);
  if (L.splitk > 1 && !(L.sched == SCHED_DENSE && L.epi == EPI_STORE && !L.accumulate))
    return MOE_ERR_UNSUPPORTED;
  // The SwiGLU forward epilogue (8 warps) works on 16-column chunks (smaller
  // staging, one more pipeline stage); its backward runs epilogue_loop_sbwd.
  // CTA pairs (256-row tiles, cta_group::2 MMAs, half of B per CTA) for the dense
  // schedule with 256-wide tiles and at least two row blocks
  const bool gather = L.gather_a || L.gather_b;
  const bool pair = L.pair && L.BN == 256 && L.sched == SCHED_DENSE && L.K > 0 && L.M > BM &&
                    !gather;
  int st;
  if (L.epi == EPI_SWIGLU_BWD) {
    // 4 epilogue warps with TMA-staged g, u, h (epilogue_loop_sbwd)
    if (L.BN == 256 && pair) st = launch_bn<256, 4, false, true, 0, true>(L, stream);
    else if (gather && L.BN == 256) st = launch_bn<256, 4, false, false, kGatherWarps, true>(L, stream);
    else if (gather && L.BN == 128) st = launch_bn<128, 4, false, false, kGatherWarps, true>(L, stream);
    else if (L.BN == 256) st = launch_bn<256, 4, false, false, 0, true>(L, stream);
    else if (L.BN == 128) st = launch_bn<128, 4, false, false, 0, true>(L, stream);
    else return MOE_ERR_UNSUPPORTED;
  } else if (L.BN == 256 && pair)
    st = ew == 4 ? launch_bn<256, 4, false, true>(L, stream)
                 : launch_bn<256, 8, true, true>(L, stream);
  else if (gather && L.BN == 256)
    st = ew == 4 ? launch_bn<256, 4, false, false, kGatherWarps>(L, stream)
                 : launch_bn<256, 8, true, false, kGatherWarps>(L, stream);
  else if (gather && L.BN == 128)
    st = ew == 4 ? launch_bn<128, 4, false, false, kGatherWarps>(L, stream)
                 : launch_bn<128, 8, true, false, kGatherWarps>(L, stream);
  else if (L.BN == 256)
    st = ew == 4 ? launch_bn<256, 4, false, false>(L, stream)
                 : launch_bn<256, 8, true, false>(L, stream);
  else if (L.BN == 128)
    st = ew == 4 ? launch_bn<128, 4, false, false>(L, stream)
                 : launch_bn<128, 8, true, false>(L, stream);
  else
    return MOE_ERR_UNSUPPORTED;
  if (st != MOE_OK || L.splitk <= 1) return st;
  const int kslice = ((L.K + L.splitk - 1) / L.splitk + BK - 1) / BK * BK;
  const int nslices = (L.K + kslice - 1) / kslice;
  const long long n4 = static_cast<long long>(L.M) * (L.N / 4);
  long long blocks = (n4 + 255) / 256;
  if (blocks > 4L * num_sms()) blocks = 4L * num_sms();
  {
    LaunchTimer lt("splitk_reduce", stream);
    splitk_reduce_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
        L.splitk_ws, nslices, L.M, L.N, L.C, L.c_bf16, L.ldc, L.c_batch_n, L.c_batch_stride);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe
