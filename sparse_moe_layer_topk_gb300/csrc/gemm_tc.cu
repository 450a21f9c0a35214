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
//               work (SwiGLU, routing-weight scale, SwiGLU backward), stores.
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

template <int BN>
struct Cfg {
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
};

struct Params {
  int sched, M, N, K, G;
  const int* offsets;
  const int* tile_sched;
  int a_mn, b_mn, b_rank3;
  int b_batch_mode, n_tiles_per_batch, k_per_batch;
  int swiglu_b, f;
  int mt, nt;         // m tiles (dense / grouped-K), n tiles
  int total_static;   // tile count when it does not depend on device data
  int epi;
  void* C;
  long long ldc, c_batch_stride;
  int c_batch_n, c_bf16, accumulate;
  const float* row_w;
  bf16* gu;
  long long ldgu;
  bf16* h;
  long long ldh;
  bf16* aux;
  long long ldaux;
  float* dw_part;
  int dw_nparts;
  int* err_flag;
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

__device__ __forceinline__ int total_tiles(const Params& p) {
  if (p.sched == SCHED_GROUPED_M) return __ldg(p.tile_sched + p.G) * p.nt;
  return p.total_static;
}

template <int BN>
__device__ __forceinline__ Tile decode(const Params& p, int t) {
  Tile ti;
  const int bn_eff = p.swiglu_b ? BN / 2 : BN;
  if (p.sched == SCHED_GROUPED_M) {
    int lo = 0, hi = p.G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.tile_sched + mid) * p.nt <= t) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int ts0 = __ldg(p.tile_sched + g);
    const int mtg = __ldg(p.tile_sched + g + 1) - ts0;
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
    ti.g = 0;
    ti.n_blk = t / p.mt;
    const int m_blk = t - ti.n_blk * p.mt;
    ti.m0 = m_blk * BM;
    ti.rows = min(BM, p.M - ti.m0);
    if (p.b_batch_mode == BATCH_FROM_N) {
      ti.batch = ti.n_blk / p.n_tiles_per_batch;
      ti.nb0 = (ti.n_blk - ti.batch * p.n_tiles_per_batch) * bn_eff;
    } else {
      ti.batch = 0;
      ti.nb0 = ti.n_blk * bn_eff;
    }
    ti.k0 = 0;
    ti.krows = p.K;
    ti.nk = (p.K + BK - 1) / BK;
  }
  return ti;
}

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, int* err_flag) {
  *abort_flag = 1;
  set_flag(err_flag, MOE_FLAG_TIMEOUT);
}

// ------------------------------------------------------------------ producer

template <int BN>
__device__ void producer_loop(const Params& p, const CUtensorMap* mapA, const CUtensorMap* mapB,
                              uint8_t* smem, uint64_t* full, uint64_t* empty,
                              volatile int* abort_flag) {
  using C = Cfg<BN>;
  int stage = 0;
  uint32_t phase = 0;
  long long issued = 0;
  const int total = total_tiles(p);
  bool ok = true;
  for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
    const Tile ti = decode<BN>(p, t);
    for (int kb = 0; kb < ti.nk; ++kb) {
      if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
        raise_abort(abort_flag, p.err_flag);
        ok = false;
        break;
      }
      const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
      const uint32_t sB = sA + A_BYTES;
      mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
      const int k = ti.k0 + kb * BK;
      // A
      if (!p.a_mn) {
        tma_load_2d(sA, mapA, &full[stage], k, ti.m0);
      } else {
        tma_load_2d(sA, mapA, &full[stage], ti.m0, k);
        tma_load_2d(sA + CHUNK_BYTES, mapA, &full[stage], ti.m0 + 64, k);
      }
      // B
      int kb_coord = k, batch = ti.batch;
      if (p.b_batch_mode == BATCH_FROM_K) {
        batch = k / p.k_per_batch;
        kb_coord = k - batch * p.k_per_batch;
      }
      if (!p.b_mn) {
        if (p.b_rank3) tma_load_3d(sB, mapB, &full[stage], kb_coord, ti.nb0, batch);
        else tma_load_2d(sB, mapB, &full[stage], kb_coord, ti.nb0);
      } else {
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) {
          int ncoord;
          if (p.swiglu_b) {
            ncoord = (c < BN / 128) ? ti.nb0 + 64 * c : p.f + ti.nb0 + 64 * (c - BN / 128);
          } else {
            ncoord = ti.nb0 + 64 * c;
          }
          if (p.b_rank3) tma_load_3d(sB + c * CHUNK_BYTES, mapB, &full[stage], ncoord, kb_coord, batch);
          else tma_load_2d(sB + c * CHUNK_BYTES, mapB, &full[stage], ncoord, kb_coord);
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
  } else {
    // Wait (bounded, ignoring the abort flag) for the copies still in flight so
    // that none lands in shared memory after the CTA exits.
    int s = stage;
    uint32_t ph = phase;
    volatile int never = 0;
    for (long long i = 0; i < issued && i < C::STAGES; ++i) {
      if (--s < 0) { s = C::STAGES - 1; ph ^= 1u; }
      mbar_wait(&full[s], ph, &never);
    }
  }
}

// ------------------------------------------------------------------ MMA

template <int BN>
__device__ void mma_loop(const Params& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                         uint64_t* tfull, uint64_t* tempty, uint64_t* drain, uint32_t tmem_base,
                         volatile int* abort_flag) {
  using C = Cfg<BN>;
  const uint32_t lane = lane_id();
  const uint32_t idesc = make_idesc_bf16(BM, BN, p.a_mn, p.b_mn);
  const uint32_t a_lbo = p.a_mn ? CHUNK_BYTES : 16, b_lbo = p.b_mn ? CHUNK_BYTES : 16;
  const uint32_t a_kstep = p.a_mn ? 2048 : 32, b_kstep = p.b_mn ? 2048 : 32;
  int stage = 0;
  uint32_t phase = 0;
  bool issued_any = false;
  const int total = total_tiles(p);
  int it = 0;
  bool ok = true;
  for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
    const Tile ti = decode<BN>(p, t);
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
      uint8_t* sA = smem + stage * C::STAGE_BYTES;
      if (p.sched == SCHED_GROUPED_K) {
        const int valid = ti.krows - kb * BK;
        if (valid < BK) {
          // Rows past this expert's segment belong to the next expert: zero them
          // in every 64-wide chunk of A and B (rows are whole 128-byte lines).
          const int nchunks = 2 + BN / 64;
          const int per_chunk = (BK - valid) * 8;
          const uint4 zero = make_uint4(0, 0, 0, 0);
          for (int i = lane; i < per_chunk * nchunks; i += 32) {
            const int c = i / per_chunk;
            const int rem = i - c * per_chunk;
            const int row = valid + (rem >> 3);
            *reinterpret_cast<uint4*>(sA + c * CHUNK_BYTES + row * 128 + (rem & 7) * 16) = zero;
          }
          fence_proxy_async_smem();
        }
      }
      __syncwarp();
      if (lane == 0) {
        const uint32_t a0 = smem_u32(sA), b0 = a0 + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = make_sdesc(a0 + kk * a_kstep, a_lbo, 1024);
          const uint64_t bd = make_sdesc(b0 + kk * b_kstep, b_lbo, 1024);
          mma_bf16_ss(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
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

// ------------------------------------------------------------------ epilogue

__device__ __forceinline__ void store16(void* dst, uint4 v) { *reinterpret_cast<uint4*>(dst) = v; }

template <int BN>
__device__ void epilogue_loop(const Params& p, uint64_t* tfull, uint64_t* tempty,
                              uint32_t tmem_base, volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5;
  const int q = warp & 3;  // tensor-memory lane quadrant this warp may read
  const uint32_t lane = lane_id();
  const int r_loc = q * 32 + static_cast<int>(lane);
  const int total = total_tiles(p);
  int it = 0;
  for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
    const Tile ti = decode<BN>(p, t);
    const int buf = it & 1;
    const uint32_t use = static_cast<uint32_t>(it >> 1);
    if (!mbar_wait(&tfull[buf], use & 1u, abort_flag)) {
      raise_abort(abort_flag, p.err_flag);
      break;
    }
    tc_fence_after();
    const bool row_ok = r_loc < ti.rows;
    const long long grow = static_cast<long long>(ti.m0) + r_loc;
    const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(buf * BN);
    const bool has_acc = ti.nk > 0;

    if (p.epi == EPI_STORE) {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int n = ti.nb0 + c * 32;  // output column over the full N
        if (n >= p.N) break;             // warp-uniform N tail
        int ncol = n;
        long long cbase = 0;
        if (p.sched == SCHED_GROUPED_K) {
          cbase = static_cast<long long>(ti.g) * p.c_batch_stride;
        } else if (p.c_batch_n > 0) {
          const int cb = n / p.c_batch_n;
          ncol = n - cb * p.c_batch_n;
          cbase = static_cast<long long>(cb) * p.c_batch_stride;
        }
        uint32_t r[32];
        if (has_acc) {
          tmem_ld_32x32b_x32(trow + c * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (!row_ok) continue;
        const long long off = cbase + grow * p.ldc + ncol;
        if (p.c_bf16) {
          bf16* dst = reinterpret_cast<bf16*>(p.C) + off;
          if (p.accumulate) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 old = *reinterpret_cast<const uint4*>(dst + v * 8);
              const uint32_t o[4] = {old.x, old.y, old.z, old.w};
              uint32_t pk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                pk[e] = pack_bf16(__uint_as_float(r[v * 8 + 2 * e]) + bf16_lo(o[e]),
                                  __uint_as_float(r[v * 8 + 2 * e + 1]) + bf16_hi(o[e]));
              store16(dst + v * 8, make_uint4(pk[0], pk[1], pk[2], pk[3]));
            }
          } else {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t pk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                pk[e] = pack_bf16(__uint_as_float(r[v * 8 + 2 * e]),
                                  __uint_as_float(r[v * 8 + 2 * e + 1]));
              store16(dst + v * 8, make_uint4(pk[0], pk[1], pk[2], pk[3]));
            }
          }
        } else {
          float* dst = reinterpret_cast<float*>(p.C) + off;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            store16(dst + v * 4, make_uint4(r[v * 4], r[v * 4 + 1], r[v * 4 + 2], r[v * 4 + 3]));
        }
      }
    } else if (p.epi == EPI_SWIGLU) {
      // TMEM columns [0, BN/2) hold the gate, [BN/2, BN) the up projection.
      const int out_batch = (p.b_batch_mode == BATCH_FROM_N) ? ti.batch : 0;
#pragma unroll 1
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t rg[32], ru[32];
        tmem_ld_32x32b_x32(trow + c * 32, rg);
        tmem_ld_32x32b_x32(trow + BN / 2 + c * 32, ru);
        tmem_ld_wait();
        if (!row_ok) continue;
        const int j = ti.nb0 + c * 32;
        bf16* hdst = p.h + grow * p.ldh + static_cast<long long>(out_batch) * p.f + j;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i0 = v * 8 + 2 * e;
            const float g0 = __uint_as_float(rg[i0]), g1 = __uint_as_float(rg[i0 + 1]);
            const float u0 = __uint_as_float(ru[i0]), u1 = __uint_as_float(ru[i0 + 1]);
            pk[e] = pack_bf16(g0 * sigmoidf_(g0) * u0, g1 * sigmoidf_(g1) * u1);
          }
          store16(hdst + v * 8, make_uint4(pk[0], pk[1], pk[2], pk[3]));
        }
        if (p.gu) {
          bf16* gdst = p.gu + grow * p.ldgu + static_cast<long long>(out_batch) * 2 * p.f + j;
          bf16* udst = gdst + p.f;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t pg[4], pu[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i0 = v * 8 + 2 * e;
              pg[e] = pack_bf16(__uint_as_float(rg[i0]), __uint_as_float(rg[i0 + 1]));
              pu[e] = pack_bf16(__uint_as_float(ru[i0]), __uint_as_float(ru[i0 + 1]));
            }
            store16(gdst + v * 8, make_uint4(pg[0], pg[1], pg[2], pg[3]));
            store16(udst + v * 8, make_uint4(pu[0], pu[1], pu[2], pu[3]));
          }
        }
      }
    } else if (p.epi == EPI_ROWSCALE) {
      const float w = (row_ok && p.row_w) ? __ldg(p.row_w + grow) : 1.0f;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int n = ti.nb0 + c * 32;
        if (n >= p.N) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(trow + c * 32, r);
        tmem_ld_wait();
        if (!row_ok) continue;
        bf16* dst = reinterpret_cast<bf16*>(p.C) + grow * p.ldc + n;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pk[e] = pack_bf16(w * __uint_as_float(r[v * 8 + 2 * e]),
                              w * __uint_as_float(r[v * 8 + 2 * e + 1]));
          store16(dst + v * 8, make_uint4(pk[0], pk[1], pk[2], pk[3]));
        }
      }
    } else {  // EPI_SWIGLU_BWD
      const float w = (row_ok && p.row_w) ? __ldg(p.row_w + grow) : 1.0f;
      float dot = 0.0f;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int n = ti.nb0 + c * 32;  // column of dh within [0, S*f)
        if (n >= p.N) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(trow + c * 32, r);
        tmem_ld_wait();
        if (!row_ok) continue;
        const int s = n / p.f;
        const int jj = n - s * p.f;
        const bf16* gsrc = p.gu + grow * p.ldgu + static_cast<long long>(s) * 2 * p.f + jj;
        const bf16* usrc = gsrc + p.f;
        const bf16* hsrc = p.h + grow * p.ldh + n;
        bf16* dgdst = reinterpret_cast<bf16*>(p.C) + grow * p.ldc + static_cast<long long>(s) * 2 * p.f + jj;
        bf16* dudst = dgdst + p.f;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 G4 = *reinterpret_cast<const uint4*>(gsrc + v * 8);
          const uint4 U4 = *reinterpret_cast<const uint4*>(usrc + v * 8);
          const uint4 H4 = *reinterpret_cast<const uint4*>(hsrc + v * 8);
          const uint32_t Gw[4] = {G4.x, G4.y, G4.z, G4.w};
          const uint32_t Uw[4] = {U4.x, U4.y, U4.z, U4.w};
          const uint32_t Hw[4] = {H4.x, H4.y, H4.z, H4.w};
          uint32_t pdg[4], pdu[4], phw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float dgv[2], duv[2], hwv[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const float a = __uint_as_float(r[v * 8 + 2 * e + hh]);
              const float g = hh ? bf16_hi(Gw[e]) : bf16_lo(Gw[e]);
              const float u = hh ? bf16_hi(Uw[e]) : bf16_lo(Uw[e]);
              const float hv = hh ? bf16_hi(Hw[e]) : bf16_lo(Hw[e]);
              dot = fmaf(a, hv, dot);
              const float dh = w * a;
              const float sg = sigmoidf_(g);
              const float silu = g * sg;
              dgv[hh] = dh * u * sg * (1.0f + g * (1.0f - sg));
              duv[hh] = dh * silu;
              hwv[hh] = w * hv;
            }
            pdg[e] = pack_bf16(dgv[0], dgv[1]);
            pdu[e] = pack_bf16(duv[0], duv[1]);
            phw[e] = pack_bf16(hwv[0], hwv[1]);
          }
          store16(dgdst + v * 8, make_uint4(pdg[0], pdg[1], pdg[2], pdg[3]));
          store16(dudst + v * 8, make_uint4(pdu[0], pdu[1], pdu[2], pdu[3]));
          if (p.aux)
            store16(p.aux + grow * p.ldaux + n + v * 8, make_uint4(phw[0], phw[1], phw[2], phw[3]));
        }
      }
      if (row_ok && p.dw_part) p.dw_part[grow * p.dw_nparts + ti.n_blk] = dot;
    }
    tc_fence_before();
    mbar_arrive(&tempty[buf]);
  }
}

template <int BN>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA,
                   const __grid_constant__ CUtensorMap mapB, const Params p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane_id() == 0) producer_loop<BN>(p, &mapA, &mapB, smem, full, empty, abort_flag);
  } else if (warp == 1) {
    mma_loop<BN>(p, smem, full, empty, tfull, tempty, drain, tmem_base, abort_flag);
  } else {
    epilogue_loop<BN>(p, tfull, tempty, tmem_base, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
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

template <int BN>
int launch_bn(const GemmLaunch& L, cudaStream_t stream) {
  using C = Cfg<BN>;
  Params p{};
  p.sched = L.sched;
  p.M = L.M;
  p.N = L.N;
  p.K = L.K;
  p.G = L.G;
  p.offsets = L.offsets;
  p.tile_sched = L.tile_sched;
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
    p.total_static = p.mt * p.nt;
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
  p.h = reinterpret_cast<bf16*>(L.h);
  p.ldh = L.ldh;
  p.aux = reinterpret_cast<bf16*>(L.aux);
  p.ldaux = L.ldaux;
  p.dw_part = L.dw_part;
  p.dw_nparts = L.dw_nparts;
  p.err_flag = L.err_flag;
  if (upper <= 0) return MOE_OK;

  if (!get_encoder()) return MOE_ERR_CUDA;
  CUtensorMap mapA, mapB;
  if (!make_map(&mapA, L.A, L.a_mn ? 64 : BM, false)) return MOE_ERR_ARG;
  if (!make_map(&mapB, L.B, L.b_mn ? 64 : BN, b3)) return MOE_ERR_ARG;

  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return MOE_ERR_CUDA;
    }
    attr_set[dev] = true;
  }
  const int grid = static_cast<int>(upper < num_sms() ? upper : num_sms());
  {
    LaunchTimer lt(L.name, stream);
    gemm_tc_kernel<BN><<<grid, 192, C::SMEM_BYTES, stream>>>(mapA, mapB, p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace

int gemm_launch(const GemmLaunch& L, cudaStream_t stream) {
  if (L.BN == 256) return launch_bn<256>(L, stream);
  if (L.BN == 128) return launch_bn<128>(L, stream);
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
