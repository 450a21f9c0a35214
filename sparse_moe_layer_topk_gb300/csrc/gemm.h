// Host interface of the tcgen05 GEMM engine shared by every contraction of the
// layer (router logits, latent projections, grouped SwiGLU experts and all of
// their dgrad / wgrad products).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

enum GemmSched : int {
  SCHED_DENSE = 0,      // one M x N x K problem
  SCHED_GROUPED_M = 1,  // G problems over row segments offsets[g]..offsets[g+1] (ragged M)
  SCHED_GROUPED_K = 2,  // G problems whose K runs over rows offsets[g]..offsets[g+1] (ragged K)
};

enum GemmEpi : int {
  EPI_STORE = 0,       // C = acc (fp32 or bf16), or C += acc for bf16 with accumulate
  EPI_SWIGLU = 1,      // h = silu(gate) * up (+ bf16 copy of gate|up)
  EPI_ROWSCALE = 2,    // C = row_w[row] * acc (bf16)
  EPI_SWIGLU_BWD = 3,  // dgrad of SwiGLU + routing-weight partial dots
};

// B operand batch selection (3-D tensor map, third coordinate).
enum GemmBatch : int {
  BATCH_NONE = 0,
  BATCH_GROUP = 1,   // batch = group index g
  BATCH_FROM_N = 2,  // batch = n_tile / n_tiles_per_batch
  BATCH_FROM_K = 3,  // batch = k / k_per_batch
};

// A row-major bf16 matrix in device memory: [batch][rows][cols], cols contiguous.
struct MatView {
  const void* ptr = nullptr;
  long long rows = 0, cols = 0;
  long long ld = 0;            // elements between rows
  long long batch = 1;         // >1 (or force3d) gives a 3-D tensor map
  long long batch_stride = 0;  // elements between batches
};

struct GemmLaunch {
  const char* name = "gemm";  // label of the launch in the optional per-kernel timing
  int BN = 256;  // 128 or 256
  int sched = SCHED_DENSE;
  int M = 0, N = 0, K = 0, G = 1;
  const int* offsets = nullptr;     // [G+1]
  const int* tile_sched = nullptr;  // [G+1] (SCHED_GROUPED_M)
  const int* expert_order = nullptr;  // grouped-M: groups walked in this order (tile_sched
                                      // is then the scan in that order); nullptr = natural
  int R_cap = 0;                    // row capacity (SCHED_GROUPED_M grid bound)
  // Grouped-M tile shape per tile: a tile of at most 64 rows (an expert's last
  // rows, or a small expert) runs M = 64 MMAs, half the tensor work of M = 128.
  int m64 = 1;
  // operands: A is [M][K] (a_mn = 0) or [K][M] (a_mn = 1);
  //           B is [N][K] (b_mn = 0) or [K][N] (b_mn = 1), optionally batched.
  MatView A, B;
  int a_mn = 0, b_mn = 0;
  int b_batch_mode = BATCH_NONE;
  int n_tiles_per_batch = 0;
  int k_per_batch = 0;
  int swiglu_b = 0;  // B tile = BN/2 gate columns + BN/2 up columns (f apart)
  int f = 0;
  int n_tiles = 0;   // override of ceil(N / BN) (swiglu: h columns / (BN/2))
  // epilogue
  int epi = EPI_STORE;
  void* C = nullptr;
  long long ldc = 0;
  long long c_batch_stride = 0;  // SCHED_GROUPED_K: per group; EPI_STORE + c_batch_n: per N block
  int c_batch_n = 0;
  int c_bf16 = 1;
  int accumulate = 0;
  const float* row_w = nullptr;
  void* gu = nullptr;  // bf16
  long long ldgu = 0;
  // EPI_SWIGLU / EPI_SWIGLU_BWD with an FP8 cache of g|u instead of gu: E4M3
  // bytes [rows][ldgu] and fp32 scales [rows][ld_scale], one per 64 features
  // of g, then of u (ld_scale = 2 f / 64). The forward needs 256-wide tiles.
  void* gu8 = nullptr;
  float* gu_scale = nullptr;
  int ld_scale = 0;
  void* h = nullptr;  // bf16
  long long ldh = 0;
  void* aux = nullptr;  // bf16
  long long ldaux = 0;
  float* dw_part = nullptr;
  int dw_nparts = 0;
  int* err_flag = nullptr;
  // Split-K (dense EPI_STORE only): K is cut into `splitk` slices whose fp32
  // partial products go to splitk_ws [splitk][M][N]; a reduce kernel then
  // writes C. Deterministic (fixed summation order).
  int splitk = 1;
  float* splitk_ws = nullptr;
  // Row gather: with gather_a (gather_b) the A (B) view is an unpermuted source
  // tensor and permuted row r is its row gather_idx[r], copied by extra warps of
  // the kernel (16-byte cp.async). Supported for the K-major A of a grouped-M
  // GEMM and for one MN-major operand of a grouped-K GEMM.
  const int* gather_idx = nullptr;
  int gather_a = 0, gather_b = 0;
  // K concatenation (dense, K-major operands): for k >= kcat the A and B tiles
  // come from A2 ([M][K-kcat]) and B2 ([N][K-kcat]): C = A B^T + A2 B2^T in one
  // accumulator. kcat must be a multiple of 64.
  int kcat = 0;
  MatView A2, B2;
  // N concatenation (dense CTA pairs, MN-major B, plain stores): output columns
  // n >= ncat come from B2 ([K][N - ncat]) and go to C2 ([M][ldc2], bf16 when
  // c2_bf16) at column n - ncat; the others from B to C. ncat must be a multiple
  // of 128, so that neither CTA's half of a tile's B columns straddles it.
  int ncat = 0;
  void* C2 = nullptr;
  long long ldc2 = 0;
  int c2_bf16 = 1;
  // Dense schedule with 256-wide tiles: run CTA pairs on 256-row tiles
  // (cta_group::2 MMAs; each CTA stages half of B). 0 forces single CTAs.
  int pair = 1;
};

// Bytes of split workspace gemm_launch needs for M x N with `splitk` slices.
inline size_t gemm_splitk_ws_bytes(long long M, long long N, int splitk) {
  return splitk > 1 ? static_cast<size_t>(splitk) * M * N * 4 : 0;
}

// Returns MOE_OK or an MOE_ERR_* code (argument checks, launch errors).
int gemm_launch(const GemmLaunch& L, cudaStream_t stream);

// Number of epilogue warps gemm_launch uses for L (4 or 8). With 8, two warps
// share each accumulator row and EPI_SWIGLU_BWD writes two routing-weight
// partials per row and n tile (dw_nparts = 2 * n tiles).
int gemm_epilogue_warps(const GemmLaunch& L);

int num_sms();
void record_cuda_error(cudaError_t e);

}  // namespace moe
