// C-ABI entry points of libmoe: host-side argument checks, workspace carving
// and the launch sequence of each step. Every entry point enqueues work on
// the caller's stream and returns; none allocates, frees or synchronises.
#include <algorithm>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"

namespace moe {

namespace {
thread_local int g_last_cuda_error = 0;
int g_num_sms[64] = {};
}  // namespace

void record_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }

int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (g_num_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

}  // namespace moe

using namespace moe;

namespace {

inline cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t up256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

inline int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  record_cuda_error(e);
  return MOE_ERR_CUDA;
}

#define MOE_CHECK(expr)          \
  do {                           \
    const int _st = (expr);      \
    if (_st != MOE_OK) return _st; \
  } while (0)

#define MOE_REQUIRE(cond, code) \
  do {                          \
    if (!(cond)) return (code); \
  } while (0)

MatView view(const void* p, long long rows, long long cols, long long ld, long long batch = 1,
             long long batch_stride = 0) {
  MatView v;
  v.ptr = p;
  v.rows = rows;
  v.cols = cols;
  v.ld = ld;
  v.batch = batch;
  v.batch_stride = batch_stride;
  return v;
}

// Tile width: 256 unless N is narrow or a 256-wide tail would waste more than a quarter.
inline int pick_bn(int N) { return (N % 256 == 0 || (N > 512 && N % 256 >= 128)) ? 256 : 128; }

// K slices for a dense wgrad with few output tiles (K = tokens, long): enough
// slices to give ~128 tiles, at most 4, each slice at least 1024 rows of K.
inline int wgrad_splitk(int M, int N, int K) {
  const int bn = pick_bn(N);
  const int tiles = ((M + 127) / 128) * ((N + bn - 1) / bn);
  int s = 1;
  while (s < 4 && tiles * s * 2 <= 128 && K / (s * 2) >= 1024) s *= 2;
  return s;
}

size_t shared_bwd_ws(int T, int l, int f, int S_) {
  const long long Sf = static_cast<long long>(S_) * f;
  const size_t split = std::max(gemm_splitk_ws_bytes(Sf, l, wgrad_splitk(static_cast<int>(Sf), l, T)),
                                gemm_splitk_ws_bytes(l, 2 * Sf, wgrad_splitk(l, static_cast<int>(2 * Sf), T)));
  return up256(static_cast<size_t>(T) * Sf * 2 * 2) + up256(split);
}

// C[M][N] (bf16 or fp32) = A[M][K] @ B, B given as [K][N] (b_mn) or [N][K].
int dense_gemm(const char* name, const void* A, long long lda, int a_mn, const void* B,
               long long ldb, int b_mn, int M, int N, int K, void* C, long long ldc, int c_bf16,
               int accumulate, cudaStream_t st) {
  GemmLaunch L;
  L.name = name;
  L.BN = pick_bn(N);
  L.sched = SCHED_DENSE;
  L.M = M;
  L.N = N;
  L.K = K;
  L.a_mn = a_mn;
  L.b_mn = b_mn;
  L.A = a_mn ? view(A, K, M, lda) : view(A, M, K, lda);
  L.B = b_mn ? view(B, K, N, ldb) : view(B, N, K, ldb);
  L.epi = EPI_STORE;
  L.C = C;
  L.ldc = ldc;
  L.c_bf16 = c_bf16;
  L.accumulate = accumulate;
  return gemm_launch(L, st);
}

struct WsCarver {
  char* p;
  size_t left;
  bool ok = true;
  void* take(size_t bytes) {
    bytes = up256(bytes);
    if (bytes > left) {
      ok = false;
      return nullptr;
    }
    void* r = p;
    p += bytes;
    left -= bytes;
    return r;
  }
};

size_t grouped_bwd_ws(long long R, int f) {
  // upper bound of the routing-weight partials per row: 2 epilogue warp groups
  // x n tiles (tiles are at least 128 wide)
  const int nparts = 2 * ((f + 127) / 128);
  return up256(static_cast<size_t>(R) * 2 * f * 2) + up256(static_cast<size_t>(R) * f * 2) +
         up256(static_cast<size_t>(R) * nparts * 4);
}

}  // namespace

extern "C" {

int moe_version(void) { return 1; }

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument (null pointer or dimension out of range)";
    case MOE_ERR_ALIGN: return "misaligned pointer or dimension not a multiple of 64";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or option";
    case MOE_ERR_CUDA: return "CUDA error (see moe_last_cuda_error)";
    default: return "unknown status";
  }
}

int moe_last_cuda_error(void) { return g_last_cuda_error; }

size_t moe_workspace_size(int op, int T, int d, int l, int E, int k, int f, int S) {
  (void)d;
  (void)l;
  switch (op) {
    case MOE_OP_ROUTE_TOPK: return up256(static_cast<size_t>(T) * E * 4);
    case MOE_OP_PERMUTE: return up256(static_cast<size_t>(permute_chunks(T)) * E * 4);
    case MOE_OP_GROUPED_SWIGLU_BWD:
      return grouped_bwd_ws(static_cast<long long>(T) * (k > 0 ? k : 1), f);
    case MOE_OP_SHARED_SWIGLU_BWD: return shared_bwd_ws(T, l, f, S);
    case MOE_OP_ROUTE_TOPK_BWD: return up256(static_cast<size_t>(T) * E * 2);
    case MOE_OP_ROUTER_AUX: return up256(static_cast<size_t>(aux_partial_warps(T)) * E * 4);
    default: return 0;
  }
}

// ---------------------------------------------------------------- routing

int moe_router_logits(const uint16_t* x, const uint16_t* Wr, int T, int d, int E, float* logits,
                      void* stream) {
  MOE_REQUIRE(x && Wr && logits, MOE_ERR_ARG);
  MOE_REQUIRE(T >= 0 && d > 0 && E > 0 && E <= 1024, MOE_ERR_ARG);
  MOE_REQUIRE(d % 64 == 0 && E % 64 == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(al16(x) && al16(Wr) && al16(logits), MOE_ERR_ALIGN);
  if (T == 0) return MOE_OK;
  return dense_gemm("router_logits_gemm", x, d, 0, Wr, E, 1, T, E, d, logits, E, 0, 0, S(stream));
}

int moe_topk_from_logits(const float* logits, const float* bias, int T, int E, int k,
                         int32_t* topk_idx, float* topk_w, float* topk_s, int32_t* err_flag,
                         void* stream) {
  MOE_REQUIRE(logits && topk_idx && topk_w && topk_s, MOE_ERR_ARG);
  MOE_REQUIRE(T >= 0 && E > 0 && E <= 1024 && k >= 1 && k <= 32 && k <= E, MOE_ERR_ARG);
  if (T == 0) return MOE_OK;
  return cuda_status(launch_topk(logits, bias, T, E, k, topk_idx, topk_w, topk_s, err_flag,
                                 S(stream)));
}

int moe_route_topk(const uint16_t* x, const uint16_t* Wr, const float* bias, int T, int d, int E,
                   int k, int32_t* topk_idx, float* topk_w, float* topk_s, void* ws,
                   size_t ws_bytes, int32_t* err_flag, void* stream) {
  MOE_REQUIRE(x && Wr && topk_idx && topk_w && topk_s, MOE_ERR_ARG);
  MOE_REQUIRE(T >= 0 && d > 0 && E > 0 && E <= 1024 && k >= 1 && k <= 32 && k <= E, MOE_ERR_ARG);
  MOE_REQUIRE(d % 64 == 0 && E % 64 == 0, MOE_ERR_ALIGN);
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(ws != nullptr, MOE_ERR_WORKSPACE);
  MOE_REQUIRE(ws_bytes >= moe_workspace_size(MOE_OP_ROUTE_TOPK, T, d, 0, E, k, 0, 0),
              MOE_ERR_WORKSPACE);
  float* L = reinterpret_cast<float*>(ws);
  MOE_CHECK(moe_router_logits(x, Wr, T, d, E, L, stream));
  return moe_topk_from_logits(L, bias, T, E, k, topk_idx, topk_w, topk_s, err_flag, stream);
}

int moe_route_topk_latent(const uint16_t* x, const uint16_t* Wr, const float* bias,
                          const uint16_t* W_dn, int T, int d, int E, int k, int l,
                          int32_t* topk_idx, float* topk_w, float* topk_s, uint16_t* z, void* ws,
                          size_t ws_bytes, int32_t* err_flag, void* stream) {
  MOE_REQUIRE(x && Wr && W_dn && z && topk_idx && topk_w && topk_s, MOE_ERR_ARG);
  MOE_REQUIRE(T >= 0 && d > 0 && l > 0 && E > 0 && E <= 1024 && k >= 1 && k <= 32 && k <= E,
              MOE_ERR_ARG);
  MOE_REQUIRE(d % 64 == 0 && E % 64 == 0 && l % 64 == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(al16(x) && al16(Wr) && al16(W_dn) && al16(z), MOE_ERR_ALIGN);
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(ws != nullptr, MOE_ERR_WORKSPACE);
  MOE_REQUIRE(ws_bytes >= moe_workspace_size(MOE_OP_ROUTE_TOPK, T, d, 0, E, k, 0, 0),
              MOE_ERR_WORKSPACE);
  float* L = reinterpret_cast<float*>(ws);
  cudaStream_t st = S(stream);
  if (T > 128 && E % 128 == 0 && pick_bn(E + l) == 256) {  // CTA pairs: two row blocks or more
    // one GEMM over [Wr | W_dn]: x is read once; columns < E are the fp32 logits,
    // the rest the bf16 latent z
    GemmLaunch G;
    G.name = "router_latent_gemm";
    G.BN = 256;
    G.sched = SCHED_DENSE;
    G.M = T;
    G.N = E + l;
    G.K = d;
    G.A = view(x, T, d, d);
    G.B = view(Wr, d, E, E);
    G.b_mn = 1;
    G.B2 = view(W_dn, d, l, l);
    G.ncat = E;
    G.epi = EPI_STORE;
    G.C = L;
    G.ldc = E;
    G.c_bf16 = 0;
    G.C2 = z;
    G.ldc2 = l;
    G.c2_bf16 = 1;
    MOE_CHECK(gemm_launch(G, st));
  } else {
    MOE_CHECK(moe_router_logits(x, Wr, T, d, E, L, stream));
    MOE_CHECK(moe_latent_proj(x, W_dn, T, d, l, z, stream));
  }
  return moe_topk_from_logits(L, bias, T, E, k, topk_idx, topk_w, topk_s, err_flag, stream);
}

int moe_router_aux_loss(const float* logits, const float* bias, int T, int E, float* p_mean,
                        float* loss, void* ws, size_t ws_bytes, void* stream) {
  MOE_REQUIRE(logits && p_mean && loss, MOE_ERR_ARG);
  MOE_REQUIRE(T > 0 && E > 0 && E <= 1024, MOE_ERR_ARG);
  MOE_REQUIRE(ws != nullptr && ws_bytes >= moe_workspace_size(MOE_OP_ROUTER_AUX, T, 0, 0, E, 0, 0, 0),
              MOE_ERR_WORKSPACE);
  return cuda_status(launch_aux_loss(logits, bias, T, E, reinterpret_cast<float*>(ws), p_mean, loss,
                                     S(stream)));
}

// ---------------------------------------------------------------- permute

int moe_permute(const uint16_t* z, const int32_t* topk_idx, const float* topk_w, int T, int l,
                int E, int k, uint16_t* z_perm, int32_t* counts, int32_t* offsets,
                int32_t* slot_of, int32_t* token_of, int32_t* tile_sched, float* row_w,
                void* ws, size_t ws_bytes, int32_t* err_flag, void* stream) {
  MOE_REQUIRE(topk_idx && counts && offsets && slot_of && token_of && tile_sched, MOE_ERR_ARG);
  MOE_REQUIRE(T >= 0 && E > 0 && E <= 1024 && k >= 1 && k <= 32 && k <= E, MOE_ERR_ARG);
  MOE_REQUIRE(static_cast<long long>(T) * k < (1ll << 31), MOE_ERR_ARG);
  if (z) {
    MOE_REQUIRE(z_perm != nullptr && l > 0, MOE_ERR_ARG);
    MOE_REQUIRE(l % 64 == 0 && al16(z) && al16(z_perm), MOE_ERR_ALIGN);
  }
  MOE_REQUIRE(ws != nullptr, MOE_ERR_WORKSPACE);
  MOE_REQUIRE(ws_bytes >= moe_workspace_size(MOE_OP_PERMUTE, T, 0, l, E, k, 0, 0),
              MOE_ERR_WORKSPACE);
  cudaStream_t st = S(stream);
  const float* tw = (topk_w && row_w) ? topk_w : nullptr;
  MOE_CHECK(cuda_status(launch_permute_maps(topk_idx, tw, T, E, k, reinterpret_cast<int*>(ws),
                                            counts, offsets, slot_of, token_of, tile_sched,
                                            tw ? row_w : nullptr, err_flag, st)));
  if (z) MOE_CHECK(cuda_status(launch_gather_rows("permute_gather", z, token_of, static_cast<long long>(T) * k, l,
                                                  z_perm, st)));
  return MOE_OK;
}

int moe_replica_plan(const int32_t* counts, int E, int P, int32_t* pieces, int32_t* n_pieces,
                     int32_t* rank_load, void* stream) {
  MOE_REQUIRE(counts && pieces && n_pieces && rank_load, MOE_ERR_ARG);
  MOE_REQUIRE(E > 0 && P > 0 && E % P == 0 && E + P <= 2048, MOE_ERR_ARG);
  return cuda_status(launch_replica_plan(counts, E, P, pieces, n_pieces, rank_load, S(stream)));
}

// ---------------------------------------------------------------- projections

int moe_latent_proj(const uint16_t* in, const uint16_t* W, int M, int K, int N, uint16_t* out,
                    void* stream) {
  MOE_REQUIRE(in && W && out, MOE_ERR_ARG);
  MOE_REQUIRE(M >= 0 && K > 0 && N > 0, MOE_ERR_ARG);
  MOE_REQUIRE(K % 64 == 0 && N % 64 == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(al16(in) && al16(W) && al16(out), MOE_ERR_ALIGN);
  if (M == 0) return MOE_OK;
  return dense_gemm("latent_proj_gemm", in, K, 0, W, N, 1, M, N, K, out, N, 1, 0, S(stream));
}

int moe_latent_proj_bwd(const uint16_t* dout, const uint16_t* in, const uint16_t* W, int M, int K,
                        int N, uint16_t* din, void* dW, int wgrad_dtype, void* stream) {
  MOE_REQUIRE(dout != nullptr, MOE_ERR_ARG);
  MOE_REQUIRE(M >= 0 && K > 0 && N > 0, MOE_ERR_ARG);
  MOE_REQUIRE(K % 64 == 0 && N % 64 == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(wgrad_dtype == MOE_DTYPE_F32 || wgrad_dtype == MOE_DTYPE_BF16, MOE_ERR_ARG);
  MOE_REQUIRE(!din || W != nullptr, MOE_ERR_ARG);
  MOE_REQUIRE(!din || (al16(dout) && al16(W) && al16(din)), MOE_ERR_ALIGN);
  MOE_REQUIRE(!dW || in != nullptr, MOE_ERR_ARG);
  MOE_REQUIRE(!dW || (al16(dout) && al16(in) && al16(dW)), MOE_ERR_ALIGN);
  cudaStream_t st = S(stream);
  if (din) {
    if (M > 0) MOE_CHECK(dense_gemm("latent_proj_dgrad", dout, N, 0, W, N, 0, M, K, N, din, K, 1, 0, st));
  }
  if (dW) {
    if (M == 0) {
      const size_t bytes = static_cast<size_t>(K) * N * (wgrad_dtype == MOE_DTYPE_F32 ? 4 : 2);
      return cuda_status(cudaMemsetAsync(dW, 0, bytes, st));
    }
    MOE_CHECK(dense_gemm("latent_proj_wgrad", in, K, 1, dout, N, 1, K, N, M, dW, N, wgrad_dtype == MOE_DTYPE_BF16, 0,
                         st));
  }
  return MOE_OK;
}

// ---------------------------------------------------------------- experts

}  // extern "C"

namespace {

// Grouped SwiGLU experts; A rows come from z_src ([src_rows][l]): permuted row r
// is z_src row gather[r] when gather is given, else row r.
// The FP8 cache of g|u (E4M3 bytes [R][2f] and fp32 scales [R][2f/64]) takes
// the place of the bf16 gu_save when its pointers are given.
struct Fp8Cache {
  uint8_t* gu8 = nullptr;
  float* scale = nullptr;
};

int grouped_swiglu_impl(const uint16_t* z_perm, long long src_rows, const int32_t* gather,
                        const uint16_t* W13, const uint16_t* W2, const int32_t* offsets,
                        const int32_t* tile_sched, const float* row_w, int E, int R, int l, int f,
                        uint16_t* gu_save, uint16_t* h, uint16_t* y_perm, void* stream,
                        const int32_t* expert_order = nullptr, Fp8Cache fp8 = Fp8Cache()) {
  MOE_REQUIRE(z_perm && W13 && W2 && offsets && tile_sched && h && y_perm, MOE_ERR_ARG);
  MOE_REQUIRE(E > 0 && R >= 0 && l > 0 && f > 0, MOE_ERR_ARG);
  MOE_REQUIRE(l % 64 == 0 && f % 64 == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(al16(z_perm) && al16(W13) && al16(W2) && al16(h) && al16(y_perm) &&
                  (!gu_save || al16(gu_save)) && (!fp8.gu8 || al16(fp8.gu8)),
              MOE_ERR_ALIGN);
  // the FP8 cache's 64-feature blocks are halves of the 128-feature n tiles
  MOE_REQUIRE(!fp8.gu8 || (fp8.scale && f % 128 == 0 && !gu_save), MOE_ERR_UNSUPPORTED);
  if (R == 0) return MOE_OK;
  cudaStream_t st = S(stream);
  // GEMM1 + SwiGLU: [g|u] = z_perm W13[e]; h = silu(g) * u
  GemmLaunch L1;
  L1.name = "expert_gemm1_swiglu";
  L1.BN = (f % 128 == 0) ? 256 : 128;
  L1.sched = SCHED_GROUPED_M;
  L1.G = E;
  L1.offsets = offsets;
  L1.tile_sched = tile_sched;
  L1.expert_order = expert_order;
  L1.R_cap = R;
  L1.N = f;
  L1.K = l;
  L1.A = view(z_perm, src_rows, l, l);
  L1.a_mn = 0;
  L1.gather_idx = gather;
  L1.gather_a = gather != nullptr;
  L1.B = view(W13, l, 2ll * f, 2ll * f, E, static_cast<long long>(l) * 2 * f);
  L1.b_mn = 1;
  L1.b_batch_mode = BATCH_GROUP;
  L1.swiglu_b = 1;
  L1.f = f;
  L1.n_tiles = f / (L1.BN / 2);
  L1.epi = EPI_SWIGLU;
  L1.h = h;
  L1.ldh = f;
  L1.gu = gu_save;
  L1.ldgu = 2ll * f;
  L1.gu8 = fp8.gu8;
  L1.gu_scale = fp8.scale;
  L1.ld_scale = 2 * f / 64;
  MOE_CHECK(gemm_launch(L1, st));
  // GEMM2 + routing-weight scale: y_perm = row_w * (h W2[e])
  GemmLaunch L2;
  L2.name = "expert_gemm2_rowscale";
  L2.BN = pick_bn(l);
  L2.sched = SCHED_GROUPED_M;
  L2.G = E;
  L2.offsets = offsets;
  L2.tile_sched = tile_sched;
  L2.expert_order = expert_order;
  L2.R_cap = R;
  L2.N = l;
  L2.K = f;
  L2.A = view(h, R, f, f);
  L2.a_mn = 0;
  L2.B = view(W2, f, l, l, E, static_cast<long long>(f) * l);
  L2.b_mn = 1;
  L2.b_batch_mode = BATCH_GROUP;
  L2.epi = EPI_ROWSCALE;
  L2.row_w = row_w;
  L2.C = y_perm;
  L2.ldc = l;
  return gemm_launch(L2, st);
}

}  // namespace

extern "C" {

int moe_grouped_swiglu(const uint16_t* z_perm, const uint16_t* W13, const uint16_t* W2,
                       const int32_t* offsets, const int32_t* tile_sched, const float* row_w,
                       int E, int R, int l, int f, uint16_t* gu_save, uint16_t* h,
                       uint16_t* y_perm, void* stream) {
  return grouped_swiglu_impl(z_perm, R, nullptr, W13, W2, offsets, tile_sched, row_w, E, R, l, f,
                             gu_save, h, y_perm, stream);
}

int moe_grouped_swiglu_fp8cache(const uint16_t* z_perm, const uint16_t* W13, const uint16_t* W2,
                                const int32_t* offsets, const int32_t* tile_sched,
                                const float* row_w, int E, int R, int l, int f, uint8_t* gu8,
                                float* gu_scale, uint16_t* h, uint16_t* y_perm, void* stream) {
  MOE_REQUIRE(gu8 && gu_scale, MOE_ERR_ARG);
  Fp8Cache c;
  c.gu8 = gu8;
  c.scale = gu_scale;
  return grouped_swiglu_impl(z_perm, R, nullptr, W13, W2, offsets, tile_sched, row_w, E, R, l, f,
                             nullptr, h, y_perm, stream, nullptr, c);
}

int moe_expert_buckets(const int32_t* counts, int E, int32_t* expert_order,
                       int32_t* tile_sched_ordered, void* stream) {
  MOE_REQUIRE(counts && expert_order && tile_sched_ordered, MOE_ERR_ARG);
  MOE_REQUIRE(E > 0 && E <= 1024, MOE_ERR_ARG);
  return cuda_status(launch_bucket_order(counts, E, expert_order, tile_sched_ordered, S(stream)));
}

int moe_grouped_swiglu_ordered(const uint16_t* z_perm, const uint16_t* W13, const uint16_t* W2,
                               const int32_t* offsets, const int32_t* tile_sched_ordered,
                               const int32_t* expert_order, const float* row_w, int E, int R,
                               int l, int f, uint16_t* gu_save, uint16_t* h, uint16_t* y_perm,
                               void* stream) {
  MOE_REQUIRE(expert_order != nullptr, MOE_ERR_ARG);
  return grouped_swiglu_impl(z_perm, R, nullptr, W13, W2, offsets, tile_sched_ordered, row_w, E, R,
                             l, f, gu_save, h, y_perm, stream, expert_order);
}

int moe_grouped_swiglu_gather(const uint16_t* z, const int32_t* token_of, int T,
                              const uint16_t* W13, const uint16_t* W2, const int32_t* offsets,
                              const int32_t* tile_sched, const float* row_w, int E, int R, int l,
                              int f, uint16_t* gu_save, uint16_t* h, uint16_t* y_perm,
                              void* stream) {
  MOE_REQUIRE(token_of != nullptr && T > 0, MOE_ERR_ARG);
  return grouped_swiglu_impl(z, T, token_of, W13, W2, offsets, tile_sched, row_w, E, R, l, f,
                             gu_save, h, y_perm, stream);
}

int moe_shared_swiglu(const uint16_t* z, const uint16_t* W13_sh, const uint16_t* W2_sh, int T,
                      int l, int f, int S_, uint16_t* gu_save, uint16_t* h, uint16_t* y_sh,
                      void* stream) {
  MOE_REQUIRE(z && W13_sh && W2_sh && h && y_sh, MOE_ERR_ARG);
  MOE_REQUIRE(T >= 0 && l > 0 && f > 0 && S_ >= 1, MOE_ERR_ARG);
  MOE_REQUIRE(l % 64 == 0 && f % 64 == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(al16(z) && al16(W13_sh) && al16(W2_sh) && al16(h) && al16(y_sh) &&
                  (!gu_save || al16(gu_save)),
              MOE_ERR_ALIGN);
  if (T == 0) return MOE_OK;
  cudaStream_t st = S(stream);
  GemmLaunch L1;
  L1.name = "shared_gemm1_swiglu";
  L1.BN = (f % 128 == 0) ? 256 : 128;
  L1.sched = SCHED_DENSE;
  L1.M = T;
  L1.N = S_ * f;
  L1.K = l;
  L1.A = view(z, T, l, l);
  L1.B = view(W13_sh, l, 2ll * f, 2ll * f, S_, static_cast<long long>(l) * 2 * f);
  L1.b_mn = 1;
  L1.b_batch_mode = BATCH_FROM_N;
  L1.n_tiles_per_batch = f / (L1.BN / 2);
  L1.n_tiles = S_ * L1.n_tiles_per_batch;
  L1.swiglu_b = 1;
  L1.f = f;
  L1.epi = EPI_SWIGLU;
  L1.h = h;
  L1.ldh = static_cast<long long>(S_) * f;
  L1.gu = gu_save;
  L1.ldgu = 2ll * S_ * f;
  MOE_CHECK(gemm_launch(L1, st));
  // y_sh = [h_0 | h_1 | ...] @ [W2_0; W2_1; ...]: one GEMM with K = S*f
  return dense_gemm("shared_gemm2", h, static_cast<long long>(S_) * f, 0, W2_sh, l, 1, T, l, S_ * f,
                    y_sh, l, 1, 0, st);
}

// ---------------------------------------------------------------- combine

int moe_unpermute_combine(const uint16_t* y_perm, const int32_t* slot_of,
                          const uint16_t* y_shared, int T, int k, int l, uint16_t* y_lat,
                          void* stream) {
  MOE_REQUIRE(y_perm && slot_of && y_lat, MOE_ERR_ARG);
  MOE_REQUIRE(T >= 0 && k >= 1 && k <= 32 && l > 0, MOE_ERR_ARG);
  MOE_REQUIRE(l % 64 == 0 && al16(y_perm) && al16(y_lat) && (!y_shared || al16(y_shared)),
              MOE_ERR_ALIGN);
  return cuda_status(launch_gather_sum("combine", y_perm, slot_of, k, y_shared, T, l, y_lat, l, S(stream)));
}

int moe_unpermute_combine_bwd(const uint16_t* dy_lat, const int32_t* token_of, int T, int k, int l,
                              uint16_t* dy_perm, void* stream) {
  MOE_REQUIRE(dy_lat && token_of && dy_perm, MOE_ERR_ARG);
  MOE_REQUIRE(T >= 0 && k >= 1 && k <= 32 && l > 0, MOE_ERR_ARG);
  MOE_REQUIRE(l % 64 == 0 && al16(dy_lat) && al16(dy_perm), MOE_ERR_ALIGN);
  return cuda_status(
      launch_gather_rows("combine_bwd_gather", dy_lat, token_of, static_cast<long long>(T) * k, l, dy_perm, S(stream)));
}

int moe_permute_bwd(const uint16_t* dz_perm, const int32_t* slot_of, const uint16_t* dz_shared,
                    int T, int k, int l, uint16_t* dz, void* stream) {
  MOE_REQUIRE(dz_perm && slot_of && dz, MOE_ERR_ARG);
  MOE_REQUIRE(T >= 0 && k >= 1 && k <= 32 && l > 0, MOE_ERR_ARG);
  MOE_REQUIRE(l % 64 == 0 && al16(dz_perm) && al16(dz) && (!dz_shared || al16(dz_shared)),
              MOE_ERR_ALIGN);
  return cuda_status(
      launch_gather_sum("permute_bwd_sum", dz_perm, slot_of, k, dz_shared, T, l, dz, l, S(stream)));
}

// ---------------------------------------------------------------- backward

}  // extern "C"

namespace {

// Backward of the grouped experts; dy and z rows come from [src_rows][l]
// sources, permuted row r being source row gather[r] when gather is given.
int grouped_swiglu_bwd_impl(const uint16_t* dy_perm, const uint16_t* z_perm, long long src_rows,
                            const int32_t* gather, const uint16_t* W13, const uint16_t* W2,
                            const uint16_t* gu_save, const uint16_t* h, const float* row_w,
                            const int32_t* offsets, const int32_t* tile_sched, int E, int R, int l,
                            int f, uint16_t* dz_perm, float* d_row_w, void* dW13, void* dW2,
                            int wgrad_dtype, void* ws, size_t ws_bytes, void* stream,
                            Fp8Cache fp8 = Fp8Cache()) {
  MOE_REQUIRE(dy_perm && z_perm && W13 && W2 && h && offsets && tile_sched && dz_perm && d_row_w &&
                  dW13 && dW2,
              MOE_ERR_ARG);
  MOE_REQUIRE((gu_save != nullptr) != (fp8.gu8 != nullptr), MOE_ERR_UNSUPPORTED);
  MOE_REQUIRE(!fp8.gu8 || (fp8.scale && f % 64 == 0), MOE_ERR_UNSUPPORTED);
  MOE_REQUIRE(E > 0 && R >= 0 && l > 0 && f > 0, MOE_ERR_ARG);
  MOE_REQUIRE(wgrad_dtype == MOE_DTYPE_F32 || wgrad_dtype == MOE_DTYPE_BF16, MOE_ERR_ARG);
  MOE_REQUIRE(l % 64 == 0 && f % 64 == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(al16(dy_perm) && al16(z_perm) && al16(W13) && al16(W2) && al16(gu_save) &&
                  al16(fp8.gu8) && al16(h) &&
                  al16(dz_perm) && al16(dW13) && al16(dW2),
              MOE_ERR_ALIGN);
  MOE_REQUIRE(ws != nullptr && ws_bytes >= grouped_bwd_ws(R, f), MOE_ERR_WORKSPACE);
  cudaStream_t st = S(stream);
  const int wbf16 = wgrad_dtype == MOE_DTYPE_BF16;
  if (R == 0) {  // no rows at all: every expert gradient is zero
    const size_t es = wbf16 ? 2 : 4;
    MOE_CHECK(cuda_status(cudaMemsetAsync(dW13, 0, static_cast<size_t>(E) * l * 2 * f * es, st)));
    return cuda_status(cudaMemsetAsync(dW2, 0, static_cast<size_t>(E) * f * l * es, st));
  }
  WsCarver wc{reinterpret_cast<char*>(ws), ws_bytes};
  uint16_t* dgu = reinterpret_cast<uint16_t*>(wc.take(static_cast<size_t>(R) * 2 * f * 2));
  uint16_t* hw = reinterpret_cast<uint16_t*>(wc.take(static_cast<size_t>(R) * f * 2));
  float* dw_part =
      reinterpret_cast<float*>(wc.take(static_cast<size_t>(R) * 2 * ((f + 127) / 128) * 4));
  MOE_REQUIRE(wc.ok, MOE_ERR_WORKSPACE);
  // 1. dgrad through W2 with the SwiGLU backward and routing-weight dots fused
  GemmLaunch D2;
  D2.name = "expert_dgrad2_swiglu_bwd";
  D2.BN = pick_bn(f);
  D2.sched = SCHED_GROUPED_M;
  D2.G = E;
  D2.offsets = offsets;
  D2.tile_sched = tile_sched;
  D2.R_cap = R;
  D2.N = f;
  D2.K = l;
  D2.A = view(dy_perm, src_rows, l, l);
  D2.gather_idx = gather;
  D2.gather_a = gather != nullptr;
  D2.B = view(W2, f, l, l, E, static_cast<long long>(f) * l);  // B[n=f][k=l], K-major
  D2.b_mn = 0;
  D2.b_batch_mode = BATCH_GROUP;
  D2.f = f;
  D2.epi = EPI_SWIGLU_BWD;
  D2.C = dgu;
  D2.ldc = 2ll * f;
  D2.gu = const_cast<uint16_t*>(gu_save);
  D2.ldgu = 2ll * f;
  D2.gu8 = fp8.gu8;
  D2.gu_scale = fp8.scale;
  D2.ld_scale = 2 * f / 64;
  D2.h = const_cast<uint16_t*>(h);
  D2.ldh = f;
  D2.row_w = row_w;
  D2.aux = hw;
  D2.ldaux = f;
  D2.dw_part = dw_part;
  D2.dw_nparts = (gemm_epilogue_warps(D2) / 4) * ((f + D2.BN - 1) / D2.BN);
  if (R > 0) MOE_CHECK(gemm_launch(D2, st));
  MOE_CHECK(cuda_status(launch_dw_reduce(dw_part, D2.dw_nparts, R, d_row_w, st)));
  // 2. dW2[e] = (row_w h)^T dy_perm over the expert's rows (ragged K)
  GemmLaunch W2g;
  W2g.name = "expert_wgrad2";
  W2g.BN = pick_bn(l);
  W2g.sched = SCHED_GROUPED_K;
  W2g.G = E;
  W2g.offsets = offsets;
  W2g.M = f;
  W2g.N = l;
  W2g.A = view(hw, R, f, f);
  W2g.a_mn = 1;
  W2g.B = view(dy_perm, src_rows, l, l);
  W2g.b_mn = 1;
  W2g.gather_idx = gather;
  W2g.gather_b = gather != nullptr;
  W2g.epi = EPI_STORE;
  W2g.C = dW2;
  W2g.ldc = l;
  W2g.c_batch_stride = static_cast<long long>(f) * l;
  W2g.c_bf16 = wbf16;
  MOE_CHECK(gemm_launch(W2g, st));
  // 3. dz_perm = [dg|du] W13[e]^T
  GemmLaunch D1;
  D1.name = "expert_dgrad1";
  D1.BN = pick_bn(l);
  D1.sched = SCHED_GROUPED_M;
  D1.G = E;
  D1.offsets = offsets;
  D1.tile_sched = tile_sched;
  D1.R_cap = R;
  D1.N = l;
  D1.K = 2 * f;
  D1.A = view(dgu, R, 2ll * f, 2ll * f);
  D1.B = view(W13, l, 2ll * f, 2ll * f, E, static_cast<long long>(l) * 2 * f);  // [n=l][k=2f]
  D1.b_mn = 0;
  D1.b_batch_mode = BATCH_GROUP;
  D1.epi = EPI_STORE;
  D1.C = dz_perm;
  D1.ldc = l;
  D1.c_bf16 = 1;
  if (R > 0) MOE_CHECK(gemm_launch(D1, st));
  // 4. dW13[e] = z_perm^T [dg|du] over the expert's rows (ragged K)
  GemmLaunch W1g;
  W1g.name = "expert_wgrad1";
  W1g.BN = pick_bn(2 * f);
  W1g.sched = SCHED_GROUPED_K;
  W1g.G = E;
  W1g.offsets = offsets;
  W1g.M = l;
  W1g.N = 2 * f;
  W1g.A = view(z_perm, src_rows, l, l);
  W1g.a_mn = 1;
  W1g.gather_idx = gather;
  W1g.gather_a = gather != nullptr;
  W1g.B = view(dgu, R, 2ll * f, 2ll * f);
  W1g.b_mn = 1;
  W1g.epi = EPI_STORE;
  W1g.C = dW13;
  W1g.ldc = 2ll * f;
  W1g.c_batch_stride = static_cast<long long>(l) * 2 * f;
  W1g.c_bf16 = wbf16;
  return gemm_launch(W1g, st);
}

}  // namespace

extern "C" {

int moe_grouped_swiglu_bwd(const uint16_t* dy_perm, const uint16_t* z_perm, const uint16_t* W13,
                           const uint16_t* W2, const uint16_t* gu_save, const uint16_t* h,
                           const float* row_w, const int32_t* offsets, const int32_t* tile_sched,
                           int E, int R, int l, int f, uint16_t* dz_perm, float* d_row_w,
                           void* dW13, void* dW2, int wgrad_dtype, void* ws, size_t ws_bytes,
                           void* stream) {
  return grouped_swiglu_bwd_impl(dy_perm, z_perm, R, nullptr, W13, W2, gu_save, h, row_w, offsets,
                                 tile_sched, E, R, l, f, dz_perm, d_row_w, dW13, dW2, wgrad_dtype,
                                 ws, ws_bytes, stream);
}

int moe_grouped_swiglu_bwd_fp8cache(const uint16_t* dy_perm, const uint16_t* z_perm,
                                    const uint16_t* W13, const uint16_t* W2, const uint8_t* gu8,
                                    const float* gu_scale, const uint16_t* h, const float* row_w,
                                    const int32_t* offsets, const int32_t* tile_sched, int E,
                                    int R, int l, int f, uint16_t* dz_perm, float* d_row_w,
                                    void* dW13, void* dW2, int wgrad_dtype, void* ws,
                                    size_t ws_bytes, void* stream) {
  MOE_REQUIRE(gu8 && gu_scale, MOE_ERR_ARG);
  Fp8Cache c;
  c.gu8 = const_cast<uint8_t*>(gu8);
  c.scale = const_cast<float*>(gu_scale);
  return grouped_swiglu_bwd_impl(dy_perm, z_perm, R, nullptr, W13, W2, nullptr, h, row_w, offsets,
                                 tile_sched, E, R, l, f, dz_perm, d_row_w, dW13, dW2, wgrad_dtype,
                                 ws, ws_bytes, stream, c);
}

int moe_grouped_swiglu_bwd_gather(const uint16_t* dy_lat, const uint16_t* z,
                                  const int32_t* token_of, int T, const uint16_t* W13,
                                  const uint16_t* W2, const uint16_t* gu_save, const uint16_t* h,
                                  const float* row_w, const int32_t* offsets,
                                  const int32_t* tile_sched, int E, int R, int l, int f,
                                  uint16_t* dz_perm, float* d_row_w, void* dW13, void* dW2,
                                  int wgrad_dtype, void* ws, size_t ws_bytes, void* stream) {
  MOE_REQUIRE(token_of != nullptr && T > 0, MOE_ERR_ARG);
  return grouped_swiglu_bwd_impl(dy_lat, z, T, token_of, W13, W2, gu_save, h, row_w, offsets,
                                 tile_sched, E, R, l, f, dz_perm, d_row_w, dW13, dW2, wgrad_dtype,
                                 ws, ws_bytes, stream);
}

int moe_shared_swiglu_bwd(const uint16_t* dy, const uint16_t* z, const uint16_t* W13_sh,
                          const uint16_t* W2_sh, const uint16_t* gu_save, const uint16_t* h,
                          int T, int l, int f, int S_, uint16_t* dz_sh, void* dW13_sh,
                          void* dW2_sh, int wgrad_dtype, void* ws, size_t ws_bytes,
                          void* stream) {
  MOE_REQUIRE(dy && z && W13_sh && W2_sh && gu_save && h && dz_sh && dW13_sh && dW2_sh,
              MOE_ERR_ARG);
  MOE_REQUIRE(T >= 0 && l > 0 && f > 0 && S_ >= 1, MOE_ERR_ARG);
  MOE_REQUIRE(wgrad_dtype == MOE_DTYPE_F32 || wgrad_dtype == MOE_DTYPE_BF16, MOE_ERR_ARG);
  MOE_REQUIRE(l % 64 == 0 && f % 64 == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(al16(dy) && al16(z) && al16(W13_sh) && al16(W2_sh) && al16(gu_save) && al16(h) &&
                  al16(dz_sh) && al16(dW13_sh) && al16(dW2_sh),
              MOE_ERR_ALIGN);
  MOE_REQUIRE(ws != nullptr && ws_bytes >= shared_bwd_ws(T, l, f, S_), MOE_ERR_WORKSPACE);
  cudaStream_t st = S(stream);
  const int wbf16 = wgrad_dtype == MOE_DTYPE_BF16;
  const long long Sf = static_cast<long long>(S_) * f;
  if (T == 0) {
    const size_t es = wbf16 ? 2 : 4;
    MOE_CHECK(cuda_status(cudaMemsetAsync(dW13_sh, 0, static_cast<size_t>(S_) * l * 2 * f * es, st)));
    return cuda_status(cudaMemsetAsync(dW2_sh, 0, static_cast<size_t>(Sf) * l * es, st));
  }
  uint16_t* dgu = reinterpret_cast<uint16_t*>(ws);
  float* split_ws = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) +
                                             up256(static_cast<size_t>(T) * Sf * 2 * 2));
  // 1. dh = dy W2_sh^T (all shared experts at once), SwiGLU backward fused
  GemmLaunch D2;
  D2.name = "shared_dgrad2_swiglu_bwd";
  D2.BN = pick_bn(static_cast<int>(Sf));
  D2.sched = SCHED_DENSE;
  D2.M = T;
  D2.N = static_cast<int>(Sf);
  D2.K = l;
  D2.A = view(dy, T, l, l);
  D2.B = view(W2_sh, Sf, l, l);  // B[n=S*f][k=l], K-major
  D2.b_mn = 0;
  D2.f = f;
  D2.epi = EPI_SWIGLU_BWD;
  D2.C = dgu;
  D2.ldc = 2 * Sf;
  D2.gu = const_cast<uint16_t*>(gu_save);
  D2.ldgu = 2 * Sf;
  D2.h = const_cast<uint16_t*>(h);
  D2.ldh = Sf;
  MOE_CHECK(gemm_launch(D2, st));
  // 2. dW2_sh [S*f][l] = h^T dy (K = T split into slices when there are few tiles)
  {
    GemmLaunch W2s;
    W2s.name = "shared_wgrad2";
    W2s.BN = pick_bn(l);
    W2s.sched = SCHED_DENSE;
    W2s.M = static_cast<int>(Sf);
    W2s.N = l;
    W2s.K = T;
    W2s.A = view(h, T, Sf, Sf);
    W2s.a_mn = 1;
    W2s.B = view(dy, T, l, l);
    W2s.b_mn = 1;
    W2s.epi = EPI_STORE;
    W2s.C = dW2_sh;
    W2s.ldc = l;
    W2s.c_bf16 = wbf16;
    W2s.splitk = wgrad_splitk(W2s.M, W2s.N, T);
    W2s.splitk_ws = split_ws;
    MOE_CHECK(gemm_launch(W2s, st));
  }
  // 3. dz_sh = sum_s [dg_s|du_s] W13_sh[s]^T: one GEMM with K = S*2f, B batch from K
  GemmLaunch D1;
  D1.name = "shared_dgrad1";
  D1.BN = pick_bn(l);
  D1.sched = SCHED_DENSE;
  D1.M = T;
  D1.N = l;
  D1.K = static_cast<int>(2 * Sf);
  D1.A = view(dgu, T, 2 * Sf, 2 * Sf);
  D1.B = view(W13_sh, l, 2ll * f, 2ll * f, S_, static_cast<long long>(l) * 2 * f);
  D1.b_mn = 0;
  D1.b_batch_mode = BATCH_FROM_K;
  D1.k_per_batch = 2 * f;
  D1.epi = EPI_STORE;
  D1.C = dz_sh;
  D1.ldc = l;
  D1.c_bf16 = 1;
  MOE_CHECK(gemm_launch(D1, st));
  // 4. dW13_sh[s] = z^T [dg_s|du_s]: one GEMM over N = S*2f, output block s at s*l*2f
  GemmLaunch W1g;
  W1g.name = "shared_wgrad1";
  W1g.BN = pick_bn(2 * f);
  W1g.sched = SCHED_DENSE;
  W1g.M = l;
  W1g.N = static_cast<int>(2 * Sf);
  W1g.K = T;
  W1g.A = view(z, T, l, l);
  W1g.a_mn = 1;
  W1g.B = view(dgu, T, 2 * Sf, 2 * Sf);
  W1g.b_mn = 1;
  W1g.epi = EPI_STORE;
  W1g.C = dW13_sh;
  W1g.ldc = 2ll * f;
  W1g.c_batch_n = 2 * f;
  W1g.c_batch_stride = static_cast<long long>(l) * 2 * f;
  W1g.c_bf16 = wbf16;
  W1g.splitk = wgrad_splitk(W1g.M, W1g.N, T);
  W1g.splitk_ws = split_ws;
  return gemm_launch(W1g, st);
}

int moe_route_topk_bwd(const float* d_row_w, const int32_t* slot_of, const int32_t* topk_idx,
                       const float* topk_w, const float* topk_s, const uint16_t* x,
                       const uint16_t* Wr, int T, int d, int E, int k, float* d_topk_w,
                       uint16_t* dx_accum, void* dWr, int wgrad_dtype, const float* aux_logits,
                       const float* aux_bias, const float* aux_p_mean, float aux_scale,
                       const uint16_t* dz, const uint16_t* W_dn, int l, void* ws,
                       size_t ws_bytes, int32_t* err_flag, void* stream) {
  MOE_REQUIRE(d_row_w && slot_of && topk_idx && topk_w && topk_s, MOE_ERR_ARG);
  MOE_REQUIRE(T >= 0 && d > 0 && E > 0 && E <= 1024 && k >= 1 && k <= 32 && k <= E, MOE_ERR_ARG);
  MOE_REQUIRE(wgrad_dtype == MOE_DTYPE_F32 || wgrad_dtype == MOE_DTYPE_BF16, MOE_ERR_ARG);
  MOE_REQUIRE(d % 64 == 0 && E % 64 == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(!(dx_accum && !Wr) && !(dWr && !x), MOE_ERR_ARG);
  MOE_REQUIRE(!dx_accum || (al16(dx_accum) && al16(Wr)), MOE_ERR_ALIGN);
  MOE_REQUIRE(!dWr || (al16(dWr) && al16(x)), MOE_ERR_ALIGN);
  MOE_REQUIRE(!aux_logits || aux_p_mean != nullptr, MOE_ERR_ARG);
  if (dx_accum && dz) {  // the fused input gradient dx = dz W_dn^T + dL Wr^T
    MOE_REQUIRE(W_dn != nullptr && l > 0, MOE_ERR_ARG);
    MOE_REQUIRE(l % 64 == 0 && al16(dz) && al16(W_dn), MOE_ERR_ALIGN);
  }
  MOE_REQUIRE(ws != nullptr && ws_bytes >= moe_workspace_size(MOE_OP_ROUTE_TOPK_BWD, T, d, 0, E, k, 0, 0),
              MOE_ERR_WORKSPACE);
  cudaStream_t st = S(stream);
  if (T == 0) {
    if (dWr)
      return cuda_status(cudaMemsetAsync(
          dWr, 0, static_cast<size_t>(d) * E * (wgrad_dtype == MOE_DTYPE_F32 ? 4 : 2), st));
    return MOE_OK;
  }
  uint16_t* dL = reinterpret_cast<uint16_t*>(ws);
  MOE_CHECK(cuda_status(launch_router_bwd(d_row_w, slot_of, topk_idx, topk_w, topk_s, T, E, k,
                                          d_topk_w, dL, err_flag, st)));
  if (aux_logits) {
    MOE_CHECK(cuda_status(launch_aux_bwd(aux_logits, aux_bias, aux_p_mean, T, E, aux_scale, dL, st)));
  }
  if (dx_accum && dz) {
    // dx = dz @ W_dn^T + dL @ Wr^T as one GEMM over K = l + E (overwrites dx)
    GemmLaunch L;
    L.name = "down_proj_router_dgrad";
    L.BN = pick_bn(d);
    L.sched = SCHED_DENSE;
    L.M = T;
    L.N = d;
    L.K = l + E;
    L.A = view(dz, T, l, l);
    L.B = view(W_dn, d, l, l);      // B[n = d][k = l], K-major
    L.kcat = l;
    L.A2 = view(dL, T, E, E);
    L.B2 = view(Wr, d, E, E);       // B2[n = d][k = E], K-major
    L.epi = EPI_STORE;
    L.C = dx_accum;
    L.ldc = d;
    L.c_bf16 = 1;
    MOE_CHECK(gemm_launch(L, st));
  } else if (dx_accum) {
    MOE_CHECK(dense_gemm("router_dgrad", dL, E, 0, Wr, E, 0, T, d, E, dx_accum, d, 1, 1, st));
  }
  if (dWr)
    MOE_CHECK(dense_gemm("router_wgrad", x, d, 1, dL, E, 1, d, E, T, dWr, E, wgrad_dtype == MOE_DTYPE_BF16, 0, st));
  return MOE_OK;
}

}  // extern "C"
