/*
 * libmoe - GB300 (sm_103a) hot path of a LatentMoE sparse expert layer:
 * sigmoid router with top-k selection, token permute, latent projections,
 * grouped SwiGLU experts over ragged expert batches, weighted combine, and
 * the backward of each step.
 *
 * Sources. The pages that describe this layer give its structure, not its
 * formulas:
 *   [MODEL]   "TorchTitan Ascend开源:插件化支持TorchTitan,实现Kimi K3.1 Pro的昇腾适配与训练实践",
 *             section "Kimi K3.1 Pro 模型结构", LatentMoE paragraph: 896 routed and
 *             2 shared experts, 16 routed experts active per token, expert compute
 *             in a low-dimensional latent space.
 *   [OPS]     "昇腾实现Kimi K3.1 Pro模型LoRA训练适配,助力2.8万亿级大模型高效训练",
 *             section "MoE(Mixture of Experts):算子融合与通信协同": dynamic routing,
 *             token dispatch, and Permute / Unpermute / Grouped GEMM as the core
 *             operators, with less data movement during token reordering as a goal.
 *   [LOAD]    "TorchTitan Ascend开源 ...", section "在线负载规划": per-expert load is
 *             counted from the current routing result.
 *   [GGEMM]   same page, section "权重预取与梯度归约": one Grouped GEMM runs all
 *             experts of a device through a unified compute view.
 *   [SWAP]    the [OPS] page, section "Swap Core:算子级精准缓存与异步 Offload 协同,
 *             训练性能提升 15%": outputs of selected MatMul/GMM operators are cached
 *             for the backward, optionally compressed by FP8 activation
 *             quantization and dequantization.
 * Where the pages are silent the library takes these readings: the router is
 * sigmoid(x @ Wr (+ bias)) on the model-width input, the k largest logits are
 * selected (lower expert id wins a tie) and their sigmoids renormalised to sum
 * to 1; an expert is o = (silu(z Wg) * (z Wu)) W2 on the latent z = x W_dn; the
 * routing weight scales the expert output; the shared experts run on z with
 * weight 1; out = (sum_j w_j o_j + sum_s shared_s(z)) W_up; tokens of one expert
 * are kept in ascending token order; no token is dropped.
 *
 * Conventions of every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or synchronises. Pointers must be 16-byte aligned.
 *  - bf16 tensors are passed as uint16_t (bfloat16 bit patterns), row-major.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All work is enqueued on it; the call returns before the work runs.
 *  - Return value: MOE_OK or a negative MOE_ERR_* code. Argument errors are
 *    detected on the host before anything is enqueued. MOE_ERR_CUDA means a
 *    launch failed; moe_last_cuda_error() gives the cudaError_t.
 *  - Data errors found on the device (an expert id outside [0,E), a NaN/Inf
 *    logit, a kernel wait that timed out) OR bits into the caller's device
 *    word `err_flag` (nullable where listed) instead of trapping; the caller
 *    reads it when it chooses. Rows with a bad expert id are skipped.
 *  - Dimension limits: l, f, d multiples of 64; E <= 1024 (and a multiple of
 *    64 where a GEMM has E columns); 1 <= k <= min(E, 32); T*k < 2^31.
 *  - Index arrays that moe_permute writes (offsets, tile_sched, slot_of,
 *    token_of) are trusted by the calls that read them: pass them as written,
 *    or with the same invariants. A negative slot or token entry means "no
 *    row"; other entries are not range-checked on the device. Expert ids
 *    (topk_idx) are checked, as above.
 *  - Weight layouts: W13 [E][l][2f] (gate columns 0..f-1, up columns f..2f-1),
 *    W2 [E][f][l]; shared experts use the same layout with E -> S; Wr [d][E],
 *    W_dn [d][l], W_up [l][d].
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_ARG (-1)         /* null pointer or dimension out of range        */
#define MOE_ERR_ALIGN (-2)       /* pointer not 16-byte aligned / dim not x64      */
#define MOE_ERR_WORKSPACE (-3)   /* workspace smaller than moe_workspace_size()    */
#define MOE_ERR_UNSUPPORTED (-4) /* shape or option this build does not handle     */
#define MOE_ERR_CUDA (-5)        /* a CUDA call failed, see moe_last_cuda_error()  */

/* bits of the device error word */
#define MOE_FLAG_BAD_EXPERT 1 /* expert id outside [0, E) */
#define MOE_FLAG_NONFINITE 2  /* NaN or Inf router logit   */
#define MOE_FLAG_TIMEOUT 4    /* a kernel wait gave up     */

/* wgrad output types */
#define MOE_DTYPE_F32 0
#define MOE_DTYPE_BF16 1

/* operations with a workspace, for moe_workspace_size */
#define MOE_OP_ROUTE_TOPK 1
#define MOE_OP_PERMUTE 2
#define MOE_OP_GROUPED_SWIGLU_BWD 3
#define MOE_OP_SHARED_SWIGLU_BWD 4
#define MOE_OP_ROUTE_TOPK_BWD 5
#define MOE_OP_ROUTER_AUX 6

int moe_version(void);
const char* moe_status_string(int status);
int moe_last_cuda_error(void);

/* Bytes of workspace `op` needs for these sizes (unused sizes may be 0).
 * The workspace is device memory owned by the caller, 256-byte aligned. */
size_t moe_workspace_size(int op, int T, int d, int l, int E, int k, int f, int S);

/* ---------------------------------------------------------------- routing */

/* Router logits L[T][E] (fp32) = x[T][d] @ Wr[d][E] (bf16 in, fp32 accumulate),
 * the router of [OPS] "dynamic routing" read as a linear scorer on x.
 * E must be a multiple of 64. */
int moe_router_logits(const uint16_t* x, const uint16_t* Wr, int T, int d, int E, float* logits,
                      void* stream);

/* Top-k selection and weights from given fp32 logits ([MODEL]: 16 of 896).
 * For token t: v[e] = logits[t][e] + bias[e] (fp32 add; bias nullable);
 * topk_idx[t][j] (int32) lists the k largest v, ordered by (v desc, id asc);
 * topk_s[t][j] = sigmoid(v) (fp32); topk_w[t][j] = topk_s[t][j] / sum_j topk_s[t][j].
 * A NaN/Inf v sets MOE_FLAG_NONFINITE. Any E <= 1024. err_flag nullable. */
int moe_topk_from_logits(const float* logits, const float* bias, int T, int E, int k,
                         int32_t* topk_idx, float* topk_w, float* topk_s, int32_t* err_flag,
                         void* stream);

/* moe_router_logits followed by moe_topk_from_logits; the logits live in the
 * workspace (moe_workspace_size(MOE_OP_ROUTE_TOPK, T, 0, 0, E, 0, 0, 0) bytes). */
int moe_route_topk(const uint16_t* x, const uint16_t* Wr, const float* bias, int T, int d, int E,
                   int k, int32_t* topk_idx, float* topk_w, float* topk_s, void* ws,
                   size_t ws_bytes, int32_t* err_flag, void* stream);

/* moe_route_topk and the latent down-projection z[T][l] (bf16) = x @ W_dn[d][l]
 * ([MODEL]: experts computed in the latent space; the projection reads the same x)
 * in one call: when T > 128 and E is a multiple of 128 one GEMM over [Wr | W_dn]
 * reads x once (logits and z are bit-identical to the two separate calls), else
 * moe_router_logits + moe_latent_proj. Same workspace as moe_route_topk (the
 * logits stay in it); l a multiple of 64; z 16-byte aligned. */
int moe_route_topk_latent(const uint16_t* x, const uint16_t* Wr, const float* bias,
                          const uint16_t* W_dn, int T, int d, int E, int k, int l,
                          int32_t* topk_idx, float* topk_w, float* topk_s, uint16_t* z, void* ws,
                          size_t ws_bytes, int32_t* err_flag, void* stream);

/* Auxiliary load-balance loss of the routing stage ("大模型落地昇腾" page, section
 * "三、通信侧": an auxiliary loss that constrains the entropy of the routing
 * distribution), read as the negative entropy of the batch's mean routing
 * distribution over all experts:
 *   P(e|t) = s[t][e] / sum_e' s[t][e'],  s = sigmoid(logits + bias)   (bias nullable)
 *   p_mean[e] = (1/T) sum_t P(e|t)  (fp32, E);  loss = sum_e p_mean[e] ln p_mean[e]  (fp32, 1)
 * The loss is -ln E when the routing mass is spread evenly. Deterministic
 * (fixed-order reductions). Workspace: moe_workspace_size(MOE_OP_ROUTER_AUX, T, 0, 0, E, ...).
 * Its gradient is added by moe_route_topk_bwd (aux_* arguments). */
int moe_router_aux_loss(const float* logits, const float* bias, int T, int E, float* p_mean,
                        float* loss, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- permute */

/* Token Permute of [OPS] with the per-expert load count of [LOAD].
 *   counts[e]      = #{(t,j) : topk_idx[t][j] == e}                      (int32, E)
 *   offsets[e]     = counts[0] + ... + counts[e-1]; offsets[E] = total  (int32, E+1)
 *   slot_of[t][j]  = offsets[e] + #{t' < t : e in topk_idx[t']}, e = topk_idx[t][j]
 *                    (tokens of one expert in ascending token order; -1 for a bad id)
 *   token_of[r]    = t with slot_of[t][j] == r (int32, T*k; -1 past offsets[E])
 *   tile_sched[e]  = sum_{e'<e} ceil(counts[e'] / 128) (int32, E+1): the 128-row
 *                    tile ranges the grouped GEMMs walk on the device
 *   row_w[r]       = topk_w[t][j] for r = slot_of[t][j] (fp32 [T*k]; skipped when
 *                    topk_w or row_w is NULL): the routing weight of each permuted row
 *   z_perm[r][:]   = z[token_of[r]][:] (bf16 [T*k][l]); skipped when z is NULL.
 * The k ids of a token must be distinct (a repeat sets MOE_FLAG_BAD_EXPERT).
 * Deterministic, no atomics on the output. Workspace:
 * moe_workspace_size(MOE_OP_PERMUTE, T, 0, 0, E, 0, 0, 0). err_flag nullable. */
int moe_permute(const uint16_t* z, const int32_t* topk_idx, const float* topk_w, int T, int l,
                int E, int k, uint16_t* z_perm, int32_t* counts, int32_t* offsets,
                int32_t* slot_of, int32_t* token_of, int32_t* tile_sched, float* row_w,
                void* ws, size_t ws_bytes, int32_t* err_flag, void* stream);

/* Allocation-free variant of moe_permute, for callers that cannot allocate
 * device memory (a caller that is handed only its input and output buffers,
 * or one on a fixed memory budget that must not call cudaMalloc/cudaFree,
 * which may also synchronise the device). The pages describe nothing like it;
 * it computes exactly what moe_permute computes, with the same arguments
 * except ws / ws_bytes. Its scratch is a fixed 1 MiB array inside the library
 * (held on every GPU that loads the library until it is unloaded), so it
 * handles permute_chunks(T) * E <= 262144, i.e. ceil(T / 256) * E <= 262144
 * (T <= 74,752 at E = 896); larger problems return MOE_ERR_WORKSPACE without
 * launching anything. The first call on a device (and the first one after the
 * device's current CUDA context changed, e.g. after cudaDeviceReset) looks up
 * the array's device address; make that first call before any stream capture.
 * All calls share the array, which keeps the last call's contents (no entry of
 * it needs to start at zero): calls that may overlap on the GPU race on it and
 * must be serialised by the caller. MOE_ERR_CUDA, when the address lookup
 * fails, comes with its cause in moe_last_cuda_error(). */
int moe_permute_noalloc(const uint16_t* z, const int32_t* topk_idx, const float* topk_w, int T,
                        int l, int E, int k, uint16_t* z_perm, int32_t* counts, int32_t* offsets,
                        int32_t* slot_of, int32_t* token_of, int32_t* tile_sched, float* row_w,
                        int32_t* err_flag, void* stream);

/* Online load plan with dynamic expert replicas for an expert-parallel layout
 * ("TorchTitan Ascend开源" page, sections "在线负载规划" and
 * "MoonEP动态负载均衡与专家并行优化": per-expert loads of the current batch and
 * each device's remaining capacity decide the replicas of hot experts; a token
 * keeps its expert). Reading: P ranks, rank r owns experts [r*E/P, (r+1)*E/P)
 * (E divisible by P), every rank processes at most C = ceil(sum counts / P)
 * rows. Ranks first take their own experts' rows while they have room; the
 * rest of each expert goes, in rank order, to ranks with spare capacity.
 * Output: pieces[i][4] = {expert, rank, first row within the expert's
 * segment, rows} for i < *n_pieces (capacity 2E + P pieces, int32),
 * rank_load[P] = rows per rank (max = C). Runs on the device from the counts
 * of moe_permute (no host synchronisation). E + P <= 2048. Counts that are
 * negative or sum to 2^31 or more give *n_pieces = -1 and no plan. */
int moe_replica_plan(const int32_t* counts, int E, int P, int32_t* pieces, int32_t* n_pieces,
                     int32_t* rank_load, void* stream);

/* ---------------------------------------------------------------- projections */

/* Latent projection of [MODEL]: out[M][N] (bf16) = in[M][K] @ W[K][N] (bf16,
 * fp32 accumulate) on the tcgen05 tensor cores. K, N multiples of 64. */
int moe_latent_proj(const uint16_t* in, const uint16_t* W, int M, int K, int N, uint16_t* out,
                    void* stream);

/* Backward of moe_latent_proj for dout[M][N]:
 *   din[M][K] (bf16) = dout @ W^T      (skipped when din is NULL)
 *   dW[K][N]          = in^T @ dout    (skipped when dW is NULL; fp32 or bf16 per wgrad_dtype) */
int moe_latent_proj_bwd(const uint16_t* dout, const uint16_t* in, const uint16_t* W, int M, int K,
                        int N, uint16_t* din, void* dW, int wgrad_dtype, void* stream);

/* ---------------------------------------------------------------- experts */

/* Grouped SwiGLU experts over the permuted rows ([OPS] Grouped GEMM, [GGEMM]).
 * For every expert e and row r in [offsets[e], offsets[e+1]):
 *   [g|u][r] = z_perm[r] @ W13[e]              (fp32 accumulate)
 *   h[r]     = silu(g[r]) * u[r]               (bf16 [R][f])
 *   y_perm[r]= row_w[r] * (h[r] @ W2[e])       (bf16 [R][l]; row_w nullable => 1)
 *   gu_save[r] = [g|u][r] in bf16 ([R][2f], nullable) for the backward.
 * R is the row capacity of the buffers (>= offsets[E]); rows past offsets[E]
 * are not touched. offsets/tile_sched come from moe_permute. Empty experts
 * cost nothing (no tile, no weight read). No host synchronisation. */
int moe_grouped_swiglu(const uint16_t* z_perm, const uint16_t* W13, const uint16_t* W2,
                       const int32_t* offsets, const int32_t* tile_sched, const float* row_w,
                       int E, int R, int l, int f, uint16_t* gu_save, uint16_t* h,
                       uint16_t* y_perm, void* stream);

/* moe_grouped_swiglu with the GMM output [g|u] cached for the backward in FP8
 * ([SWAP]) instead of bf16: E4M3 (round to nearest even, saturating at +-448)
 * of g / s and u / s, with one power-of-two scale s per row and 64-feature block,
 * the smallest with max |block| <= 448 s (1 when that maximum is below 2^-100):
 *   gu8[r][32q + i]         E4M3 bytes [R][2f]: g[r][16q + i] (i < 16), u[r][16q + i - 16]
 *                           (16 <= i < 32): 16-feature groups of g and u in turn
 *   gu_scale[r][b]          fp32 [R][2f/64]: blocks of g (b < f/64), then of u
 * h and y_perm are exactly those of moe_grouped_swiglu. f must be a multiple of
 * 128 (MOE_ERR_UNSUPPORTED otherwise); gu8 16-byte aligned. The cache takes 1 + 1/16
 * bytes per value instead of 2. */
int moe_grouped_swiglu_fp8cache(const uint16_t* z_perm, const uint16_t* W13, const uint16_t* W2,
                                const int32_t* offsets, const int32_t* tile_sched,
                                const float* row_w, int E, int R, int l, int f, uint8_t* gu8,
                                float* gu_scale, uint16_t* h, uint16_t* y_perm, void* stream);

/* Multi-bucket batching ("大模型落地昇腾" page, section "二、算力侧": experts with
 * similar token counts grouped into buckets, each with one batch shape), read
 * for this engine as an expert order: bucket class 0 for an empty expert, else
 * 1 + floor(log2(ceil(count / 128))); experts by class, largest first,
 * ascending id within a class, empty experts last (expert_order[E]); and
 * tile_sched_ordered[E+1], the exclusive scan of ceil(count / 128) in that
 * order. One CTA on the device from moe_permute's counts; E <= 1024. */
int moe_expert_buckets(const int32_t* counts, int E, int32_t* expert_order,
                       int32_t* tile_sched_ordered, void* stream);

/* moe_grouped_swiglu walking the experts in a given order (tile_sched_ordered
 * and expert_order from moe_expert_buckets): the persistent tiles then run
 * the big experts first. Results are identical to moe_grouped_swiglu. */
int moe_grouped_swiglu_ordered(const uint16_t* z_perm, const uint16_t* W13, const uint16_t* W2,
                               const int32_t* offsets, const int32_t* tile_sched_ordered,
                               const int32_t* expert_order, const float* row_w, int E, int R,
                               int l, int f, uint16_t* gu_save, uint16_t* h, uint16_t* y_perm,
                               void* stream);

/* moe_grouped_swiglu with the permute fused into GEMM1's operand load: the
 * permuted rows are never written. z is the unpermuted latent [T][l] and
 * permuted row r is z[token_of[r]] (token_of from moe_permute, which can then
 * be called with z = NULL); warps of the GEMM kernel copy the rows (16-byte
 * cp.async, z kept in L2) straight into the swizzled shared-memory tile. Results
 * are identical to moe_permute + moe_grouped_swiglu. This is the "less data
 * movement during token reordering" direction of [OPS]. */
int moe_grouped_swiglu_gather(const uint16_t* z, const int32_t* token_of, int T,
                              const uint16_t* W13, const uint16_t* W2, const int32_t* offsets,
                              const int32_t* tile_sched, const float* row_w, int E, int R, int l,
                              int f, uint16_t* gu_save, uint16_t* h, uint16_t* y_perm,
                              void* stream);

/* Shared experts of [MODEL] on all T latent rows, weight 1:
 *   [g_s|u_s] = z @ W13_sh[s];  h[:, s*f:(s+1)*f] = silu(g_s) * u_s   (h: bf16 [T][S*f])
 *   y_sh = sum_s h_s @ W2_sh[s]  (bf16 [T][l]);  gu_save: bf16 [T][S*2f], block s
 *   at columns s*2f.. (nullable). */
int moe_shared_swiglu(const uint16_t* z, const uint16_t* W13_sh, const uint16_t* W2_sh, int T,
                      int l, int f, int S, uint16_t* gu_save, uint16_t* h, uint16_t* y_sh,
                      void* stream);

/* ---------------------------------------------------------------- combine */

/* Unpermute + weighted combine of [OPS]: for every token t,
 *   y_lat[t] = sum_{j=0..k-1} y_perm[slot_of[t][j]] (+ y_shared[t])
 * summed in fp32 in that order, stored as bf16 [T][l]. y_shared nullable;
 * slot_of entries < 0 are skipped. With k = 1 this is the return of permuted
 * rows to arrival order. */
int moe_unpermute_combine(const uint16_t* y_perm, const int32_t* slot_of,
                          const uint16_t* y_shared, int T, int k, int l, uint16_t* y_lat,
                          void* stream);

/* Backward of the combine: dy_perm[r] = dy_lat[token_of[r]] for r < T*k
 * (zeros where token_of[r] < 0). bf16. */
int moe_unpermute_combine_bwd(const uint16_t* dy_lat, const int32_t* token_of, int T, int k, int l,
                              uint16_t* dy_perm, void* stream);

/* ---------------------------------------------------------------- backward */

/* Backward of moe_grouped_swiglu for dy_perm = d loss / d y_perm, routing fixed:
 *   dh_u[r]   = dy_perm[r] @ W2[e]^T;  d_row_w[r] = <dh_u[r], h[r]>  (fp32 [R])
 *   dh[r]     = row_w[r] * dh_u[r]
 *   dg = dh * u * s(g) * (1 + g (1 - s(g))),  du = dh * silu(g)   (s = sigmoid)
 *   dz_perm[r]= [dg|du][r] @ W13[e]^T                               (bf16 [R][l])
 *   dW2[e]    = sum_r (row_w[r] h[r])^T dy_perm[r]                  ([E][f][l])
 *   dW13[e]   = sum_r z_perm[r]^T [dg|du][r]                         ([E][l][2f])
 * dW13/dW2 are fp32 or bf16 per wgrad_dtype; an expert with no rows gets exact
 * zeros. The weight gradients of expert e read no more than a few of the rows
 * that follow its segment, multiplied by zero: they are exact as long as every
 * row of dy_perm / [dg|du] is finite (a non-finite row of expert e+1 may also
 * turn dW of expert e into NaN). gu_save and h from the forward are required. Workspace:
 * moe_workspace_size(MOE_OP_GROUPED_SWIGLU_BWD, 0, 0, l, E, 0, f, 0) with T*k = R
 * passed as T (k = 1). */
int moe_grouped_swiglu_bwd(const uint16_t* dy_perm, const uint16_t* z_perm, const uint16_t* W13,
                           const uint16_t* W2, const uint16_t* gu_save, const uint16_t* h,
                           const float* row_w, const int32_t* offsets, const int32_t* tile_sched,
                           int E, int R, int l, int f, uint16_t* dz_perm, float* d_row_w,
                           void* dW13, void* dW2, int wgrad_dtype, void* ws, size_t ws_bytes,
                           void* stream);

/* moe_grouped_swiglu_bwd reading g and u from the FP8 cache of
 * moe_grouped_swiglu_fp8cache (gu8 * scale of its block) in the SwiGLU
 * derivative (dg, du); h, and with it dW2 and d_row_w, is the bf16 forward's
 * as in moe_grouped_swiglu_bwd. Same workspace. */
int moe_grouped_swiglu_bwd_fp8cache(const uint16_t* dy_perm, const uint16_t* z_perm,
                                    const uint16_t* W13, const uint16_t* W2, const uint8_t* gu8,
                                    const float* gu_scale, const uint16_t* h, const float* row_w,
                                    const int32_t* offsets, const int32_t* tile_sched, int E,
                                    int R, int l, int f, uint16_t* dz_perm, float* d_row_w,
                                    void* dW13, void* dW2, int wgrad_dtype, void* ws,
                                    size_t ws_bytes, void* stream);

/* moe_grouped_swiglu_bwd with both permutes fused into the operand loads:
 * dy_perm[r] = dy_lat[token_of[r]] and z_perm[r] = z[token_of[r]] are gathered
 * inside the dgrad and wgrad GEMMs (dy_lat, z: [T][l]), so neither the
 * combine backward gather nor the permuted activations are materialised.
 * Results are identical to moe_grouped_swiglu_bwd on the permuted tensors. */
int moe_grouped_swiglu_bwd_gather(const uint16_t* dy_lat, const uint16_t* z,
                                  const int32_t* token_of, int T, const uint16_t* W13,
                                  const uint16_t* W2, const uint16_t* gu_save, const uint16_t* h,
                                  const float* row_w, const int32_t* offsets,
                                  const int32_t* tile_sched, int E, int R, int l, int f,
                                  uint16_t* dz_perm, float* d_row_w, void* dW13, void* dW2,
                                  int wgrad_dtype, void* ws, size_t ws_bytes, void* stream);

/* Backward of moe_shared_swiglu for dy = d loss / d y_sh ([T][l]):
 *   dz_sh = sum_s [dg_s|du_s] @ W13_sh[s]^T (bf16 [T][l]); dW13_sh [S][l][2f];
 *   dW2_sh [S][f][l] (fp32 or bf16). gu_save from the forward is required; `h`
 *   (the forward's [T][S*f] SwiGLU output) is the A operand of the dW2_sh product.
 * Workspace: moe_workspace_size(MOE_OP_SHARED_SWIGLU_BWD, T, 0, l, 0, 0, f, S) (the gate/up
 * gradients plus, at large T, fp32 partials of the K-split weight gradients). */
int moe_shared_swiglu_bwd(const uint16_t* dy, const uint16_t* z, const uint16_t* W13_sh,
                          const uint16_t* W2_sh, const uint16_t* gu_save, const uint16_t* h,
                          int T, int l, int f, int S, uint16_t* dz_sh, void* dW13_sh,
                          void* dW2_sh, int wgrad_dtype, void* ws, size_t ws_bytes,
                          void* stream);

/* Backward of the permute: dz[t] = sum_j dz_perm[slot_of[t][j]] (+ dz_shared[t]),
 * fp32 sum in j order, bf16 [T][l]. dz_shared nullable. */
int moe_permute_bwd(const uint16_t* dz_perm, const int32_t* slot_of, const uint16_t* dz_shared,
                    int T, int k, int l, uint16_t* dz, void* stream);

/* Backward of the router for d_row_w (from moe_grouped_swiglu_bwd):
 *   d_topk_w[t][j] = d_row_w[slot_of[t][j]]                         (fp32, nullable out)
 *   ds_j = (d_topk_w_j - sum_i w_i d_topk_w_i) / sum_i s_i;  dL[t][idx_j] = ds_j s_j (1 - s_j),
 *   zero for unselected experts (the selection is piecewise constant; the bias
 *   is a constant and gets no gradient)
 *   with aux_logits != NULL, dL also gets the gradient of aux_scale * the
 *   auxiliary balance loss (moe_router_aux_loss on aux_logits + aux_bias, whose
 *   p_mean is aux_p_mean): dense over all E experts,
 *   dL[t][e] += aux_scale s(1-s) / (T S_t) (ln p_mean[e] - sum_e' P(e'|t) ln p_mean[e'])
 *   dx_accum[T][d] += dL @ Wr^T  (bf16, read-modify-write), or, when dz is given,
 *   dx_accum = dz @ W_dn^T + dL @ Wr^T (overwrite; one GEMM over K = l + E that
 *   fuses the down-projection's input gradient: dz [T][l], W_dn [d][l])
 *   dWr[d][E] = x^T @ dL         (fp32 or bf16)
 * E must be a multiple of 64. Workspace (dL in bf16):
 * moe_workspace_size(MOE_OP_ROUTE_TOPK_BWD, T, 0, 0, E, 0, 0, 0). */
int moe_route_topk_bwd(const float* d_row_w, const int32_t* slot_of, const int32_t* topk_idx,
                       const float* topk_w, const float* topk_s, const uint16_t* x,
                       const uint16_t* Wr, int T, int d, int E, int k, float* d_topk_w,
                       uint16_t* dx_accum, void* dWr, int wgrad_dtype, const float* aux_logits,
                       const float* aux_bias, const float* aux_p_mean, float aux_scale,
                       const uint16_t* dz, const uint16_t* W_dn, int l, void* ws,
                       size_t ws_bytes, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------- diagnostics */

/* Per-kernel timing. While enabled, every kernel launch of the library is
 * bracketed by two CUDA events recorded on the launch's own stream (event
 * objects are created on first use and reused). moe_timing_report, called
 * after the caller synchronised those streams, writes one line per kernel
 * label, "label launches total_ms", into buf (NUL-terminated, truncated to
 * len), forgets the recorded pairs and returns the length of the full text.
 * With buf == NULL it only returns that length and keeps the pairs. */
int moe_timing_enable(int on);
int moe_timing_report(char* buf, size_t len);

/* Check of the bounded waits. Every wait of a library kernel on an mbarrier
 * (a copy landing, an accumulator filling or draining) gives up after a time
 * limit, ORs MOE_FLAG_TIMEOUT into the caller's error word and lets the kernel
 * return, so a wait that can never end does not hang the GPU. This call runs
 * that same wait, with the limit `limit_ns` (1e3 .. 1e9 ns), in one thread of
 * a one-warp kernel, on an mbarrier that nothing arrives at: it always times
 * out, sets MOE_FLAG_TIMEOUT in *err_flag (device int32) and writes the
 * nanoseconds it waited to *waited_ns (device int64). It uses no TMA copy, no
 * tensor map and no tensor memory. The pages describe nothing like it. */
int moe_diag_wait_timeout(long long limit_ns, int32_t* err_flag, long long* waited_ns,
                          void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
