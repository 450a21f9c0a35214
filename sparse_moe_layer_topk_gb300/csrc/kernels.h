// Launchers of the non-GEMM kernels of libmoe (route_permute.cu).
#pragma once

#include <cuda_runtime.h>

namespace moe {

int num_sms();

cudaError_t launch_topk(const float* L, const float* bias, int T, int E, int k, int* idx, float* w,
                        float* s, int* err_flag, cudaStream_t st);
int permute_chunks(int T);
cudaError_t launch_permute_maps(const int* idx, const float* topk_w, int T, int E, int k,
                                int* hist_ws, int* counts, int* offsets, int* slot_of,
                                int* token_of, int* tile_sched, float* row_w, int* err_flag,
                                cudaStream_t st);
cudaError_t launch_gather_rows(const char* name, const void* src, const int* index, long long R,
                               int l, void* dst, cudaStream_t st);
cudaError_t launch_gather_sum(const char* name, const void* src, const int* slot, int k,
                              const void* add, int T, int l, void* out, long long ld_out,
                              cudaStream_t st);
cudaError_t launch_dw_reduce(const float* part, int nparts, long long R, float* out,
                             cudaStream_t st);
cudaError_t launch_router_bwd(const float* d_row_w, const int* slot_of, const int* topk_idx,
                              const float* topk_w, const float* topk_s, int T, int E, int k,
                              float* d_topk_w, void* dL, int* err_flag, cudaStream_t st);

int aux_partial_warps(int T);
cudaError_t launch_aux_loss(const float* L, const float* bias, int T, int E, float* part,
                            float* p_mean, float* loss, cudaStream_t st);
cudaError_t launch_aux_bwd(const float* L, const float* bias, const float* p_mean, int T, int E,
                           float scale, void* dL, cudaStream_t st);

cudaError_t launch_replica_plan(const int* counts, int E, int P, int* pieces, int* n_pieces,
                                int* load, cudaStream_t st);

cudaError_t launch_bucket_order(const int* counts, int E, int* order, int* sched,
                                cudaStream_t st);

}  // namespace moe
