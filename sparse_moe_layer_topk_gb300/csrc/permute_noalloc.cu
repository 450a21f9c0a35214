// moe_permute_noalloc: the token permute for callers that cannot allocate
// device memory.
//
// moe_permute needs a small scratch buffer (one int per 256-token chunk and
// expert) that the caller allocates and passes as `ws`. Some callers have no
// way to do that: code embedded in a host framework that hands it only its
// input and output buffers, or a caller on a fixed device-memory budget that
// must not call cudaMalloc / cudaFree (which can also synchronise the whole
// device and stall other streams). For them this entry point keeps the
// scratch in a fixed array in the library's own device memory instead.
//
// The array below lives in every GPU that loads the library, for as long as
// the library stays loaded. Its device address is looked up on the first call
// made on a device (and again if that device's current context has changed
// since, e.g. after a cudaDeviceReset); make that first call before any stream
// capture. All calls share the one array: calls that overlap on the GPU (on
// different streams, or from several threads) race on it and must be
// serialised by the caller. No entry of it has to start at zero: every entry a
// call reads was written earlier in the same call.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"

namespace moe {
namespace {

// 1 MiB: enough for T <= 256 * (262144 / E) tokens (74,752 tokens at E = 896).
constexpr long long kNoAllocScratchInts = 262144;

static __device__ __align__(256) int g_permute_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
  CUcontext ctx;  // the context the address was looked up in
  int* addr;
};
Cached g_cache[kMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_ctx_once;

// The CUDA driver API's current context (nullptr when it cannot be queried).
CUcontext current_context() {
  std::call_once(g_ctx_once, []() {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  });
  CUcontext c = nullptr;
  if (g_ctx_current == nullptr || g_ctx_current(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of g_permute_scratch in the current device's context, or
// nullptr with the cause recorded for moe_last_cuda_error().
int* scratch_address() {
  int dev = 0;
  const cudaError_t ed = cudaGetDevice(&dev);
  if (ed != cudaSuccess) {
    record_cuda_error(ed);
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    record_cuda_error(cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  // (cudaGetSymbolAddress makes the runtime's context current first: look the
  // context up after it, so that the pair cached belongs together)
  const CUcontext before = current_context();
  Cached& c = g_cache[dev];
  if (c.addr == nullptr || before == nullptr || c.ctx != before) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      c.addr = nullptr;
      return nullptr;
    }
    c.addr = static_cast<int*>(p);
    c.ctx = current_context();
  }
  return c.addr;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_permute_noalloc(const uint16_t* z, const int32_t* topk_idx,
                                   const float* topk_w, int T, int l, int E, int k,
                                   uint16_t* z_perm, int32_t* counts, int32_t* offsets,
                                   int32_t* slot_of, int32_t* token_of, int32_t* tile_sched,
                                   float* row_w, int32_t* err_flag, void* stream) {
  if (!(topk_idx && counts && offsets && slot_of && token_of && tile_sched)) return MOE_ERR_ARG;
  if (!(T >= 0 && E > 0 && E <= 1024 && k >= 1 && k <= 32 && k <= E)) return MOE_ERR_ARG;
  if (static_cast<long long>(T) * k >= (1ll << 31)) return MOE_ERR_ARG;
  if (z) {
    if (z_perm == nullptr || l <= 0) return MOE_ERR_ARG;
    if (l % 64 != 0 || (reinterpret_cast<uintptr_t>(z) & 15u) ||
        (reinterpret_cast<uintptr_t>(z_perm) & 15u))
      return MOE_ERR_ALIGN;
  }
  // The fixed scratch holds one int per (256-token chunk, expert).
  if (static_cast<long long>(permute_chunks(T)) * E > kNoAllocScratchInts) return MOE_ERR_WORKSPACE;
  int* scratch = scratch_address();
  if (scratch == nullptr) return MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const float* tw = (topk_w && row_w) ? topk_w : nullptr;
  cudaError_t e = launch_permute_maps(topk_idx, tw, T, E, k, scratch, counts, offsets, slot_of,
                                      token_of, tile_sched, tw ? row_w : nullptr, err_flag, st);
  if (e == cudaSuccess && z)
    e = launch_gather_rows("permute_gather", z, token_of, static_cast<long long>(T) * k, l, z_perm,
                           st);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
