// Routing, permute bookkeeping and row-movement kernels of libmoe (sm_103a).
//
//   topk_sigmoid_kernel   warp per token: top-k of (logit + bias) among the
//                         values that reach the k-th largest lane maximum, by
//                         warp redux over 64-bit (value, ~id) keys, then
//                         sigmoid and renormalisation.
//   chunk_hist_kernel     per 256-token chunk (four threads per token): one bit
//                         per (expert, token) in shared memory -> per-chunk
//                         expert histogram.
//   scan_kernel           one CTA: per-expert prefix over chunks, exclusive
//                         scan over experts (offsets), 128-row tile schedule.
//   maps_kernel           slot = expert offset + chunk prefix + popcount of the
//                         expert's token bits below this token: stable,
//                         atomics-free ranks.
//   gather_rows_kernel    dst[r] = src[index[r]] with 16-byte vectors (permute,
//                         combine backward).
//   gather_sum_kernel     out[t] = sum_j src[slot[t][j]] (+ add[t]) in fp32
//                         (combine, permute backward).
//   router_bwd_kernel     routing-weight gradient -> dense bf16 dL row.
//
// Sources: token Permute / Unpermute of the "昇腾实现Kimi K3.1 Pro模型LoRA训练适配"
// page, section "MoE(Mixture of Experts):算子融合与通信协同"; the per-expert load
// count of the "TorchTitan Ascend开源" page, section "在线负载规划"; top-16 of 896
// routed experts from section "Kimi K3.1 Pro 模型结构" of the same page.
#include "common.cuh"
#include "kernels.h"
#include "timing.h"

namespace moe {

namespace {

constexpr int kChunk = 256;  // tokens per chunk of the histogram / maps kernels
constexpr int kChunkThreads = 1024;  // 4 threads per token, each taking every 4th slot j


__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Selection keys: (order-preserving bits of the value) << 32 | ~id, so a larger
// key is a larger value or, for equal values, a lower expert id; 0 = no entry.
__device__ __forceinline__ unsigned long long sel_key(uint32_t value_key, int e) {
  return (static_cast<unsigned long long>(value_key) << 32) |
         static_cast<unsigned long long>(~static_cast<uint32_t>(e));
}

// Order-preserving bits of a float, in two integer operations: negative values
// have all bits flipped, non-negative ones the sign bit set. -0 and +0 are one
// value (they compare equal, so a tie between them goes to the lower expert id
// like any other): -0 is first made +0 by an IEEE add of +0, on the
// floating-point pipe.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

// Warp-wide maximum of 64-bit keys, as two 32-bit reductions: the high words,
// then the low words of the lanes holding the maximal high word.
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long x) {
  const uint32_t mh = __reduce_max_sync(0xFFFFFFFFu, static_cast<uint32_t>(x >> 32));
  const uint32_t ml = __reduce_max_sync(
      0xFFFFFFFFu, static_cast<uint32_t>(x >> 32) == mh ? static_cast<uint32_t>(x) : 0u);
  return (static_cast<unsigned long long>(mh) << 32) | ml;
}

// NPL keys per lane. VEC (E a multiple of 128): lane holds experts
// 128 i + 4 lane + j, read as float4; otherwise experts lane + 32 i. FULL:
// E = 32 NPL, every lane holds NPL experts.
//
// Fast path: every one of the k largest values is at least tau, the k-th
// largest of the 32 lanes' maxima (those k maxima are k values >= tau). The
// values >= tau (typically about twenty of 896) are compacted into shared
// memory; up to 32 of them are put in order by one bitonic sort across the
// warp (lane j then holds the j-th largest), up to 64 by k rounds of a
// warp-wide maximum. When more than 64 values reach tau (many equal values, or
// k close to 32), the selection falls back to k rounds over all of the lanes'
// keys, each lane tracking its largest and second largest key.
template <int NPL, bool VEC, bool FULL>
__global__ void __launch_bounds__(256, 4) topk_sigmoid_kernel(const float* __restrict__ L,
                                                              const float* __restrict__ bias,
                                                              int T, int E, int k,
                                                              int* __restrict__ idx,
                                                              float* __restrict__ w_out,
                                                              float* __restrict__ s_out,
                                                              int* err_flag) {
  __shared__ unsigned long long cand_s[8][64];  // 256 threads: 8 warps, one token each
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  if (t >= T) return;
  const float* row = L + static_cast<size_t>(t) * E;
  auto expert_of = [&](int i) { return VEC ? 128 * (i >> 2) + 4 * lane + (i & 3) : lane + 32 * i; };
  auto valid_at = [&](int i) { return VEC ? 128 * (i >> 2) < E : lane + 32 * i < E; };
  uint32_t kv[NPL];  // order keys of logit + bias; 0 where this lane holds no expert
  bool bad = false;
  if (VEC) {
    float4 lv[NPL / 4 > 0 ? NPL / 4 : 1];
#pragma unroll
    for (int i = 0; i < NPL / 4; ++i)
      lv[i] = (128 * i < E) ? __ldg(reinterpret_cast<const float4*>(row + 128 * i) + lane)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < NPL / 4; ++i) {
      const float vv[4] = {lv[i].x, lv[i].y, lv[i].z, lv[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = 128 * i + 4 * lane + j;
        if (128 * i < E) {
          const float v = vv[j] + (bias ? __ldg(bias + e) : 0.0f);
          if (!FULL) bad |= !isfinite(v);
          kv[4 * i + j] = order_key(v);
        } else {
          kv[4 * i + j] = 0u;
        }
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        const float v = __ldg(row + e) + (bias ? __ldg(bias + e) : 0.0f);
        if (!FULL) bad |= !isfinite(v);
        kv[i] = order_key(v);
      } else {
        kv[i] = 0u;
      }
    }
  }
  // tau: the k-th largest lane maximum (bitonic sort of the 32 maxima, descending)
  uint32_t mx = 0u;
#pragma unroll
  for (int i = 0; i < NPL; ++i) mx = max(mx, kv[i]);
  if (FULL) {
    // The order keys of the finite values lie strictly between those of -inf
    // (0x007FFFFF) and +inf (0xFF800000); NaNs fall outside them too.
    uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < NPL; ++i) mn = min(mn, kv[i]);
    bad = mx >= 0xFF800000u || mn <= 0x007FFFFFu;
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) set_flag(err_flag, MOE_FLAG_NONFINITE);
  uint32_t srt = mx;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xFFFFFFFFu, srt, stride);
      const bool take_max = ((lane & size) == 0) == ((lane & stride) == 0);
      srt = take_max ? max(srt, o) : min(srt, o);
    }
  }
  const uint32_t tau = __shfl_sync(0xFFFFFFFFu, srt, k - 1);
  uint32_t cmask = 0u;  // bit i: kv[i] reaches tau
#pragma unroll
  for (int i = 0; i < NPL; ++i) cmask |= ((FULL || valid_at(i)) && kv[i] >= tau) ? (1u << i) : 0u;
  const int cnt = __popc(cmask);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  unsigned long long mine = 0ull;  // the j-th selection, kept by lane j
  if (total <= 64) {
    unsigned long long* cs = cand_s[wib];
    int pos = incl - cnt;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (cmask & (1u << i)) cs[pos++] = sel_key(kv[i], expert_of(i));
    __syncwarp();
  }
  if (total <= 32) {
    // one candidate per lane (0 past them), sorted descending across the warp
    unsigned long long c = lane < total ? cand_s[wib][lane] : 0ull;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, c, stride);
        const bool take_max = ((lane & size) == 0) == ((lane & stride) == 0);
        c = take_max ? (o > c ? o : c) : (o < c ? o : c);
      }
    }
    mine = c;
  } else if (total <= 64) {
    unsigned long long* cs = cand_s[wib];
    for (int q = total + lane; q < 64; q += 32) cs[q] = 0ull;
    __syncwarp();
    unsigned long long c0 = cs[lane], c1 = cs[lane + 32];
    if (c1 > c0) { const unsigned long long x = c0; c0 = c1; c1 = x; }
    for (int j = 0; j < k; ++j) {
      // the value maximum first; the id reduction only when values tie exactly
      const uint32_t hi = static_cast<uint32_t>(c0 >> 32);
      const uint32_t mh = __reduce_max_sync(0xFFFFFFFFu, hi);
      const unsigned tied = __ballot_sync(0xFFFFFFFFu, hi == mh);
      unsigned long long m;
      if (__popc(tied) == 1) {
        m = __shfl_sync(0xFFFFFFFFu, c0, __ffs(tied) - 1);
      } else {
        const uint32_t ml =
            __reduce_max_sync(0xFFFFFFFFu, hi == mh ? static_cast<uint32_t>(c0) : 0u);
        m = (static_cast<unsigned long long>(mh) << 32) | ml;
      }
      if (lane == j) mine = m;
      if (c0 == m) { c0 = c1; c1 = 0ull; }
    }
  } else {
    unsigned long long key[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      key[i] = valid_at(i) ? sel_key(kv[i], expert_of(i)) : 0ull;
    // this lane's largest and second largest key
    unsigned long long b1 = 0ull, b2 = 0ull;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      if (key[i] > b1) { b2 = b1; b1 = key[i]; } else if (key[i] > b2) { b2 = key[i]; }
    }
    bool has2 = true;
    for (int j = 0; j < k; ++j) {
      const unsigned long long m = warp_max_key(b1);
      if (lane == j) mine = m;
      if (b1 == m) {
        // The winner's keys at or above m are all taken (a lane always gives up its
        // largest remaining key), so its next key is its second largest, or the
        // largest key below m once the second has been used as well.
        if (has2) {
          b1 = b2;
          has2 = false;
        } else {
          b1 = 0ull;
#pragma unroll
          for (int i = 0; i < NPL; ++i)
            if (key[i] < m && key[i] > b1) b1 = key[i];
        }
      }
    }
  }
  const float my_v = key_value(static_cast<uint32_t>(mine >> 32));
  const int my_e = static_cast<int>(~static_cast<uint32_t>(mine));
  const float s = (lane < k) ? 1.0f / (1.0f + expf(-my_v)) : 0.0f;
  float sum = s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  if (lane < k) {
    const size_t o = static_cast<size_t>(t) * k + lane;
    idx[o] = my_e;
    s_out[o] = s;
    w_out[o] = s / sum;
  }
}

__device__ __forceinline__ void build_bits(uint32_t* bits, const int* __restrict__ idx, int T,
                                           int E, int k, int* err_flag, bool check) {
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) bits[i] = 0u;
  __syncthreads();
  const int tk = threadIdx.x % kChunk;  // token within the chunk
  const int t = blockIdx.x * kChunk + tk;
  if (t < T) {
    const uint32_t bit = 1u << (tk & 31);
    const int word = tk >> 5;
    for (int j = threadIdx.x / kChunk; j < k; j += kChunkThreads / kChunk) {
      const int e = __ldg(idx + static_cast<size_t>(t) * k + j);
      if (e < 0 || e >= E) {
        if (check) set_flag(err_flag, MOE_FLAG_BAD_EXPERT);
        continue;
      }
      const uint32_t old = atomicOr(&bits[e * 8 + word], bit);
      if (check && (old & bit)) set_flag(err_flag, MOE_FLAG_BAD_EXPERT);  // repeated id
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kChunkThreads)
    chunk_hist_kernel(const int* __restrict__ idx, int T, int E, int k, int* __restrict__ hist,
                      int* err_flag) {
  extern __shared__ uint32_t bits[];
  build_bits(bits, idx, T, E, k, err_flag, true);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int wd = 0; wd < 8; ++wd) c += __popc(bits[e * 8 + wd]);
    hist[static_cast<size_t>(blockIdx.x) * E + e] = c;
  }
}

// Inclusive block scan of one int per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_inclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += n;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int r = v + (wid > 0 ? warp_sums[wid - 1] : 0);
  if (total) *total = warp_sums[31];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024) scan_kernel(int* __restrict__ hist, int nchunks, int E,
                                                    long long rows_cap, int* __restrict__ counts,
                                                    int* __restrict__ offsets,
                                                    int* __restrict__ tile_sched,
                                                    int* __restrict__ token_of) {
  __shared__ int warp_sums[32];
  const int e = threadIdx.x;
  int cnt = 0;
  if (e < E) {
    // sixteen chunks' counts loaded together, then the running prefix stored
    for (int c0 = 0; c0 < nchunks; c0 += 16) {
      int v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        v[i] = (c0 + i < nchunks) ? hist[static_cast<size_t>(c0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (c0 + i < nchunks) hist[static_cast<size_t>(c0 + i) * E + e] = cnt;
        cnt += v[i];
      }
    }
    counts[e] = cnt;
  }
  const int tiles = (cnt + 127) >> 7;
  int rows_total = 0, tiles_total = 0;
  const int off = block_inclusive_scan(cnt, warp_sums, &rows_total) - cnt;
  const int ts = block_inclusive_scan(tiles, warp_sums, &tiles_total) - tiles;
  if (e < E) {  // (the maps kernel adds offsets[e] to the per-chunk prefixes)
    offsets[e] = off;
    tile_sched[e] = ts;
  }
  if (e == 0) {
    offsets[E] = rows_total;
    tile_sched[E] = tiles_total;
  }
  // rows never filled (only when bad ids were dropped) point at no token
  for (long long r = rows_total + e; r < rows_cap; r += blockDim.x) token_of[r] = -1;
}

__global__ void __launch_bounds__(kChunkThreads)
    maps_kernel(const int* __restrict__ idx, int T, int E, int k, const int* __restrict__ base,
                const int* __restrict__ offsets, const float* __restrict__ topk_w,
                int* __restrict__ slot_of, int* __restrict__ token_of, float* __restrict__ row_w) {
  extern __shared__ uint32_t bits[];
  build_bits(bits, idx, T, E, k, nullptr, false);
  const int tk = threadIdx.x % kChunk;
  const int t = blockIdx.x * kChunk + tk;
  if (t >= T) return;
  const int word = tk >> 5;
  const uint32_t below = (1u << (tk & 31)) - 1u;
  for (int j = threadIdx.x / kChunk; j < k; j += kChunkThreads / kChunk) {
    const size_t o = static_cast<size_t>(t) * k + j;
    const int e = __ldg(idx + o);
    if (e < 0 || e >= E) {
      slot_of[o] = -1;
      continue;
    }
    int rank = __popc(bits[e * 8 + word] & below);
    for (int wd = 0; wd < word; ++wd) rank += __popc(bits[e * 8 + wd]);
    const int slot = __ldg(base + static_cast<size_t>(blockIdx.x) * E + e) + __ldg(offsets + e) + rank;
    slot_of[o] = slot;
    token_of[slot] = t;
    if (row_w) row_w[slot] = __ldg(topk_w + o);
  }
}

// One warp per destination row; l/8 16-byte vectors per row. The rows are
// written with evict-first (streaming) stores: the permuted copy is several
// times larger than L2 and is next read by another kernel, so its lines should
// not displace the source, which every row is gathered from.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ src,
                                                          const int* __restrict__ index,
                                                          long long R, int nvec,
                                                          uint4* __restrict__ dst) {
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < R;
       r += nwarps) {
    const int t = __ldg(index + r);
    uint4* d = dst + r * nvec;
    if (t < 0) {
      for (int v = lane; v < nvec; v += 32) d[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* s = src + static_cast<long long>(t) * nvec;
#pragma unroll 4
    for (int v = lane; v < nvec; v += 32) __stcs(d + v, __ldg(s + v));
  }
}

// One warp per token: lane j reads slot j of the token once; the rows are
// summed four at a time (their loads issued together, the sums taken in slot
// order), each lane owning up to 4 16-byte column vectors per pass. The k rows
// are read once, with evict-first (streaming) loads, so that they do not push
// the small summed output, which the next GEMM reads, out of L2.
__global__ void __launch_bounds__(256, 2) gather_sum_kernel(const uint4* __restrict__ src,
                                                            const int* __restrict__ slot, int k,
                                                            const uint4* __restrict__ add, int T,
                                                            int nvec, uint4* __restrict__ out,
                                                            long long ld_out_vec) {
  constexpr int U = 4;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int my_slot = lane < k ? __ldg(slot + static_cast<size_t>(t) * k + lane) : -1;
  const uint4 z4 = make_uint4(0, 0, 0, 0);
  for (int v0 = 0; v0 < nvec; v0 += 128) {
    float acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[i][e] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += U) {
      int r[U];
#pragma unroll
      for (int u = 0; u < U; ++u) r[u] = __shfl_sync(0xFFFFFFFFu, my_slot, (j0 + u) & 31);
      uint4 x[U][4];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int v = v0 + lane + 32 * i;
          x[u][i] = (j0 + u < k && r[u] >= 0 && v < nvec)
                        ? __ldcs(src + static_cast<long long>(r[u]) * nvec + v)
                        : z4;
        }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (j0 + u >= k || r[u] < 0) continue;  // warp-uniform
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t wv[4] = {x[u][i].x, x[u][i].y, x[u][i].z, x[u][i].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[i][2 * e] += bf16_lo(wv[e]);
            acc[i][2 * e + 1] += bf16_hi(wv[e]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int v = v0 + lane + 32 * i;
      if (v >= nvec) continue;
      if (add) {
        const uint4 a = __ldg(add + static_cast<long long>(t) * nvec + v);
        const uint32_t wv[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[i][2 * e] += bf16_lo(wv[e]);
          acc[i][2 * e + 1] += bf16_hi(wv[e]);
        }
      }
      out[static_cast<long long>(t) * ld_out_vec + v] =
          make_uint4(pack_bf16(acc[i][0], acc[i][1]), pack_bf16(acc[i][2], acc[i][3]),
                     pack_bf16(acc[i][4], acc[i][5]), pack_bf16(acc[i][6], acc[i][7]));
    }
  }
}

__global__ void dw_reduce_kernel(const float* __restrict__ part, int nparts, long long R,
                                 float* __restrict__ out) {
  for (long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; r < R;
       r += static_cast<long long>(gridDim.x) * blockDim.x) {
    float s = 0.0f;
    for (int p = 0; p < nparts; ++p) s += part[r * nparts + p];
    out[r] = s;
  }
}

// One warp per token (k <= 32): dL[t][:] = 0 except dL[t][idx_j] = ds_j s_j (1 - s_j).
__global__ void __launch_bounds__(256) router_bwd_kernel(
    const float* __restrict__ d_row_w, const int* __restrict__ slot_of,
    const int* __restrict__ topk_idx, const float* __restrict__ topk_w,
    const float* __restrict__ topk_s, int T, int E, int k, float* __restrict__ d_topk_w,
    bf16* __restrict__ dL, int* err_flag) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const size_t o = static_cast<size_t>(t) * k + lane;
  float dw = 0.0f, w = 0.0f, s = 0.0f;
  int e = -1;
  if (lane < k) {
    const int slot = __ldg(slot_of + o);
    dw = slot >= 0 ? __ldg(d_row_w + slot) : 0.0f;
    w = __ldg(topk_w + o);
    s = __ldg(topk_s + o);
    e = __ldg(topk_idx + o);
    if (d_topk_w) d_topk_w[o] = dw;
  }
  float ssum = s, dS = w * dw;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, off);
    dS += __shfl_xor_sync(0xFFFFFFFFu, dS, off);
  }
  bf16* row = dL + static_cast<size_t>(t) * E;
  uint4* row4 = reinterpret_cast<uint4*>(row);
  for (int v = lane; v < E / 8; v += 32) row4[v] = make_uint4(0, 0, 0, 0);
  __syncwarp();
  if (lane < k) {
    if (e >= 0 && e < E) {
      const float ds = (dw - dS) / ssum;
      row[e] = __float2bfloat16_rn(ds * s * (1.0f - s));
    } else {
      set_flag(err_flag, MOE_FLAG_BAD_EXPERT);
    }
  }
}

// ---- auxiliary balance loss: -H(pbar), pbar_e = mean_t s_te / sum_e' s_te'

// Warp w sums P(e|t) over its token range [w*tpw, (w+1)*tpw) into part[w][e].
template <int NPL>
__global__ void __launch_bounds__(256) aux_partial_kernel(const float* __restrict__ L,
                                                          const float* __restrict__ bias, int T,
                                                          int E, int tpw, int nwarps,
                                                          float* __restrict__ part) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= nwarps) return;
  float acc[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) acc[i] = 0.0f;
  const int t1 = min(T, (w + 1) * tpw);
  for (int t = w * tpw; t < t1; ++t) {
    const float* row = L + static_cast<size_t>(t) * E;
    float sv[NPL];
    float ssum = 0.0f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      sv[i] = 0.0f;
      if (e < E) {
        const float v = __ldg(row + e) + (bias ? __ldg(bias + e) : 0.0f);
        sv[i] = 1.0f / (1.0f + expf(-v));
        ssum += sv[i];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, o);
    const float inv = 1.0f / ssum;
#pragma unroll
    for (int i = 0; i < NPL; ++i) acc[i] = fmaf(sv[i], inv, acc[i]);
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) part[static_cast<size_t>(w) * E + e] = acc[i];
  }
}

// One CTA of 1024 threads: pbar_e = sum_w part[w][e] / T (in w order), loss = sum pbar log pbar.
__global__ void __launch_bounds__(1024) aux_reduce_kernel(const float* __restrict__ part,
                                                          int nwarps, int E, int T,
                                                          float* __restrict__ p_mean,
                                                          float* __restrict__ loss) {
  __shared__ float red[32];
  const int e = threadIdx.x;
  float term = 0.0f;
  if (e < E) {
    float sum = 0.0f;
    for (int w = 0; w < nwarps; ++w) sum += part[static_cast<size_t>(w) * E + e];
    const float p = sum / static_cast<float>(T);
    p_mean[e] = p;
    term = p > 0.0f ? p * logf(p) : 0.0f;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xFFFFFFFFu, term, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = term;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = red[threadIdx.x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (threadIdx.x == 0) *loss = v;
  }
}

// One warp per token: dL[t][e] += scale * s(1-s)/(T S) * (log pbar_e - sum_e' P_e' log pbar_e').
template <int NPL>
__global__ void __launch_bounds__(256) aux_bwd_kernel(const float* __restrict__ L,
                                                      const float* __restrict__ bias,
                                                      const float* __restrict__ p_mean, int T,
                                                      int E, float scale, bf16* __restrict__ dL) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* row = L + static_cast<size_t>(t) * E;
  float sv[NPL], cv[NPL];
  float ssum = 0.0f, csum = 0.0f;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    sv[i] = 0.0f;
    cv[i] = 0.0f;
    if (e < E) {
      const float v = __ldg(row + e) + (bias ? __ldg(bias + e) : 0.0f);
      sv[i] = 1.0f / (1.0f + expf(-v));
      cv[i] = logf(__ldg(p_mean + e));
      ssum += sv[i];
      csum = fmaf(cv[i], sv[i], csum);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, o);
    csum += __shfl_xor_sync(0xFFFFFFFFu, csum, o);
  }
  const float inner = csum / ssum;  // sum_e P_e log pbar_e
  const float k0 = scale / (static_cast<float>(T) * ssum);
  bf16* drow = dL + static_cast<size_t>(t) * E;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float g = k0 * sv[i] * (1.0f - sv[i]) * (cv[i] - inner);
      drow[e] = __float2bfloat16_rn(__bfloat162float(drow[e]) + g);
    }
  }
}

}  // namespace

// ------------------------------------------------------------------ launchers

cudaError_t launch_topk(const float* L, const float* bias, int T, int E, int k, int* idx,
                        float* w, float* s, int* err_flag, cudaStream_t st) {
  const int grid = (T + 7) / 8;
  const int npl = (E + 31) / 32;
  LaunchTimer lt("topk_sigmoid", st);
  const bool vec = (E % 128) == 0 && (reinterpret_cast<uintptr_t>(L) & 15u) == 0;
#define MOE_TOPK(N, V) topk_sigmoid_kernel<N, V, false><<<grid, 256, 0, st>>>(L, bias, T, E, k, idx, w, s, err_flag)
  if (vec && E == 32 * 28) {
    topk_sigmoid_kernel<28, true, true><<<grid, 256, 0, st>>>(L, bias, T, E, k, idx, w, s,
                                                             err_flag);
  } else if (vec) {
    if (npl <= 4) MOE_TOPK(4, true);
    else if (npl <= 8) MOE_TOPK(8, true);
    else if (npl <= 16) MOE_TOPK(16, true);
    else if (npl <= 28) MOE_TOPK(28, true);
    else MOE_TOPK(32, true);
  } else {
    if (npl <= 2) MOE_TOPK(2, false);
    else if (npl <= 4) MOE_TOPK(4, false);
    else if (npl <= 8) MOE_TOPK(8, false);
    else if (npl <= 16) MOE_TOPK(16, false);
    else if (npl <= 28) MOE_TOPK(28, false);
    else MOE_TOPK(32, false);
  }
#undef MOE_TOPK
  return cudaGetLastError();
}

int permute_chunks(int T) { return (T + kChunk - 1) / kChunk; }

cudaError_t launch_permute_maps(const int* idx, const float* topk_w, int T, int E, int k,
                                int* hist_ws, int* counts, int* offsets, int* slot_of,
                                int* token_of, int* tile_sched, float* row_w, int* err_flag,
                                cudaStream_t st) {
  const int nch = permute_chunks(T);
  const size_t sm = static_cast<size_t>(E) * 8 * sizeof(uint32_t);
  if (nch > 0) {
    LaunchTimer lt("permute_hist", st);
    chunk_hist_kernel<<<nch, kChunkThreads, sm, st>>>(idx, T, E, k, hist_ws, err_flag);
  }
  {
    // with no tokens the scan alone writes the zero counts, offsets and schedule
    LaunchTimer lt("permute_scan", st);
    scan_kernel<<<1, 1024, 0, st>>>(hist_ws, nch, E, static_cast<long long>(T) * k, counts,
                                    offsets, tile_sched, token_of);
  }
  if (nch > 0) {
    LaunchTimer lt("permute_maps", st);
    maps_kernel<<<nch, kChunkThreads, sm, st>>>(idx, T, E, k, hist_ws, offsets, topk_w, slot_of,
                                                token_of, row_w);
  }
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const char* name, const void* src, const int* index, long long R,
                               int l, void* dst, cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  const long long warps = R;
  long long blocks = (warps + 7) / 8;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  LaunchTimer lt(name, st);
  gather_rows_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(
      reinterpret_cast<const uint4*>(src), index, R, l / 8, reinterpret_cast<uint4*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_gather_sum(const char* name, const void* src, const int* slot, int k,
                              const void* add, int T, int l, void* out, long long ld_out,
                              cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  LaunchTimer lt(name, st);
  gather_sum_kernel<<<(T + 7) / 8, 256, 0, st>>>(
      reinterpret_cast<const uint4*>(src), slot, k, reinterpret_cast<const uint4*>(add), T, l / 8,
      reinterpret_cast<uint4*>(out), ld_out / 8);
  return cudaGetLastError();
}

cudaError_t launch_dw_reduce(const float* part, int nparts, long long R, float* out,
                             cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  long long blocks = (R + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  LaunchTimer lt("routing_weight_grad_reduce", st);
  dw_reduce_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(part, nparts, R, out);
  return cudaGetLastError();
}

cudaError_t launch_router_bwd(const float* d_row_w, const int* slot_of, const int* topk_idx,
                              const float* topk_w, const float* topk_s, int T, int E, int k,
                              float* d_topk_w, void* dL, int* err_flag, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  LaunchTimer lt("router_bwd_dlogits", st);
  router_bwd_kernel<<<(T + 7) / 8, 256, 0, st>>>(d_row_w, slot_of, topk_idx, topk_w, topk_s, T, E,
                                                 k, d_topk_w, reinterpret_cast<bf16*>(dL),
                                                 err_flag);
  return cudaGetLastError();
}

}  // namespace moe

namespace moe {

int aux_partial_warps(int T) {
  const int w = (T + 15) / 16;
  return w < 1024 ? (w < 1 ? 1 : w) : 1024;
}

#define MOE_AUX_DISPATCH(KERNEL, GRID, ...)                                   \
  do {                                                                         \
    const int npl_ = (E + 31) / 32;                                            \
    if (npl_ <= 2) KERNEL<2><<<GRID, 256, 0, st>>>(__VA_ARGS__);               \
    else if (npl_ <= 4) KERNEL<4><<<GRID, 256, 0, st>>>(__VA_ARGS__);          \
    else if (npl_ <= 8) KERNEL<8><<<GRID, 256, 0, st>>>(__VA_ARGS__);          \
    else if (npl_ <= 16) KERNEL<16><<<GRID, 256, 0, st>>>(__VA_ARGS__);        \
    else if (npl_ <= 28) KERNEL<28><<<GRID, 256, 0, st>>>(__VA_ARGS__);        \
    else KERNEL<32><<<GRID, 256, 0, st>>>(__VA_ARGS__);                        \
  } while (0)

cudaError_t launch_aux_loss(const float* L, const float* bias, int T, int E, float* part,
                            float* p_mean, float* loss, cudaStream_t st) {
  const int nw = aux_partial_warps(T);
  const int tpw = (T + nw - 1) / nw;
  {
    LaunchTimer lt("router_aux_partial", st);
    MOE_AUX_DISPATCH(aux_partial_kernel, (nw + 7) / 8, L, bias, T, E, tpw, nw, part);
  }
  {
    LaunchTimer lt("router_aux_reduce", st);
    aux_reduce_kernel<<<1, 1024, 0, st>>>(part, nw, E, T, p_mean, loss);
  }
  return cudaGetLastError();
}

cudaError_t launch_aux_bwd(const float* L, const float* bias, const float* p_mean, int T, int E,
                           float scale, void* dL, cudaStream_t st) {
  LaunchTimer lt("router_aux_bwd", st);
  MOE_AUX_DISPATCH(aux_bwd_kernel, (T + 7) / 8, L, bias, p_mean, T, E, scale,
                   reinterpret_cast<bf16*>(dL));
  return cudaGetLastError();
}

}  // namespace moe

namespace moe {
namespace {

// Online replica plan (one thread; E + P <= 2048 steps): rank r owns experts
// [r*E/P, (r+1)*E/P) and may process C = ceil(rows / P) rows. Ranks first take
// their own experts' rows while they have room; the rest of each expert goes,
// in rank order, to ranks with spare capacity (replicas that keep the expert).
// pieces[i] = {expert, rank, first row within the expert's segment, rows}.
__global__ void replica_plan_kernel(const int* __restrict__ counts, int E, int P,
                                    int* __restrict__ pieces, int* __restrict__ n_pieces,
                                    int* __restrict__ load_out) {
  extern __shared__ int sm[];
  int* load = sm;       // [P]
  int* done = sm + P;   // [E]
  if (threadIdx.x != 0) return;
  const int per = E / P;
  long long R = 0;
  for (int e = 0; e < E; ++e) {
    if (counts[e] < 0) {  // not a count: no plan
      *n_pieces = -1;
      return;
    }
    R += counts[e];
  }
  if (R >= (1ll << 31)) {
    *n_pieces = -1;
    return;
  }
  const int C = static_cast<int>((R + P - 1) / P);
  int n = 0;
  for (int r = 0; r < P; ++r) {
    load[r] = 0;
    for (int e = r * per; e < (r + 1) * per; ++e) {
      const int take = min(counts[e], C - load[r]);
      done[e] = 0;
      if (take > 0) {
        pieces[4 * n] = e; pieces[4 * n + 1] = r; pieces[4 * n + 2] = 0; pieces[4 * n + 3] = take;
        ++n;
        load[r] += take;
        done[e] = take;
      }
    }
  }
  for (int e = 0; e < E; ++e) {
    int r = 0;
    while (done[e] < counts[e]) {
      // P * C >= R rows, so a rank with spare capacity remains while rows do
      while (r < P && load[r] >= C) ++r;
      if (r == P) {
        *n_pieces = -1;
        return;
      }
      const int take = min(counts[e] - done[e], C - load[r]);
      pieces[4 * n] = e; pieces[4 * n + 1] = r; pieces[4 * n + 2] = done[e]; pieces[4 * n + 3] = take;
      ++n;
      load[r] += take;
      done[e] += take;
    }
  }
  *n_pieces = n;
  for (int r = 0; r < P; ++r) load_out[r] = load[r];
}

}  // namespace

cudaError_t launch_replica_plan(const int* counts, int E, int P, int* pieces, int* n_pieces,
                                int* load, cudaStream_t st) {
  LaunchTimer lt("replica_plan", st);
  replica_plan_kernel<<<1, 32, static_cast<size_t>(E + P) * sizeof(int), st>>>(counts, E, P, pieces,
                                                                                n_pieces, load);
  return cudaGetLastError();
}

}  // namespace moe

namespace moe {
namespace {

// Expert order for bucketed batching (one CTA of 1024 threads, E <= 1024):
// class 0 = empty, else 1 + floor(log2(row tiles)); largest class first,
// ascending expert id within a class; then the exclusive scan of the row
// tiles in that order.
__global__ void __launch_bounds__(1024) bucket_order_kernel(const int* __restrict__ counts, int E,
                                                           int* __restrict__ order,
                                                           int* __restrict__ sched) {
  __shared__ int warp_sums[32];
  __shared__ int class_n[32];
  __shared__ int tiles_at[1024];
  const int e = threadIdx.x;
  const int nt = e < E ? (counts[e] + 127) >> 7 : 0;
  const int cls = e < E ? (nt == 0 ? 0 : 32 - __clz(nt)) : -1;  // 1 + floor(log2 nt)
  if (e < 32) class_n[e] = 0;
  __syncthreads();
  if (e < E) atomicAdd(&class_n[cls], 1);
  __syncthreads();
  int pos = -1;
  int base = 0;
  for (int c = 31; c >= 0; --c) {  // classes in descending order
    const int n = class_n[c];      // uniform across the block
    if (n == 0) continue;
    const int flag = (cls == c) ? 1 : 0;
    const int rank = block_inclusive_scan(flag, warp_sums, nullptr) - flag;
    if (flag) pos = base + rank;
    base += n;
  }
  if (e < E) {
    order[pos] = e;
    tiles_at[pos] = nt;
  }
  __syncthreads();
  const int v = e < E ? tiles_at[e] : 0;
  int total = 0;
  const int incl = block_inclusive_scan(v, warp_sums, &total);
  if (e < E) sched[e] = incl - v;
  if (e == 0) sched[E] = total;
}

}  // namespace

cudaError_t launch_bucket_order(const int* counts, int E, int* order, int* sched,
                                cudaStream_t st) {
  LaunchTimer lt("bucket_order", st);
  bucket_order_kernel<<<1, 1024, 0, st>>>(counts, E, order, sched);
  return cudaGetLastError();
}

}  // namespace moe
