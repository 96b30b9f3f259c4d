// Vocabulary-parallel merge: the global top-k and the sampler over the
// candidates of several vocabulary shards ("GPT-OSS Tail Chunked Megakernel
// Kernel API Reference", section "Background": each rank computes the top-k
// of its own vocabulary slice, and one top-k over the union is the global one;
// parameters `k` and `sampling_params`).
//
// Every shard's sorted top-k holds all of that shard's elements that can be in
// the global top-k, so the top K of the union, ordered by (value desc, global
// index asc), is the global top-K.  One CTA per row: the union's keys and
// global indices in shared memory, its exact top K, a rank sort, the top-k
// outputs and the draw.
#include <stdio.h>

#include <mutex>

#include "../../include/tail.h"
#include "abi_common.h"
#include "common.cuh"
#include "internal.h"
#include "sampler.cuh"
#include "select.cuh"
#include "shard_merge.h"

namespace tail {

namespace {

constexpr int SHARD_THREADS = 256;

__global__ void __launch_bounds__(SHARD_THREADS) shard_merge_kernel(const ShardMergeArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint32_t s_red[64];
  __shared__ uint32_t s_list[SEL_BLOCK_BUCKET_MAX];
  __shared__ uint32_t s_misc[4];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int n = a.nshard * a.k_in, K = a.K;
  const int n2 = (n + 1) & ~1;  // both arrays padded to an even length: comp starts 8-byte aligned
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  int32_t* ids = reinterpret_cast<int32_t*>(keys + n2);
  uint64_t* comp = reinterpret_cast<uint64_t*>(ids + n2);
  uint64_t* sorted = comp + a.sortP;
  float* ebuf = reinterpret_cast<float*>(sorted + K);
  for (int row = blockIdx.x; row < a.B; row += gridDim.x) {
    SampleParams prm = {};
    if (a.params != nullptr) prm = load_sample_params(a.params + static_cast<int64_t>(row) * a.ncols, a.ncols);
    for (int j = tid; j < n; j += nt) {
      const int s = j / a.k_in, i = j - s * a.k_in;
      const int64_t src = (static_cast<int64_t>(s) * a.B + row) * a.k_in + i;
      keys[j] = float_key(a.vals[src]);
      ids[j] = a.idx[src] + a.offsets[s];
    }
    __syncthreads();
    int nr = n;
    if (n <= RANK_SORT_MAX) {
      for (int j = tid; j < n; j += nt) comp[j] = composite(keys[j], ids[j]);
      __syncthreads();
    } else {
      for (int j = tid; j < a.sortP; j += nt) comp[j] = 0ull;
      __syncthreads();
      block_top_composites(keys, ids, n, K, comp, s_red, s_list, s_misc);
      nr = K;
    }
    sort_runs(comp, sorted, nr, K);
    if (a.topk_val != nullptr)
      for (int j = tid; j < K; j += nt) a.topk_val[static_cast<int64_t>(row) * K + j] = key_float(composite_key(sorted[j]));
    if (a.topk_idx != nullptr)
      for (int j = tid; j < K; j += nt) a.topk_idx[static_cast<int64_t>(row) * K + j] = composite_idx(sorted[j]);
    if (a.params != nullptr && a.tokens != nullptr && (tid >> 5) == 0) {  // the draw: warp 0
      const int32_t tok = sample_sorted_warp(prm, sorted, K, ebuf);
      if (tid == 0) a.tokens[row] = tok;
    }
    __syncthreads();
  }
}

int next_pow2_host(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

int shard_merge_smem(int nshard, int k_in, int K, int* sortP) {
  const int n2 = (nshard * k_in + 1) & ~1;
  *sortP = next_pow2_host(K) > RANK_SORT_MAX ? next_pow2_host(K) : RANK_SORT_MAX;
  return n2 * 8 + *sortP * 8 + K * 8 + K * 4;
}

cudaError_t launch_shard_merge(const ShardMergeArgs& a, cudaStream_t stream) {
  static_assert(SHARD_THREADS % 32 == 0, "whole warps");
  // the shared-memory opt-in only grows, per device (set once for the largest size asked so far)
  static std::mutex mu;
  static int opted[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (a.smem_bytes > opted[dev]) {
      e = cudaFuncSetAttribute(shard_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, a.smem_bytes);
      if (e != cudaSuccess) return e;
      opted[dev] = a.smem_bytes;
    }
  }
  shard_merge_kernel<<<a.B, SHARD_THREADS, a.smem_bytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace tail

using namespace tail;

extern "C" int tail_merge_shards(int32_t nshard, int32_t k_in, int32_t k, int32_t gbs, const float* cand_vals,
                                 const int32_t* cand_idx, const int32_t* shard_offsets, const float* params,
                                 int32_t n_param_cols, int32_t* out_tokens, float* out_topk_vals_opt,
                                 int32_t* out_topk_idx_opt, void* stream) {
  if (nshard < 1 || nshard > SHARD_MAX || k < 1 || k > MAX_K || k_in < 1 || gbs < 0) return TAIL_ERR_INVALID_ARG;
  if (k > static_cast<int64_t>(nshard) * k_in) return TAIL_ERR_INVALID_ARG;
  if (static_cast<int64_t>(nshard) * k_in > SHARD_CAND_MAX) {
    set_last_error("tail_merge_shards: more than 16384 candidates a row");
    return TAIL_ERR_UNSUPPORTED;
  }
  if (gbs == 0) return TAIL_OK;
  if (!cand_vals || !cand_idx || !shard_offsets) return TAIL_ERR_INVALID_ARG;
  if (!aligned(cand_vals, 4) || !aligned(cand_idx, 4)) return TAIL_ERR_INVALID_ARG;
  if (params) {
    if (n_param_cols != 3 && n_param_cols != 4) return TAIL_ERR_INVALID_ARG;
    if (!out_tokens || !aligned(params, 4) || !aligned(out_tokens, 4)) return TAIL_ERR_INVALID_ARG;
  }
  if ((out_topk_vals_opt && !aligned(out_topk_vals_opt, 4)) || (out_topk_idx_opt && !aligned(out_topk_idx_opt, 4)))
    return TAIL_ERR_INVALID_ARG;
  ShardMergeArgs a = {};
  a.vals = cand_vals;
  a.idx = cand_idx;
  for (int s = 0; s < nshard; ++s) {
    if (shard_offsets[s] < 0) return TAIL_ERR_INVALID_ARG;
    a.offsets[s] = shard_offsets[s];
  }
  a.nshard = nshard;
  a.k_in = k_in;
  a.K = k;
  a.B = gbs;
  a.params = params;
  a.ncols = n_param_cols;
  a.tokens = params ? out_tokens : nullptr;
  a.topk_val = out_topk_vals_opt;
  a.topk_idx = out_topk_idx_opt;
  a.smem_bytes = shard_merge_smem(nshard, k_in, k, &a.sortP);
  const cudaError_t e = launch_shard_merge(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "tail_merge_shards: kernel launch");
  return TAIL_OK;
}
