// Host-side declarations of the vocabulary-parallel merge.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tail {

constexpr int SHARD_MAX = 64;          // vocabulary shards one merge takes
constexpr int SHARD_CAND_MAX = 16384;  // shards x candidates per row held in shared memory

struct ShardMergeArgs {
  const float* vals;     // [nshard][B][k_in] each shard's top-k logits, descending
  const int32_t* idx;    // [nshard][B][k_in] their ids within the shard
  int32_t offsets[SHARD_MAX];  // first global vocabulary id of each shard
  int nshard, k_in, K, B;
  const float* params;   // [B][ncols] or null
  int ncols;
  int32_t* tokens;       // [B] or null
  float* topk_val;       // [B][K] or null
  int32_t* topk_idx;     // [B][K] or null
  int sortP, smem_bytes;
};

// dynamic shared memory of a merge over nshard x k_in candidates a row; sets *sortP
int shard_merge_smem(int nshard, int k_in, int K, int* sortP);
cudaError_t launch_shard_merge(const ShardMergeArgs& a, cudaStream_t stream);

}  // namespace tail
