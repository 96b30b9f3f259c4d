// Host-side declarations of the tensor-core path (batches above 8 rows):
// activation split, tcgen05 lm_head with per-tile candidate lists, and the
// per-row merge + sampler.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_internal.h"

namespace tail {

constexpr int TC_M = 128;        // rows of one MMA tile (tensor-memory lanes)
// vocabulary columns of one tile: three 64-column TMA boxes while hi and lo
// share a tile (the weight-bound sizes, where a narrower stage leaves room for
// more of the weight in flight), four (the whole 256-column accumulator) when
// they have tiles of their own (fewer activation bytes per MMA flop, which
// matters once the tensor pipe is the limit)
constexpr int TC_N_STACKED = 192;
constexpr int TC_N_SEPARATE = 256;
constexpr int TC_KB = 64;        // k extent of one ring stage (one 128-byte swizzle row of bf16)
constexpr int TC_LIST = 8;       // candidates each (row, tile) keeps: its top 8 by (value desc, index asc)
constexpr int TC_STACK_MAX = 64; // up to this many rows, hi and lo parts share one 128-row tile
constexpr int MERGE_THREADS = 256;
constexpr int TC_MIN_ROWS = 9;   // batches of at least this many rows take the tensor-core path

// Rows of the activation buffer for a batch of B rows: stacked (B <= 64) puts
// hi parts in rows [0, 64) and lo parts in rows [64, 128); otherwise m-block mb
// (128 batch rows) owns rows [256 mb, 256 mb + 128) for hi and the next 128 for lo.
inline int tc_stacked(int B) { return B <= TC_STACK_MAX ? 1 : 0; }
inline int tc_mblocks(int B) { return tc_stacked(B) ? 1 : (B + TC_M - 1) / TC_M; }
inline int64_t tc_act_rows(int B) { return tc_stacked(B) ? TC_M : static_cast<int64_t>(tc_mblocks(B)) * 2 * TC_M; }
inline int tc_tile_n(int B) { return tc_stacked(B) ? TC_N_STACKED : TC_N_SEPARATE; }
inline int tc_col_tiles(int V, int tile_n) { return (V + tile_n - 1) / tile_n; }

struct SplitArgs {
  const void* hidden;
  int dtype;
  const float* gamma;
  int B, H, Hu;
  float eps;
  int zero_pad;
  int deferred;
  int stacked;
  uint16_t* act;     // [tc_act_rows(B)][H] bf16 bits
  float* row_scale;  // [B]: rstd (deferred) or 1
  int use_moe = 0;   // 1: the rows are formed by the producer step from `moe` (hidden is unused)
  MoeIn moe;
};
// widest hidden state the split kernel forms from the producer step itself (h row in shared memory)
constexpr int SPLIT_MOE_MAX_H = 24576;

struct TcArgs {
  const float* row_scale;  // [B]
  float* logits;           // [B][ld] fp32: the caller's logits or scratch (always written)
  int64_t ld;
  uint64_t* lists;         // [B][ntn][TC_LIST] composites, descending
  int* err;
  int B, V, ntn, n_mb, kblocks;
  uint64_t timeout_ns;
};

struct MergeArgs {
  const uint64_t* lists;   // [B][ntn][TC_LIST]
  const float* logits;     // [B][ld]
  int64_t ld;
  float* topk_val;         // [B][topk_ld]
  int32_t* topk_idx;
  int64_t topk_ld;
  const float* params;     // [B][ncols] or null
  int ncols;
  int32_t* tokens;         // [B] or null
  int B, V, K, ntn;
  int tile_n;              // vocabulary columns of one tile (tc_tile_n of the batch)
  int capc, sortP, smem_bytes;
  int* err;                // device error flag (a bounded wait ran out)
  uint64_t timeout_ns;
};

cudaError_t launch_split(const SplitArgs& a, cudaStream_t stream);
// mapA: activation buffer [rows][H] bf16, box 64 x 128, 128-byte swizzle;
// mapW: w_t [H][V] bf16, box 64 x 64, 128-byte swizzle;
// mapL: logits [B][V] fp32, box 32 x 32, 128-byte swizzle.
cudaError_t launch_tc(const TcArgs& a, const CUtensorMap& mapA, const CUtensorMap& mapW, const CUtensorMap& mapL,
                      int stacked, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_merge(const MergeArgs& a, int grid, cudaStream_t stream, bool pdl);
cudaError_t prepare_tc_gemm(int max_smem_optin);
// per device: shared-memory opt-in of the tensor-core kernels; returns the
// merge kernel's dynamic shared-memory budget
cudaError_t prepare_tc(int max_smem_optin, int* merge_dyn_max);
// merge kernel plan for K candidates over ntn tiles within `dyn_max` bytes; false if it cannot fit
bool plan_merge(int K, int ntn, int dyn_max, int* capc, int* sortP, int* smem_bytes);

}  // namespace tail
