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

// The activation operand is kept in global memory as the very image of the
// tensor-core kernel's shared-memory stages, so that one bulk copy loads a
// stage (a 128-row tile of 64 k-columns is 16 KB: row R at byte 128 R, its
// 16-byte chunk j at chunk position j ^ (R % 8), the 128-byte swizzle the
// MMA descriptors read).  Stacked batches (B <= 64) hold hi parts in rows
// [0, 64) and lo parts in rows [64, 128) of one tile per k-block; larger
// batches hold, per m-block of 128 rows and k-block, a hi tile then a lo tile.
// k-columns past H read as zeros.
inline int tc_stacked(int B) { return B <= TC_STACK_MAX ? 1 : 0; }
inline int tc_mblocks(int B) { return tc_stacked(B) ? 1 : (B + TC_M - 1) / TC_M; }
inline int tc_kblocks(int H) { return (H + TC_KB - 1) / TC_KB; }
constexpr int TC_A_TILE_BYTES = TC_M * TC_KB * 2;  // one 128-row, 64-column bf16 tile
inline int64_t tc_act_image_bytes(int B, int H) {
  return static_cast<int64_t>(tc_mblocks(B)) * tc_kblocks(H) * TC_A_TILE_BYTES * (tc_stacked(B) ? 1 : 2);
}
// Byte offset in the image of batch row b's hi (lo = 0) or lo (lo = 1) part at k-column h.
__host__ __device__ inline int64_t tc_act_image_offset(int stacked, int kblocks, int b, int lo, int h) {
  int R;
  int64_t base;
  if (stacked) {
    R = lo ? 64 + b : b;
    base = static_cast<int64_t>(h >> 6) * TC_A_TILE_BYTES;
  } else {
    R = b & (TC_M - 1);
    base = ((static_cast<int64_t>(b / TC_M) * kblocks + (h >> 6)) * 2 + lo) * TC_A_TILE_BYTES;
  }
  const int c = h & 63;
  return base + R * 128 + ((((c >> 3) ^ R) & 7) << 4) + (c & 7) * 2;
}
inline int tc_tile_n(int B) { return tc_stacked(B) ? TC_N_STACKED : TC_N_SEPARATE; }
inline int tc_col_tiles(int V, int tile_n) { return (V + tile_n - 1) / tile_n; }

// The prepared weight (weight_pack.cu): 8 KB blocks of 64 k-rows x 64 columns
// in the shared-memory image of one weight box, k-block major.
constexpr int TC_W_BLOCK_BYTES = 64 * 64 * 2;
inline int tc_weight_groups(int V) { return (V + 63) / 64; }
int64_t tc_packed_weight_bytes(int H, int V);
// weight stages the tensor-core kernel keeps in flight from the prepared weight (its ring holds 6
// stages of 24 KB when hi and lo share a tile, 3 of 32 KB otherwise)
constexpr int TC_PACKED_AHEAD_STACKED = 5;
constexpr int TC_PACKED_AHEAD_SEPARATE = 3;
cudaError_t launch_weight_pack(const uint16_t* w, int H, int V, uint8_t* out, int num_sms, cudaStream_t stream);


struct SplitArgs {
  const void* hidden;
  int dtype;
  const float* gamma;
  int B, H, Hu;
  float eps;
  int zero_pad;
  int deferred;
  int stacked;
  uint8_t* act_img;  // the activation image (tc_act_image_bytes(B, H) bytes)
  float* row_scale;  // [B]: rstd (deferred) or 1
  int use_moe = 0;   // 1: the rows are formed by the producer step from `moe` (hidden is unused)
  MoeIn moe;
};
// widest hidden state the split kernel forms from the producer step itself (h row in shared memory)
constexpr int SPLIT_MOE_MAX_H = 24576;

struct TcArgs {
  const uint8_t* act_img;  // the activation image written by the split kernel
  const uint8_t* w_packed = nullptr;  // the prepared weight, or null: tensor-tile loads through mapW
  int w_groups = 0;                   // 64-column groups of the prepared weight
  int w_ahead = 0;                    // weight stages kept in flight (0: the whole ring)
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
// mapW: w_t [H][V] bf16, box 64 x 64, 128-byte swizzle;
// mapL: logits [B][V] fp32, box 32 x 32, 128-byte swizzle.
cudaError_t launch_tc(const TcArgs& a, const CUtensorMap& mapW, const CUtensorMap& mapL,
                      int stacked, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_merge(const MergeArgs& a, int grid, cudaStream_t stream, bool pdl);
cudaError_t prepare_tc_gemm(int max_smem_optin);
// per device: shared-memory opt-in of the tensor-core kernels; returns the
// merge kernel's dynamic shared-memory budget
cudaError_t prepare_tc(int max_smem_optin, int* merge_dyn_max);
// merge kernel plan for K candidates over ntn tiles within `dyn_max` bytes; false if it cannot fit
bool plan_merge(int K, int ntn, int dyn_max, int* capc, int* sortP, int* smem_bytes);

}  // namespace tail
