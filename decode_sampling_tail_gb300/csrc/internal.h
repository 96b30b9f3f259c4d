// Host-side declarations shared by the translation units of libtail.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tail {

constexpr int KSTEP = 16;            // k extent of one mma.sync / one ring stage
constexpr int MTILE_ROWS = 8;        // batch rows per m-tile (hi and lo parts stacked to 16)
constexpr int APACK_TILE_BYTES = 512;  // one 16x16 bf16 A fragment set: 32 lanes x 16 bytes
constexpr int MAX_ROWS_PER_PASS = 64;  // rows one lm_head pass covers (mt <= 8)
constexpr int GEMV_CONSUMER_WARPS = 8;
constexpr int GEMV_THREADS = (GEMV_CONSUMER_WARPS + 1) * 32;
constexpr int HIST_BINS = 2048;      // radix digit histogram of the selections (11-bit digits)
constexpr int MAX_K = 1024;
constexpr int MERGE_THREADS = 256;
constexpr uint64_t DEFAULT_TIMEOUT_NS = 1000000000ull;  // 1 s bound on every device wait

// Slab c of nslab covers column pairs [pair_lo(c), pair_lo(c+1)) of V/16 pairs.
__host__ __device__ inline int64_t slab_pair_lo(int64_t npairs, int nslab, int c) { return npairs * c / nslab; }

struct RmsArgs {
  const void* hidden;
  int dtype;
  const float* gamma;
  int B;          // rows of this pass
  int B_pad;      // rows written into the pack (multiple of 8)
  int H, Hu;
  float eps;
  int zero_pad;
  int deferred;
  uint32_t* apack;   // [H/16][mt][32][4] u32
  float* row_scale;  // [B_pad]: rstd (deferred) or 1
  int mt;
};

struct GemvArgs {
  const uint16_t* w;        // [H, V] bf16
  const uint8_t* apack;     // [ksteps][mt][512 B]
  const float* row_scale;   // [B_pad]
  float* logits_out;        // [B, V] caller logits for this pass, or null
  int64_t logits_out_ld;    // row stride of logits_out in floats
  float* logits_scratch;    // [B, V] staging when the slab logits do not fit in shared memory
  uint32_t* cand_key;       // [B][nslab][K] order keys
  int32_t* cand_idx;        // [B][nslab][K] vocabulary ids
  int* err;
  int B, H, V, K, ksteps, mt, nslab;
  int64_t npairs;
  int cb_pairs;             // column-block width in 16-column pairs
  int pitch;                // shared-memory row pitch of a W stage, bytes
  int stage_bytes, nstages;
  int logits_in_smem;
  int max_slab_cols;
  int smem_bytes;
  uint64_t timeout_ns;
};

struct MergeArgs {
  const uint32_t* cand_key;  // stage-1 output
  const int32_t* cand_idx;
  uint32_t* m1_key;          // [B][G][K]
  int32_t* m1_idx;
  int32_t* m1_cnt;           // [B][G]
  float* topk_val;           // [B][K] sorted output (caller or scratch)
  int32_t* topk_idx;
  int64_t topk_ld;           // row stride of topk outputs
  const float* params;       // [B][ncols] or null
  int ncols;
  int32_t* tokens;           // [B] or null
  int B, V, K, nslab, G;
  int64_t npairs;
  int* err;
};

// Launchers (all enqueue on `stream` with programmatic dependent launch).
cudaError_t launch_rms_pack(const RmsArgs& a, cudaStream_t stream);
cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t stream);
cudaError_t prepare_gemv(int max_smem);  // per device: opt the lm_head kernels into max_smem bytes
cudaError_t prepare_merge(int max_smem);
cudaError_t launch_merge1(const MergeArgs& a, cudaStream_t stream);
cudaError_t launch_merge2_sample(const MergeArgs& a, cudaStream_t stream);

// Shared-memory plan of the lm_head kernel for a pass of B rows.
struct GemvPlan {
  int mt, pw, cb_pairs, pitch, stage_bytes, nstages, logits_in_smem, max_slab_cols, smem_bytes;
  bool ok;
};
GemvPlan plan_gemv(int B, int H, int V, int K, int nslab, int max_smem);
int merge_groups(int nslab, int K);
size_t merge1_smem_bytes(int nslab, int G, int K);
size_t merge2_smem_bytes(int G, int K);

}  // namespace tail
