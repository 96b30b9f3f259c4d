// Host-side declarations shared by the translation units of libtail.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_internal.h"

namespace tail {

constexpr int KSTEP = 16;            // k extent of one mma.sync / one ring stage
constexpr int MTILE_ROWS = 8;        // batch rows per m-tile (hi and lo parts stacked to 16)
constexpr int APACK_TILE_BYTES = 512;  // one 16x16 bf16 A fragment set: 32 lanes x 16 bytes
constexpr int MAX_ROWS_PER_PASS = 64;  // rows one lm_head pass covers (mt <= 8)
constexpr int GEMV_CONSUMER_WARPS = 8;
constexpr int GEMV_PRODUCER_WARP = GEMV_CONSUMER_WARPS;      // weight (and packed activation) copies
constexpr int GEMV_PACK_WARP = GEMV_CONSUMER_WARPS + 1;      // activations built in-kernel (fused RMSNorm)
constexpr int GEMV_THREADS = (GEMV_CONSUMER_WARPS + 2) * 32;
constexpr int FUSED_MAX_MT = 2;      // the lm_head kernel forms the activations itself for up to 16 rows
constexpr int HID_DEPTH = 4;         // fused: stages of hidden columns in flight (async copies)
constexpr int HID_ROW_BYTES = 128;   // one row's 32 k columns, fp32 at most
constexpr int HID_SLOT_BYTES = FUSED_MAX_MT * 8 * HID_ROW_BYTES;
constexpr int GEMV_KPB = 2;          // ring stage = 32 rows of W
constexpr int GEMV_MAX_STAGES = 8;
constexpr int MAX_K = 1024;
constexpr int MAX_SLABS = 160;       // vocabulary slabs (lm_head CTAs) at most
constexpr int SLAB_LEADERS = 8;      // lane maxima behind each (row, slab)'s publication bound b
constexpr int SLAB_BOUND_KEYS = 4;   // of them, published for the owner's global bound
constexpr int SLAB_META_WORDS = 8;   // per (row, slab): 4 leader keys, candidate count, b, 2 spare
constexpr int SLAB_CAND = 32;        // candidate slots per (row, slab); more elements >= b: none published
constexpr int RANK_SORT_MAX = 640;   // up to this many candidates the row owner ranks them all directly
constexpr uint64_t DEFAULT_TIMEOUT_NS = 1000000000ull;  // 1 s bound on every device wait

// Slab c of nslab covers column pairs [pair_lo(c), pair_lo(c+1)) of V/16 pairs:
// floor(npairs * c / nslab), written as q * c + floor(r * c / nslab) with
// npairs = q * nslab + r so that only 32-bit divisions occur (npairs < 2^27).
__host__ __device__ inline int64_t slab_pair_lo(int64_t npairs, int nslab, int c) {
  const int np = static_cast<int>(npairs);
  return static_cast<int64_t>(np / nslab) * c + (np % nslab) * c / nslab;
}

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
  const uint8_t* apack;     // [ksteps][mt][512 B] (not fused)
  const float* row_scale;   // [B_pad] (not fused)
  // fused: the kernel forms the activations x * gamma (deferred RMSNorm) and rstd itself
  int fused;
  const void* hidden;       // [B, H] of hidden_dtype
  int dtype;
  const float* gamma;       // [H]
  int Hu;
  float eps;
  int zero_pad;
  float* logits_out;        // [B, V] caller logits for this pass, or null
  int64_t logits_out_ld;    // row stride of logits_out in floats
  float* logits_scratch;    // [B, V] the logits when the caller takes none (the row owner rescans it)
  uint32_t* meta;           // [B][nslab][SLAB_META_WORDS] each slab's publication per row
  uint64_t* cand;           // [B][nslab][SLAB_CAND] published candidates as (key, id) composites
  unsigned long long* row_sync;  // [B]: slabs that have published the row; 0 between runs
  unsigned long long* row_copy;  // [B]: slabs whose logits copy of the row is written; 0 between runs
  float* topk_val;          // [B][topk_ld] sorted top-k logits
  int32_t* topk_idx;        // [B][topk_ld] their vocabulary ids
  int64_t topk_ld;
  const float* params;      // [B][ncols] sampling parameters, or null
  int ncols;
  int32_t* tokens;          // [B], or null
  int* err;
  int B, H, V, K, ksteps, mt, nslab;
  int64_t npairs;
  int cb_pairs;             // column-block width in 16-column pairs
  int kpb;                  // k-steps of 16 rows per ring stage
  int pitch;                // shared-memory row pitch of a W stage, bytes
  int stage_bytes, nstages;
  int logits_in_smem;
  int max_slab_cols;
  int smem_bytes;
  int capc;                 // row owner candidate capacity (shared memory)
  int sortP;                // composite buffer entries: max(next power of two >= K, RANK_SORT_MAX)
  uint64_t timeout_ns;
  int drop_iter;            // test hook: ring iteration the producer never issues (-1: none)
  // fused form only: bytes of one slot of the hidden staging ring, and the producer step (the
  // activation warp forms each row from the residual and up to MOE_FUSED_MAX_SLOTS expert slots)
  int hid_slot_bytes = HID_SLOT_BYTES;
  int use_moe = 0;
  MoeIn moe;
  // producer step: tensor maps of this pass's residual rows (2-D [B][H] bf16, box 32 x B) and
  // slots (3-D [B][S][H], box 32 x MOE_FUSED_MAX_SLOTS x B: slots past S read as zeros)
  CUtensorMap moe_map_x;
  CUtensorMap moe_map_y;
};
// Byte offsets inside a staging slot of the producer-step form: the residual rows (64 bytes each),
// then, from moe_y_offset, MOE_FUSED_MAX_SLOTS slot rows of 32 elements per batch row.
__host__ __device__ inline int moe_y_offset(int B) { return (B * 64 + 127) & ~127; }
__host__ __device__ inline int moe_slot_bytes_for(int B) { return moe_y_offset(B) + B * MOE_FUSED_MAX_SLOTS * 32 * 4; }

// Launchers (all enqueue on `stream`; the lm_head tail is one launch,
// chained to the previous kernel on the stream with programmatic dependent launch when pdl).
cudaError_t launch_rms_pack(const RmsArgs& a, cudaStream_t stream, bool pdl = true);
cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t stream, bool pdl);
// per device: opt the lm_head kernels into the largest dynamic shared memory
// the opt-in limit leaves after their static shared memory
cudaError_t prepare_gemv(int max_smem_optin, int* max_dynamic);

// Shared-memory plan of the lm_head kernel for a pass of B rows.
struct GemvPlan {
  int mt, pw, cb_pairs, pitch, kpb, stage_bytes, nstages, logits_in_smem, max_slab_cols, smem_bytes;
  int capc, sortP;
  int hid_slot_bytes;  // one slot of the fused form's hidden staging ring
  bool ok;
};
// kpb: k-steps per ring stage (1 or 2); max_stages caps the ring depth.  moe_slots >= 0 plans the
// fused form with the producer step inside the kernel: its hidden staging ring then holds the
// bf16 residual and that many expert slots of moe_slot_bytes (4: fp32, 2: bf16) per element.
GemvPlan plan_gemv(int B, int H, int V, int K, int nslab, int max_smem, int kpb = GEMV_KPB,
                   int max_stages = GEMV_MAX_STAGES, int moe_slots = -1, int moe_slot_bytes = 4);
constexpr int SEL_NPL = 48;          // register keys per lane of the slab selects: slabs up to 1536 columns

}  // namespace tail
