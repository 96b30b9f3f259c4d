// Host-side declarations of the one-launch tail for small problems (the
// latency path: cfg.path = TAIL_PATH_SMALL).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tail {

constexpr int SMALL_THREADS = 512;
constexpr int SMALL_MAX_ROWS = 8;      // rows a launch covers: one owner CTA each
constexpr int SMALL_MAX_H = 8192;
constexpr int SMALL_MAX_V = 16384;     // a row's keys and indices sit in one CTA's shared memory
static_assert(SMALL_MAX_V % SMALL_THREADS == 0, "the owner holds SMALL_MAX_V / SMALL_THREADS keys a thread");
constexpr int SMALL_PREFETCH = 4;      // weight chunks a thread loads before the dependency wait
constexpr int SMALL_MAX_SLABS = 160;   // CTAs a launch may have (5 slab maxima a lane of one warp)

struct SmallArgs {
  const void* hidden = nullptr;  // [B][H], dtype 0 fp32, 1 fp16, 2 bf16
  int dtype = 0;
  const float* gamma = nullptr;  // [H]
  const uint16_t* w = nullptr;   // [H][V] bf16 bits
  float* logits = nullptr;       // [B][V] fp32: the caller's, or the handle's scratch
  float* topk_val = nullptr;     // [B][topk_ld]
  int32_t* topk_idx = nullptr;
  int topk_ld = 0;
  const float* params = nullptr;  // [B][ncols] or null: no draw
  int ncols = 0;
  int32_t* tokens = nullptr;
  unsigned long long* sync = nullptr;  // [B] arrival words, zero between launches
  uint32_t* smax = nullptr;            // [B][nslab] each slab's largest order key of the row
  int* err = nullptr;
  uint64_t timeout_ns = 0;
  int B = 0, H = 0, Hu = 0, V = 0, K = 0;
  int zero_pad = 0, deferred = 1;
  float eps = 0.f;
  int slab_cols = 0;  // columns of one CTA's slab (a multiple of 8)
  int nslab = 0;      // CTAs: ceil(V / slab_cols)
  int sortP = 0;      // a power of two >= K
  int cap = 0;        // composites the owner's gather holds (a multiple of 32, >= sortP)
  int smem_bytes = 0;
};

struct SmallPlan {
  bool ok = false;
  int slab_cols = 0, nslab = 0, sortP = 0, cap = 0, smem_bytes = 0;
};

// The launch shape for up to B rows of an H x V problem on num_sms SMs with dyn_max bytes of
// dynamic shared memory a CTA; ok is false when the problem is outside the path's limits.
SmallPlan plan_small(int B, int H, int V, int K, int num_sms, int dyn_max);

// Raises the kernel's dynamic shared memory limit to what the opt-in limit leaves beside its static
// shared memory, and returns that in *dyn_max.
cudaError_t prepare_small(int max_smem_optin, int* dyn_max);

cudaError_t launch_small(const SmallArgs& a, cudaStream_t stream, bool pdl);

}  // namespace tail
