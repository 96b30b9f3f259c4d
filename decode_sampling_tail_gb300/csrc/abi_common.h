// Host helpers shared by the C-ABI translation units: config validation, the
// thread's last-error text and small argument checks.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tail.h"

namespace tail {

// Records the failing CUDA call for tail_last_error(), clears CUDA's non-sticky
// error state and returns TAIL_ERR_OOM or TAIL_ERR_CUDA.
int cuda_fail(cudaError_t e, const char* what);
// Sets the text tail_last_error() returns on this thread.
void set_last_error(const char* msg);
// TAIL_OK, or the status a config with these sizes earns (shared by every entry point).
int validate_config(const tail_config* c);

inline int elem_bytes(int dtype) { return dtype == TAIL_F32 ? 4 : 2; }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Vocabulary slabs (= lm_head CTAs): one per SM, at least 8 column pairs
// (128 columns) per slab, at most `max_slabs`.
inline int slab_count(int64_t npairs, int num_sms, int max_slabs) {
  int64_t nslab = npairs / 8;
  if (nslab < 1) nslab = 1;
  if (nslab > num_sms) nslab = num_sms;
  if (nslab > max_slabs) nslab = max_slabs;
  return static_cast<int>(nslab);
}

}  // namespace tail
