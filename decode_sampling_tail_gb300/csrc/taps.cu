// Stage-1 taps: the chunked top-k's per-chunk output, exported for inspection
// ("GPT-OSS Tail Chunked Megakernel Kernel API Reference", parameter
// `debug_taps`: the stage taps that let a hardware-only index defect be seen;
// section "Background": the chunked top-k's first stage feeds one global
// top-k).  A chunk is a vocabulary slab of the mma.sync lm_head kernel or a
// column tile of the tensor-core lm_head.  For every (row, chunk) the export
// writes the candidates the chunk handed to the merge (logit and vocabulary
// id), their count, and a bound: every element of the chunk that is not among
// its candidates has a logit <= bound.
//   slab (mma.sync): candidates = every element >= b, the chunk's publication
//     bound, when they fit its slots (bound = b); none otherwise (bound = +inf:
//     every element may be hidden, and the merge rescans the slab when it needs to)
//   tile (tensor cores): candidates = the tile's top TC_LIST by (value desc,
//     column asc); bound = the last of them, or -inf when they are all of its columns
// One thread per (row, chunk, slot); slots past the count hold (-inf, -1).
#include "common.cuh"
#include "internal.h"
#include "select.cuh"
#include "taps_internal.h"
#include "tc_internal.h"

namespace tail {

namespace {

constexpr int TAP_THREADS = 256;

__global__ void __launch_bounds__(TAP_THREADS) tap_export_kernel(const TapArgs a) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * TAP_THREADS + threadIdx.x;
  const int64_t total = static_cast<int64_t>(a.B) * a.nchunk * a.cap;
  if (i >= total) return;
  const int j = static_cast<int>(i % a.cap);
  const int64_t rc = i / a.cap;  // row * nchunk + chunk
  const int c = static_cast<int>(rc % a.nchunk);
  int count;
  float bound;
  uint64_t comp = 0ull;
  if (a.kind == TAP_SLABS) {
    const uint32_t* m = a.meta + rc * SLAB_META_WORDS;
    const uint32_t b = m[5];
    const bool fits = b != 0xFFFFFFFFu;
    count = fits ? static_cast<int>(m[4]) : 0;
    bound = fits ? key_float(b) : __int_as_float(0x7f800000);
    if (j < count) comp = a.cand[rc * SLAB_CAND + j];
  } else {
    const int64_t c0 = static_cast<int64_t>(c) * a.tile_n;
    const int width = static_cast<int>(min(static_cast<int64_t>(a.tile_n), static_cast<int64_t>(a.V) - c0));
    const uint64_t* l = a.lists + rc * TC_LIST;
    count = 0;
#pragma unroll
    for (int q = 0; q < TC_LIST; ++q) count += composite_key(l[q]) != 0u ? 1 : 0;
    bound = count >= width ? __int_as_float(0xff800000) : key_float(composite_key(l[TC_LIST - 1]));
    if (j < count) comp = l[j];
  }
  a.vals[i] = j < count ? key_float(composite_key(comp)) : __int_as_float(0xff800000);
  a.idx[i] = j < count ? composite_idx(comp) : -1;
  if (j == 0) {
    a.count[rc] = count;
    a.bound[rc] = bound;
  }
}

}  // namespace

cudaError_t launch_tap_export(const TapArgs& a, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(a.B) * a.nchunk * a.cap;
  if (total == 0) return cudaSuccess;
  tap_export_kernel<<<static_cast<unsigned>((total + TAP_THREADS - 1) / TAP_THREADS), TAP_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace tail
