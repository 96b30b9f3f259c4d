// Host-side declarations of the stage-1 tap export.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tail {

enum TapKind : int { TAP_SLABS = 1, TAP_TILES = 2 };

struct TapArgs {
  int kind;                  // TAP_SLABS: meta + cand of the mma.sync pass; TAP_TILES: the tile lists
  const uint32_t* meta;      // [B][nchunk][SLAB_META_WORDS]
  const uint64_t* cand;      // [B][nchunk][SLAB_CAND]
  const uint64_t* lists;     // [B][nchunk][TC_LIST]
  int B, V, nchunk, cap, tile_n;
  float* vals;               // [B][nchunk][cap]
  int32_t* idx;              // [B][nchunk][cap]
  int32_t* count;            // [B][nchunk]
  float* bound;              // [B][nchunk]
};

cudaError_t launch_tap_export(const TapArgs& a, cudaStream_t stream);

}  // namespace tail
