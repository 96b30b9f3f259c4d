// The tensor-core lm_head's own copy of the weight ("GPT-OSS Tail Chunked
// Megakernel Kernel API Reference", parameter `lm_head_weight_t`: the [H][V]
// weight, read once a step).  The copy holds the same bf16 values laid out as
// the shared-memory image the MMA reads, so that one weight ring stage (the
// 64-column boxes of one column tile at one k-block) arrives as a single
// contiguous bulk copy instead of one tensor-tile request per box.
//
// Block (kb, g), 8 KB, covers k-rows [64 kb, 64 kb + 64) and columns
// [64 g, 64 g + 64).  Its k-row r is the 128 bytes at r * 128; the 16-byte
// chunk c of that row (columns 64 g + 8 c .. + 8) sits at chunk position
// c ^ (r & 7), the 128-byte swizzle of the MMA's B descriptor.  Blocks are
// k-block major: (kb, g) starts at (kb * groups + g) * 8 KB, so the groups of a
// column tile are adjacent within a k-block.  Rows past H and columns past V
// are zero, as the tensor-tile loads fill them.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tc_internal.h"

namespace tail {

namespace {

__global__ void __launch_bounds__(256) weight_pack_kernel(const uint16_t* __restrict__ w, int H, int V, int kblocks,
                                                          int groups, uint8_t* __restrict__ out) {
  // one 16-byte chunk per step; consecutive steps read consecutive chunks of a weight row
  const int64_t total = static_cast<int64_t>(kblocks) * 64 * groups * 8;
  for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; q < total;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(q & 7);
    const int64_t rg = q >> 3;
    const int g = static_cast<int>(rg % groups);
    const int h = static_cast<int>(rg / groups);  // k-row: 64 kb + r
    const int kb = h >> 6, r = h & 63;
    const int col = 64 * g + 8 * c;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (h < H && col < V)  // V is a multiple of 16: the chunk is whole
      v = *reinterpret_cast<const uint4*>(w + static_cast<int64_t>(h) * V + col);
    const int64_t dst = ((static_cast<int64_t>(kb) * groups + g) * 64 + r) * 128 + ((c ^ (r & 7)) << 4);
    *reinterpret_cast<uint4*>(out + dst) = v;
  }
}

}  // namespace

int64_t tc_packed_weight_bytes(int H, int V) {
  return static_cast<int64_t>(tc_kblocks(H)) * tc_weight_groups(V) * TC_W_BLOCK_BYTES;
}

cudaError_t launch_weight_pack(const uint16_t* w, int H, int V, uint8_t* out, int num_sms, cudaStream_t stream) {
  const int kblocks = tc_kblocks(H), groups = tc_weight_groups(V);
  weight_pack_kernel<<<4 * num_sms, 256, 0, stream>>>(w, H, V, kblocks, groups, out);
  return cudaGetLastError();
}

}  // namespace tail
