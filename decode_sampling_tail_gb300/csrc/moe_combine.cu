// The tail's producer step as a kernel of its own: the MoE combine and
// residual add that form the bf16 hidden state the final RMSNorm reads (the
// arithmetic is in moe.cuh: the routed fma chain and the shared-slot chain
// kept apart, their sum rounded to bf16, added to the residual, rounded to
// bf16).  One thread per (row, column pair); the launch is chained to the
// tail's first kernel with programmatic dependent launch.  It serves the
// forms that do not combine inside their first kernel (more than
// MOE_FUSED_MAX_SLOTS slots, or a pass whose lm_head kernel takes its
// activations from the RMSNorm kernel).
#include "common.cuh"
#include "internal.h"
#include "moe.cuh"

namespace tail {

namespace {

constexpr int MOE_THREADS = 256;

__global__ void __launch_bounds__(MOE_THREADS) moe_combine_kernel(const MoeIn m, int H) {
  pdl_wait();  // the slots may come from the previous kernel; h is reused across steps
  pdl_launch_dependents();
  const int b = blockIdx.y;
  const int j2 = 2 * (blockIdx.x * MOE_THREADS + threadIdx.x);  // columns j2, j2 + 1
  if (j2 >= H) return;
  const uint32_t h0 = moe_lane_h(m, b, H, j2);
  const uint32_t h1 = moe_lane_h(m, b, H, j2 + 1);
  *reinterpret_cast<uint32_t*>(m.h_out + static_cast<int64_t>(b) * H + j2) = h0 | (h1 << 16);
}

}  // namespace

cudaError_t launch_moe_combine(const MoeIn& m, int B, int H, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((H / 2 + MOE_THREADS - 1) / MOE_THREADS, B);
  cfg.blockDim = dim3(MOE_THREADS);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, moe_combine_kernel, m, H);
}

}  // namespace tail
