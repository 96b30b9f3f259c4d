// The tail's producer step: the MoE combine and residual add that form the
// bf16 hidden state the final RMSNorm reads ("nemotron CUDA: RMSNorm rows run
// on the shared norms and combine (#548, step 1)", TensorFold pull request
// #1353, section "What moves", entry tf_nemo_add_moe_norm: one fp32 fma per
// slot, slots in index order, then a bf16 rounding before the residual add).
// Per hidden lane j of row b:
//   acc = 0;  acc = fma(w[b][s], y[b][s][j], acc) for s = 0, 1, ..., S-1
//   h[b][j] = bf16(x[b][j] + bf16(acc))
// with IEEE fp32 fmas and adds and bf16 rounding to nearest, ties to even.
// One thread per (row, column pair); the launch is chained to the tail's
// first kernel with programmatic dependent launch.
#include "common.cuh"
#include "internal.h"
#include "moe_internal.h"

namespace tail {

namespace {

constexpr int MOE_THREADS = 256;

__device__ __forceinline__ float slot_value(const void* slots, int dtype, int64_t i) {
  if (dtype == 0) return static_cast<const float*>(slots)[i];
  return __bfloat162float(static_cast<const __nv_bfloat16*>(slots)[i]);
}

__device__ __forceinline__ uint32_t to_bf16_bits(float v) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

__global__ void __launch_bounds__(MOE_THREADS) moe_combine_kernel(const MoeArgs a) {
  pdl_wait();  // the slots may come from the previous kernel; h is reused across steps
  pdl_launch_dependents();
  const int b = blockIdx.y;
  const int j2 = 2 * (blockIdx.x * MOE_THREADS + threadIdx.x);  // columns j2, j2 + 1
  if (j2 >= a.H) return;
  const float* w = a.w + static_cast<int64_t>(b) * a.S;
  uint32_t out[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int j = j2 + t;
    float acc = 0.0f;
    for (int s = 0; s < a.S; ++s)
      acc = __fmaf_rn(w[s], slot_value(a.slots, a.slot_dtype, (static_cast<int64_t>(b) * a.S + s) * a.H + j), acc);
    const float d = __uint_as_float(to_bf16_bits(acc) << 16);
    const float x = __uint_as_float(static_cast<uint32_t>(a.x[static_cast<int64_t>(b) * a.H + j]) << 16);
    out[t] = to_bf16_bits(__fadd_rn(x, d));
  }
  *reinterpret_cast<uint32_t*>(a.h + static_cast<int64_t>(b) * a.H + j2) = out[0] | (out[1] << 16);
}

}  // namespace

cudaError_t launch_moe_combine(const MoeArgs& a, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.H / 2 + MOE_THREADS - 1) / MOE_THREADS, a.B);
  cfg.blockDim = dim3(MOE_THREADS);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, moe_combine_kernel, a);
}

}  // namespace tail
