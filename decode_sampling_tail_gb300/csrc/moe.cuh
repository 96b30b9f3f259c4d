// Device form of the tail's producer step, the MoE combine + residual add
// ("nemotron CUDA: RMSNorm rows run on the shared norms and combine (#548,
// step 1)", TensorFold pull request #1353, section "What moves", entry
// tf_nemo_add_moe_norm, with the author's fix reply: the fused residual keeps
// the routed chain and the shared sum apart).  Per hidden lane:
//   r  = 0;  r  = fma(w_s, y_s, r)  for the routed slots s = 0 .. n_routed-1
//   sh = 0;  sh = fma(w_s, y_s, sh) for the shared slots s = n_routed .. S-1
//   h  = bf16(x + bf16(r + sh))
// with IEEE fp32 fmas and adds (no contraction) and bf16 rounding to nearest,
// ties to even.  Nemotron's 2 shared slots carry weight 1: each of their fmas
// is the plain add s0 + s1.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_internal.h"

namespace tail {

__device__ __forceinline__ uint32_t moe_bf16_bits(float v) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

__device__ __forceinline__ float moe_slot_value(const void* slots, int dtype, int64_t i) {
  if (dtype == 0) return static_cast<const float*>(slots)[i];
  return __bfloat162float(static_cast<const __nv_bfloat16*>(slots)[i]);
}

// One step of the two chains: slot s goes to r when routed, else to sh.
__device__ __forceinline__ void moe_accumulate(int s, int n_routed, float w, float y, float& r, float& sh) {
  const float acc = __fmaf_rn(w, y, s < n_routed ? r : sh);
  if (s < n_routed)
    r = acc;
  else
    sh = acc;
}

// h = bf16(x + bf16(r + sh)) as bf16 bits, x given as bf16 bits
__device__ __forceinline__ uint32_t moe_finish(uint32_t x_bits, float r, float sh) {
  const float d = __uint_as_float(moe_bf16_bits(__fadd_rn(r, sh)) << 16);
  return moe_bf16_bits(__fadd_rn(__uint_as_float(x_bits << 16), d));
}

// h[b][j] as bf16 bits, reading the slots straight from global memory.
__device__ __forceinline__ uint32_t moe_lane_h(const MoeIn& m, int64_t b, int H, int j) {
  const float* w = m.w + b * m.S;
  float r = 0.f, sh = 0.f;
  for (int s = 0; s < m.S; ++s)
    moe_accumulate(s, m.n_routed, w[s], moe_slot_value(m.slots, m.slot_dtype, (b * m.S + s) * H + j), r, sh);
  return moe_finish(static_cast<uint32_t>(m.x[b * H + j]), r, sh);
}

}  // namespace tail
