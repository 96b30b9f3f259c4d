// Host-side declarations of the producer step (MoE combine + residual add).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tail {

// The step that forms the bf16 hidden state ahead of the tail, for one lane j of row b:
//   r  = fp32 fma chain over the routed slots s < n_routed (index order, from 0)
//   sh = the same chain over the shared slots s >= n_routed
//   h  = bf16(x + bf16(r + sh))
struct MoeIn {
  const uint16_t* x = nullptr;     // [B][H] bf16 residual
  const void* slots = nullptr;     // [B][S][H] expert outputs, fp32 (slot_dtype 0) or bf16 (2)
  int slot_dtype = 0;
  const float* w = nullptr;        // [B][S] slot weights
  int S = 0;                       // slots per row; 0: no producer step
  int n_routed = 0;                // the first n_routed slots are routed, the rest shared
  uint16_t* h_out = nullptr;       // [B][H] bf16 h, or null
};

// Slots the lm_head kernel's activation warp combines itself (Nemotron: 6 routed + 2 shared).
constexpr int MOE_FUSED_MAX_SLOTS = 8;

// The combine as a kernel of its own: h for every row into m.h_out (4-byte aligned).
cudaError_t launch_moe_combine(const MoeIn& m, int B, int H, cudaStream_t stream, bool pdl);

}  // namespace tail
