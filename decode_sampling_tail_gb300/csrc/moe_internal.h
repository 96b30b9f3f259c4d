// Host-side declarations of the producer step (MoE combine + residual add).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tail {

// The step that forms the bf16 hidden state ahead of the tail.
struct MoeArgs {
  const uint16_t* x;        // [B][H] bf16 residual
  const void* slots;        // [B][S][H] expert outputs, fp32 (slot_dtype 0) or bf16 (2)
  int slot_dtype;
  const float* w;           // [B][S] slot weights
  uint16_t* h;              // [B][H] bf16 hidden state (4-byte aligned)
  int B, H, S;
};
cudaError_t launch_moe_combine(const MoeArgs& a, cudaStream_t stream, bool pdl);

}  // namespace tail
