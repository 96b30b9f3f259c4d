// Per-row sampler of the tail ("GPT-OSS Tail Chunked Megakernel Kernel API
// Reference", parameter `sampling_params`: per row [top_k, top_p, temperature]
// and an optional inverse-transform draw u in [0, 1), 0.5 when the 4th column
// is absent).  One warp, over the row's candidates sorted by
// (logit desc, index asc), l_0 >= l_1 >= ...:
//   kk = trunc(top_k) when 1 <= top_k < n + 1, else n (the cut is disabled);
//   temperature <= 0 (or NaN) or kk == 1: greedy, token = idx_0;
//   e_i = exp((l_i - l_0) / T) for i < kk, S_j = sum_{i<=j} e_i, Z = S_{kk-1};
//   m = kk when top_p >= 1, else the smallest j+1 with S_j >= top_p * Z;
//   token = idx_j for the smallest j < m with u * S_{m-1} < S_j, else idx_{m-1}.
// The running sums use one fixed order (each lane sums a contiguous chunk on
// top of the warp-scanned sum of the chunks before it), so a row's token never
// depends on the batch it runs in.
#pragma once

#include "common.cuh"
#include "select.cuh"

namespace tail {

// sorted[0..nc): composites in descending order; ebuf: nc floats of shared scratch.
__device__ __forceinline__ int32_t sample_sorted_row(const float* p, int ncols, const uint64_t* sorted, int nc,
                                                     float* ebuf) {
  const int lane = threadIdx.x & 31;
  const float top_k = p[0], top_p = p[1], temp = p[2];
  const float u = ncols == 4 ? p[3] : 0.5f;
  auto val_at = [&](int i) { return key_float(composite_key(sorted[i])); };
  const int kk = (top_k >= 1.0f && top_k < static_cast<float>(nc) + 1.0f) ? static_cast<int>(top_k) : nc;
  if (!(temp > 0.0f) || kk == 1) return composite_idx(sorted[0]);
  const float l0 = val_at(0);
  const int E = (kk + 31) / 32;
  const int i0 = min(kk, lane * E), i1 = min(kk, i0 + E);
  float ls = 0.f;
  for (int i = i0; i < i1; ++i) {
    const float e = expf((val_at(i) - l0) / temp);
    ebuf[i] = e;
    ls += e;
  }
  float incl = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.f;
  __syncwarp();
  // S_j = excl(owner lane of j) + e_{i0} + ... + e_j, the same order everywhere
  auto S_at = [&](int j) {
    const int owner = j / E;
    float S = excl;
    if (lane == owner)
      for (int i = i0; i <= j; ++i) S += ebuf[i];
    return __shfl_sync(0xffffffffu, S, owner);
  };
  const float Z = S_at(kk - 1);
  int m = kk;
  if (top_p < 1.0f) {
    const float tp = top_p * Z;
    unsigned found = 0x7fffffffu;
    float S = excl;
    for (int i = i0; i < i1; ++i) {
      S += ebuf[i];
      if (S >= tp) {
        found = static_cast<unsigned>(i);
        break;
      }
    }
    found = __reduce_min_sync(0xffffffffu, found);
    m = found == 0x7fffffffu ? kk : static_cast<int>(found) + 1;
  }
  const float Cm = S_at(m - 1);
  const float target = u * Cm;
  unsigned pick = 0x7fffffffu;
  {
    float S = excl;
    for (int i = i0; i < min(i1, m); ++i) {
      S += ebuf[i];
      if (target < S) {
        pick = static_cast<unsigned>(i);
        break;
      }
    }
  }
  pick = __reduce_min_sync(0xffffffffu, pick);
  const int j = pick == 0x7fffffffu ? m - 1 : static_cast<int>(pick);
  return composite_idx(sorted[j]);
}

}  // namespace tail
