// Per-row sampler of the tail ("GPT-OSS Tail Chunked Megakernel Kernel API
// Reference", parameter `sampling_params`: per row [top_k, top_p, temperature]
// and an optional inverse-transform draw u in [0, 1), 0.5 when the 4th column
// is absent).  One warp, over the row's candidates sorted by (logit desc,
// index asc), l_0 >= l_1 >= ...:
//   kk = trunc(top_k) when 1 <= top_k < n + 1, else n (the cut is disabled);
//   temperature <= 0 (or NaN) or kk == 1: greedy, token = idx_0;
//   e_i = exp((l_i - l_0) / T) for i < kk, S_j = sum_{i<=j} e_i, Z = S_{kk-1};
//   m = kk when top_p >= 1, else the smallest j+1 with S_j >= top_p * Z;
//   token = idx_j for the smallest j < m with u * S_{m-1} < S_j, else idx_{m-1}.
// The running sums use one fixed order: lane l sums its contiguous chunk of
// E = ceil(kk / 32) candidates on top of the warp-scanned sum of the chunks
// before it.  It depends on kk only, so a row's token never depends on the
// batch, the kernel or the block size it runs in.
#pragma once

#include "common.cuh"
#include "select.cuh"

namespace tail {

// The row's parameters, read once (early, so their latency overlaps other work).
struct SampleParams {
  float top_k, top_p, temp, u;
};
__device__ __forceinline__ SampleParams load_sample_params(const float* p, int ncols) {
  SampleParams sp;
  sp.top_k = __ldg(p);
  sp.top_p = __ldg(p + 1);
  sp.temp = __ldg(p + 2);
  sp.u = ncols == 4 ? __ldg(p + 3) : 0.5f;
  return sp;
}

// The draw, by one whole warp (every lane returns the token).  sorted[0, nc):
// composites in descending order; ebuf: nc floats of shared scratch (each lane
// writes and reads only its own chunk).
__device__ __forceinline__ int32_t sample_sorted_warp(const SampleParams& sp, const uint64_t* sorted, int nc,
                                                      float* ebuf) {
  const int lane = threadIdx.x & 31;
  const float top_k = sp.top_k, top_p = sp.top_p, temp = sp.temp, u = sp.u;
  auto val_at = [&](int i) { return key_float(composite_key(sorted[i])); };
  const int kk = (top_k >= 1.0f && top_k < static_cast<float>(nc) + 1.0f) ? static_cast<int>(top_k) : nc;
  if (!(temp > 0.0f) || kk == 1) return composite_idx(sorted[0]);
  const float l0 = val_at(0);
  const int E = (kk + 31) >> 5;
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
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);      // sum of the chunks before this lane's
  if (lane == 0) excl = 0.f;
  const float Z = __shfl_sync(0xffffffffu, incl, 31);     // S_{kk-1}
  int m = kk;
  float Cm = Z;                                           // S_{m-1}
  if (top_p < 1.0f) {
    const float tp = top_p * Z;
    int found = -1;
    float S = excl, Sf = 0.f;
    for (int i = i0; i < i1; ++i) {
      S += ebuf[i];
      if (S >= tp) {
        found = i;
        Sf = S;
        break;
      }
    }
    const uint32_t who = __ballot_sync(0xffffffffu, found >= 0);
    if (who != 0u) {
      const int src = __ffs(who) - 1;
      m = __shfl_sync(0xffffffffu, found, src) + 1;
      Cm = __shfl_sync(0xffffffffu, Sf, src);
    }
  }
  const float target = u * Cm;
  int pick = -1;
  {
    float S = excl;
    for (int i = i0; i < min(i1, m); ++i) {
      S += ebuf[i];
      if (target < S) {
        pick = i;
        break;
      }
    }
  }
  const uint32_t who = __ballot_sync(0xffffffffu, pick >= 0);
  const int j = who != 0u ? __shfl_sync(0xffffffffu, pick, __ffs(who) - 1) : m - 1;
  return composite_idx(sorted[j]);
}

}  // namespace tail
