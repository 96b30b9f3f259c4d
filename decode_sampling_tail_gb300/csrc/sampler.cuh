// Per-row sampler of the tail ("GPT-OSS Tail Chunked Megakernel Kernel API
// Reference", parameter `sampling_params`: per row [top_k, top_p, temperature]
// and an optional inverse-transform draw u in [0, 1), 0.5 when the 4th column
// is absent).  All threads of the CTA, over the row's candidates sorted by
// (logit desc, index asc), l_0 >= l_1 >= ...:
//   kk = trunc(top_k) when 1 <= top_k < n + 1, else n (the cut is disabled);
//   temperature <= 0 (or NaN) or kk == 1: greedy, token = idx_0;
//   e_i = exp((l_i - l_0) / T) for i < kk, S_j = sum_{i<=j} e_i, Z = S_{kk-1};
//   m = kk when top_p >= 1, else the smallest j+1 with S_j >= top_p * Z;
//   token = idx_j for the smallest j < m with u * S_{m-1} < S_j, else idx_{m-1}.
// The running sums use one fixed order (each thread sums a contiguous chunk on
// top of the block-scanned sum of the chunks before it), so a row's token never
// depends on the batch it runs in.
#pragma once

#include "common.cuh"
#include "select.cuh"

namespace tail {

// Block-wide exclusive prefix sum of one float per thread (fixed order: within
// a warp by its shuffle scan, then the warp totals in warp order).  red: 64
// floats of shared scratch.  Returns the exclusive prefix; *total the sum.
__device__ __forceinline__ float block_excl_scan(float v, float* red, float* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  float base = 0.f, tot = 0.f;
  for (int w = 0; w < nw; ++w) {
    const float x = red[w];
    if (w < warp) base += x;
    tot += x;
  }
  *total = tot;
  __syncthreads();  // red is reused by the caller
  return base + incl - v;
}

__device__ __forceinline__ unsigned block_min_u32(unsigned v, unsigned* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = __reduce_min_sync(0xffffffffu, v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  unsigned m = 0xffffffffu;
  for (int w = 0; w < nw; ++w) m = min(m, red[w]);
  __syncthreads();
  return m;
}

// The draw, with every thread of the CTA.  sorted[0..nc): composites in
// descending order; ebuf: nc floats and red: 64 words of shared scratch.
// Thread t owns the contiguous candidates [t*E, (t+1)*E) (E = ceil(kk / threads)),
// so S_j = (sum over the chunks before t's) + e_{tE} + ... + e_j in one fixed
// order: a row's token does not depend on the batch it runs in.  Every
// thread returns the token.
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

__device__ __forceinline__ int32_t sample_sorted_row(const SampleParams& sp, const uint64_t* sorted, int nc,
                                                     float* ebuf, float* red) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const float top_k = sp.top_k, top_p = sp.top_p, temp = sp.temp, u = sp.u;
  auto val_at = [&](int i) { return key_float(composite_key(sorted[i])); };
  const int kk = (top_k >= 1.0f && top_k < static_cast<float>(nc) + 1.0f) ? static_cast<int>(top_k) : nc;
  if (!(temp > 0.0f) || kk == 1) return composite_idx(sorted[0]);
  const float l0 = val_at(0);
  const int E = (kk + nt - 1) / nt;
  const int i0 = min(kk, tid * E), i1 = min(kk, i0 + E);
  float ls = 0.f;
  for (int i = i0; i < i1; ++i) {
    const float e = expf((val_at(i) - l0) / temp);
    ebuf[i] = e;
    ls += e;
  }
  float Z;
  const float excl = block_excl_scan(ls, red, &Z);  // Z = S_{kk-1}
  unsigned* ured = reinterpret_cast<unsigned*>(red);
  int m = kk;
  if (top_p < 1.0f) {
    const float tp = top_p * Z;
    unsigned found = 0xffffffffu;
    float S = excl;
    for (int i = i0; i < i1; ++i) {
      S += ebuf[i];
      if (S >= tp) {
        found = static_cast<unsigned>(i);
        break;
      }
    }
    found = block_min_u32(found, ured);
    m = found == 0xffffffffu ? kk : static_cast<int>(found) + 1;
  }
  // C_{m-1}, from the thread that owns candidate m - 1
  float Cm = Z;
  if (m < kk) {
    if (i0 <= m - 1 && m - 1 < i1) {
      float S = excl;
      for (int i = i0; i <= m - 1; ++i) S += ebuf[i];
      red[32] = S;
    }
    __syncthreads();
    Cm = red[32];
    __syncthreads();
  }
  const float target = u * Cm;
  unsigned pick = 0xffffffffu;
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
  pick = block_min_u32(pick, ured);
  const int j = pick == 0xffffffffu ? m - 1 : static_cast<int>(pick);
  return composite_idx(sorted[j]);
}

}  // namespace tail
