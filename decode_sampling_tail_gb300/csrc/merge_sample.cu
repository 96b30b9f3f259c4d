// Global top-k merge and the per-row sampler.
//
// The stage-1 output holds, for every (row, vocabulary slab), the slab's top K
// in index order.  Their union contains the global top K of the row, because
// the global top K restricted to one slab is a subset of that slab's top K.
// Two launches reduce it ("GPT-OSS Tail Chunked Megakernel Kernel API
// Reference", section "Background": the global top-k is computed locally by a
// chunked top-k; parameter `k`):
//   merge1  grid (G, B): CTA (g, b) selects the top K of slab group g of row b;
//   merge2  grid (B):    CTA b selects the top K of the G group results, sorts
//                        them by (logit desc, index asc) and runs the sampler.
// Candidates stay in ascending vocabulary order through both selections, so
// ties at the boundary keep the lowest indices.
//
// Sampler (parameter `sampling_params`: per row [top_k, top_p, temperature]
// and an optional draw u in [0, 1), 0.5 when absent), one warp per row over
// the sorted candidates l_0 >= l_1 >= ...:
//   kk = trunc(top_k) when 1 <= top_k < n + 1, else n (disabled);
//   temperature <= 0 (or NaN) or kk == 1: greedy, token = idx_0;
//   e_i = exp((l_i - l_0) / T) for i < kk, S_j = sum_{i<=j} e_i, Z = S_{kk-1};
//   m = kk when top_p >= 1, else the smallest j+1 with S_j >= top_p * Z;
//   token = idx_j for the smallest j < m with u * S_{m-1} < S_j, else idx_{m-1}.
// The running sums use one fixed order (each lane sums a contiguous chunk,
// then a warp scan), so a row's token never depends on the batch.
#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace tail {

namespace {

constexpr int MERGE_CAP = 16384;  // candidates one merge CTA holds in shared memory

__device__ __forceinline__ int slab_cols(const MergeArgs& a, int s) {
  return static_cast<int>(slab_pair_lo(a.npairs, a.nslab, s + 1) - slab_pair_lo(a.npairs, a.nslab, s)) * 16;
}

__global__ void __launch_bounds__(MERGE_THREADS) merge1_kernel(const MergeArgs a) {
  extern __shared__ __align__(16) uint32_t sm[];
  pdl_wait();
  pdl_launch_dependents();
  const int g = blockIdx.x, b = blockIdx.y;
  const int s0 = static_cast<int>(static_cast<int64_t>(a.nslab) * g / a.G);
  const int s1 = static_cast<int>(static_cast<int64_t>(a.nslab) * (g + 1) / a.G);
  const int cap = ((s1 - s0) > 0 ? (a.nslab + a.G - 1) / a.G : 1) * a.K;
  uint32_t* keys = sm;
  int32_t* idx = reinterpret_cast<int32_t*>(sm + cap);
  uint32_t* hist = sm + 2 * cap;
  uint32_t* scan = hist + HIST_BINS;

  int n = 0;
  for (int s = s0; s < s1; ++s) {
    const int cnt = min(a.K, slab_cols(a, s));
    const int64_t base = (static_cast<int64_t>(b) * a.nslab + s) * a.K;
    for (int j = threadIdx.x; j < cnt; j += MERGE_THREADS) {
      keys[n + j] = a.cand_key[base + j];
      idx[n + j] = a.cand_idx[base + j];
    }
    n += cnt;
  }
  __syncthreads();
  const int want = min(a.K, n);
  const int64_t obase = (static_cast<int64_t>(b) * a.G + g) * a.K;
  Threshold th;
  if (want == n) {
    th.key = 0u;
    th.take_eq = -1;
  } else {
    th = block_select(keys, n, want, hist, scan);
  }
  block_compact(keys, n, th, scan, [&](int pos, int i, uint32_t k) {
    a.m1_key[obase + pos] = k;
    a.m1_idx[obase + pos] = idx[i];
  });
  if (threadIdx.x == 0) a.m1_cnt[static_cast<int64_t>(b) * a.G + g] = want;
}

__device__ __forceinline__ uint64_t sort_key(uint32_t key, int32_t idx) {
  // descending order of this composite = (value desc, index asc)
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

__global__ void __launch_bounds__(MERGE_THREADS) merge2_sample_kernel(const MergeArgs a, int P) {
  extern __shared__ __align__(16) uint32_t sm[];
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int cap = a.G * a.K;
  uint64_t* sorted = reinterpret_cast<uint64_t*>(sm);          // P entries
  float* ebuf = reinterpret_cast<float*>(sorted + P);            // K entries
  uint32_t* keys = reinterpret_cast<uint32_t*>(ebuf + a.K);
  int32_t* idx = reinterpret_cast<int32_t*>(keys + cap);
  uint32_t* hist = reinterpret_cast<uint32_t*>(idx + cap);
  uint32_t* scan = hist + HIST_BINS;

  int n = 0;
  for (int g = 0; g < a.G; ++g) {
    const int cnt = a.m1_cnt[static_cast<int64_t>(b) * a.G + g];
    const int64_t base = (static_cast<int64_t>(b) * a.G + g) * a.K;
    for (int j = threadIdx.x; j < cnt; j += MERGE_THREADS) {
      keys[n + j] = a.m1_key[base + j];
      idx[n + j] = a.m1_idx[base + j];
    }
    n += cnt;
  }
  for (int j = threadIdx.x; j < P; j += MERGE_THREADS) sorted[j] = 0ull;
  __syncthreads();
  const int want = min(a.K, n);
  Threshold th;
  if (want == n) {
    th.key = 0u;
    th.take_eq = -1;
  } else {
    th = block_select(keys, n, want, hist, scan);
  }
  block_compact(keys, n, th, scan, [&](int pos, int i, uint32_t k) { sorted[pos] = sort_key(k, idx[i]); });

  // bitonic sort, descending, over P (power of two >= want) entries
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P / 2; i += MERGE_THREADS) {
        const int lo = (i / stride) * (2 * stride) + (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t x = sorted[lo], y = sorted[hi];
        if ((x < y) == desc) {
          sorted[lo] = y;
          sorted[hi] = x;
        }
      }
      __syncthreads();
    }
  }

  for (int j = threadIdx.x; j < want; j += MERGE_THREADS) {
    const uint64_t e = sorted[j];
    a.topk_val[static_cast<int64_t>(b) * a.topk_ld + j] = key_float(static_cast<uint32_t>(e >> 32));
    a.topk_idx[static_cast<int64_t>(b) * a.topk_ld + j] =
        static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(e & 0xFFFFFFFFull));
  }

  // ---------------- sampler: warp 0
  if (a.params == nullptr || a.tokens == nullptr || threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const float* p = a.params + static_cast<int64_t>(b) * a.ncols;
  const float top_k = p[0], top_p = p[1], temp = p[2];
  const float u = a.ncols == 4 ? p[3] : 0.5f;
  const int nc = want;
  auto val_at = [&](int i) { return key_float(static_cast<uint32_t>(sorted[i] >> 32)); };
  auto idx_at = [&](int i) {
    return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(sorted[i] & 0xFFFFFFFFull));
  };
  const int kk = (top_k >= 1.0f && top_k < static_cast<float>(nc) + 1.0f) ? static_cast<int>(top_k) : nc;
  if (!(temp > 0.0f) || kk == 1) {
    if (lane == 0) a.tokens[b] = idx_at(0);
    return;
  }
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
  // S_j = excl(owner lane of j) + e_{i0} + ... + e_j, always in this order, so
  // Z, the top-p cut and the draw all see the same running sums.
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
    int found = 0x7fffffff;
    float S = excl;
    for (int i = i0; i < i1; ++i) {
      S += ebuf[i];
      if (S >= tp) {
        found = i;
        break;
      }
    }
    int best = found;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, o));
    m = best == 0x7fffffff ? kk : best + 1;
  }
  const float Cm = S_at(m - 1);
  const float target = u * Cm;
  int pick = 0x7fffffff;
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
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) pick = min(pick, __shfl_xor_sync(0xffffffffu, pick, o));
  if (pick == 0x7fffffff) pick = m - 1;
  if (lane == 0) a.tokens[b] = idx_at(pick);
}

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

cudaLaunchConfig_t pdl_config(dim3 grid, size_t smem, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(MERGE_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

int merge_groups(int nslab, int K) {
  // G near sqrt(nslab) balances the two stages; both must fit MERGE_CAP candidates.
  int best = -1, best_cost = 0x7fffffff;
  for (int G = 1; G <= nslab; ++G) {
    const int n1 = ((nslab + G - 1) / G) * K, n2 = G * K;
    if (n1 > MERGE_CAP || n2 > MERGE_CAP) continue;
    const int cost = n1 > n2 ? n1 : n2;
    if (cost < best_cost) {
      best_cost = cost;
      best = G;
    }
  }
  return best;  // -1: no split fits
}

size_t merge1_smem_bytes(int nslab, int G, int K) {
  const size_t cap = static_cast<size_t>((nslab + G - 1) / G) * K;
  return (2 * cap + HIST_BINS + 2 * MERGE_THREADS) * 4;
}

size_t merge2_smem_bytes(int G, int K) {
  const size_t cap = static_cast<size_t>(G) * K;
  return static_cast<size_t>(next_pow2(K)) * 8 + static_cast<size_t>(K) * 4 +
         (2 * cap + HIST_BINS + 2 * MERGE_THREADS) * 4;
}

cudaError_t prepare_merge(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(merge1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(merge2_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

cudaError_t launch_merge1(const MergeArgs& a, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(a.G, a.B), merge1_smem_bytes(a.nslab, a.G, a.K), stream, attr);
  return cudaLaunchKernelEx(&cfg, merge1_kernel, a);
}

cudaError_t launch_merge2_sample(const MergeArgs& a, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(a.B), merge2_smem_bytes(a.G, a.K), stream, attr);
  return cudaLaunchKernelEx(&cfg, merge2_sample_kernel, a, next_pow2(a.K));
}

}  // namespace tail
