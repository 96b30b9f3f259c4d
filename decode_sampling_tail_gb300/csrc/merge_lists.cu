// Global top-k and sampler of the tensor-core path ("GPT-OSS Tail Chunked
// Megakernel Kernel API Reference", section "Background" — stage-1 top-k per
// vocabulary chunk, then one top-k over the chunk results — and parameters `k`
// and `sampling_params`).
//
// One CTA per batch row.  Input: for every column tile the row's top TC_LIST
// composites (value desc, index asc), written by the tensor-core lm_head, and
// the row's fp32 logits.
//   1. x = a lower bound (exact in its top 16 bits) of the K-th largest key
//      among the list heads, each tile's largest element.  These are distinct
//      elements of the row, so the row's K-th largest element has key >= x.
//      (With fewer tiles than K, the K-th largest key of all list entries;
//      with fewer entries than K, x = 0.)
//   2. Every element with key >= x is gathered: from a list whose last entry
//      is below x, the list holds all of its tile's elements >= x; a list whose
//      last entry is >= x (a tile with TC_LIST or more elements at or above x)
//      is replaced by a scan of that tile's logits row.
//   3. The exact top K of the gathered set, sorted by (value desc, index asc),
//      is written out and the row's token is drawn from it.
#include "common.cuh"
#include "internal.h"
#include "sampler.cuh"
#include "select.cuh"
#include "tc_internal.h"

namespace tail {

namespace {

constexpr int MERGE_HEADS_PER_LANE = 48;  // list heads one warp holds in registers: up to 1536 tiles

int next_pow2_host(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

__global__ void __launch_bounds__(MERGE_THREADS) merge_lists_kernel(const MergeArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint32_t s_red[64];
  __shared__ uint32_t s_list[SEL_BLOCK_BUCKET_MAX];
  __shared__ uint32_t s_misc[4];
  __shared__ uint32_t s_x;
  __shared__ int s_nsat;
  pdl_wait();  // lists and logits come from the lm_head kernel

  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31;
  const int K = a.K, ntn = a.ntn;
  const int nl = ntn * TC_LIST;                           // list entries of a row
  uint32_t* lk = reinterpret_cast<uint32_t*>(smem);       // [nl]: the keys of every list entry
  uint32_t* keys = lk + nl;                               // [capc]: gathered candidates
  int32_t* idx = reinterpret_cast<int32_t*>(keys + a.capc);
  uint64_t* comp = reinterpret_cast<uint64_t*>(idx + a.capc);
  uint64_t* sorted = comp + a.sortP;
  float* ebuf = reinterpret_cast<float*>(sorted + K);
  int* cnt = reinterpret_cast<int*>(ebuf + K);  // [ntn]: list entries >= x (0 for a saturated list)
  int* off = cnt + ntn;                         // [ntn + 1]: exclusive scan of the counts
  int* sat = off + ntn + 1;                     // [ntn]: saturated lists

  // keeps the top K of keys/idx[0..n) (n > K), in place; returns K
  auto fold = [&](int n) {
    for (int j = tid; j < a.sortP; j += nt) comp[j] = 0ull;
    __syncthreads();
    block_top_composites(keys, idx, n, K, comp, s_red, s_list, s_misc);
    for (int j = tid; j < K; j += nt) {
      keys[j] = composite_key(comp[j]);
      idx[j] = composite_idx(comp[j]);
    }
    __syncthreads();
    return K;
  };

  for (int row = blockIdx.x; row < a.B; row += gridDim.x) {
    SampleParams prm = {};
    if (a.params != nullptr) prm = load_sample_params(a.params + static_cast<int64_t>(row) * a.ncols, a.ncols);
    const uint64_t* L = a.lists + static_cast<int64_t>(row) * ntn * TC_LIST;
    const float* lg = a.logits + static_cast<int64_t>(row) * a.ld;

    // ---- 1. the bound x: K-th largest key of all list entries (x = 0 when there are fewer than K:
    // every list is then saturated and all logits are scanned)
    constexpr int LPT = 4;  // lists per thread whose loads are in flight together
    for (int j0 = 0; j0 < ntn; j0 += LPT * nt) {
      uint4 w[LPT][TC_LIST / 2];
#pragma unroll
      for (int q = 0; q < LPT; ++q) {
        const int j = j0 + q * nt + tid;
        const uint4* src = reinterpret_cast<const uint4*>(L + static_cast<int64_t>(j < ntn ? j : 0) * TC_LIST);
#pragma unroll
        for (int i = 0; i < TC_LIST / 2; ++i) w[q][i] = j < ntn ? __ldcg(src + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < LPT; ++q) {
        const int j = j0 + q * nt + tid;
        if (j < ntn) {
#pragma unroll
          for (int i = 0; i < TC_LIST / 2; ++i) {
            lk[j * TC_LIST + 2 * i] = w[q][i].y;  // composite key = high word
            lk[j * TC_LIST + 2 * i + 1] = w[q][i].w;
          }
        }
      }
    }
    if (tid == 0) s_nsat = 0;
    __syncthreads();
    uint32_t x;
    if (ntn >= K && ntn <= 32 * MERGE_HEADS_PER_LANE) {
      // the list heads (each tile's largest element) are K or more distinct elements: one warp finds
      // a lower bound of their K-th largest key, exact in its top 16 bits
      if (warp == 0) {
        uint32_t hk[MERGE_HEADS_PER_LANE];
#pragma unroll
        for (int i = 0; i < MERGE_HEADS_PER_LANE; ++i) {
          const int j = i * 32 + lane;
          hk[i] = j < ntn ? lk[j * TC_LIST] : 0u;
        }
        const uint32_t b = warp_bound16_span_regs(hk, K);
        if (lane == 0) s_x = b;
      }
      __syncthreads();
      x = s_x;
    } else {
      // few tiles (or very many): the K-th largest key over every list entry, or 0 when they are fewer than K
      x = nl >= K ? block_kth_key(lk, nl, K, s_red, s_list, s_misc).key : 0u;
    }

    // ---- 2a. per list: how many entries reach x, or saturated
    for (int j = tid; j < ntn; j += nt) {
      int c = 0;
#pragma unroll
      for (int i = 0; i < TC_LIST; ++i) c += lk[j * TC_LIST + i] >= x ? 1 : 0;
      if (lk[j * TC_LIST + TC_LIST - 1] >= x) {
        cnt[j] = 0;
        sat[atomicAdd(&s_nsat, 1)] = j;
      } else {
        cnt[j] = c;
      }
    }
    __syncthreads();
    if (warp == 0) {  // exclusive scan of cnt into off
      const int per = (ntn + 31) / 32;
      const int s0 = min(ntn, lane * per), s1 = min(ntn, s0 + per);
      int loc = 0;
      for (int s = s0; s < s1; ++s) loc += cnt[s];
      int incl = loc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      int run = incl - loc;
      for (int s = s0; s < s1; ++s) {
        off[s] = run;
        run += cnt[s];
      }
      if (lane == 31) off[ntn] = incl;
    }
    __syncthreads();

    // ---- 2b. gather the list entries >= x (in capacity-sized runs of lists, folding between runs)
    int ncand = 0;
    int start = 0;
    while (start < ntn) {
      // lists [start, end) whose entries fit behind the ncand already held
      int lo = start, hi = ntn;
      while (lo < hi) {  // largest end with off[end] - off[start] + ncand <= capc
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] - off[start] + ncand <= a.capc) lo = mid; else hi = mid - 1;
      }
      const int end = lo > start ? lo : start + 1;  // one list (<= TC_LIST entries) always fits after a fold
      for (int j = start + tid; j < end; j += nt) {
        const int c = cnt[j];
        const int p = ncand + off[j] - off[start];
        const uint64_t* src = L + static_cast<int64_t>(j) * TC_LIST;
        for (int i = 0; i < c; ++i) {
          const uint64_t e = __ldcg(src + i);
          keys[p + i] = composite_key(e);
          idx[p + i] = composite_idx(e);
        }
      }
      ncand += off[end] - off[start];
      __syncthreads();
      start = end;
      if (start < ntn && ncand > K) ncand = fold(ncand);
    }

    // ---- 2c. saturated lists: scan their tiles' logits, as many tiles per pass as the buffer takes
    const int nsat = s_nsat;
    for (int s0 = 0; s0 < nsat;) {
      if (ncand + TC_N > a.capc) ncand = fold(ncand);
      const int ng = min(nsat - s0, (a.capc - ncand) / TC_N);  // >= 1 after the fold
      if (tid == 0) s_misc[3] = 0u;
      __syncthreads();
      for (int i = tid; i < ng * TC_N; i += nt) {
        const int cidx = sat[s0 + i / TC_N] * TC_N + i % TC_N;
        if (cidx < a.V) {
          const uint32_t kv = float_key(__ldcg(lg + cidx));
          if (kv >= x) {
            const int p = ncand + static_cast<int>(atomicAdd(&s_misc[3], 1u));
            keys[p] = kv;
            idx[p] = cidx;
          }
        }
      }
      __syncthreads();
      ncand += static_cast<int>(s_misc[3]);
      __syncthreads();
      s0 += ng;
    }

    // ---- 3. exact top K, sorted; tokens
    const int want = min(K, ncand);
    int nr = ncand;
    if (ncand > RANK_SORT_MAX && ncand <= 32 * MERGE_HEADS_PER_LANE) {
      // many candidates (ties in groups): keep those at or above a 16-bit-exact lower bound of the
      // K-th largest candidate key, found by one warp in registers; all K winners stay
      if (warp == 0) {
        uint32_t ck[MERGE_HEADS_PER_LANE];
#pragma unroll
        for (int i = 0; i < MERGE_HEADS_PER_LANE; ++i) {
          const int j = i * 32 + lane;
          ck[i] = j < ncand ? keys[j] : 0u;
        }
        const uint32_t b = warp_bound16_span_regs(ck, want);
        if (lane == 0) {
          s_x = b;
          s_misc[3] = 0u;
        }
      }
      __syncthreads();
      const uint32_t xc = s_x;
      for (int j = tid; j < ncand; j += nt) {
        if (keys[j] >= xc) {
          const unsigned pos = atomicAdd(&s_misc[3], 1u);
          if (pos < static_cast<unsigned>(RANK_SORT_MAX)) comp[pos] = composite(keys[j], idx[j]);
        }
      }
      __syncthreads();
      nr = static_cast<int>(s_misc[3]);
      __syncthreads();
    }
    if (nr <= RANK_SORT_MAX) {
      if (nr == ncand) {
        for (int j = tid; j < ncand; j += nt) comp[j] = composite(keys[j], idx[j]);
        __syncthreads();
      }
    } else {
      for (int j = tid; j < a.sortP; j += nt) comp[j] = 0ull;
      __syncthreads();
      block_top_composites(keys, idx, ncand, want, comp, s_red, s_list, s_misc);
      nr = want;
    }
    sort_runs(comp, sorted, nr, want);
    for (int j = tid; j < want; j += nt) {
      a.topk_val[static_cast<int64_t>(row) * a.topk_ld + j] = key_float(composite_key(sorted[j]));
      a.topk_idx[static_cast<int64_t>(row) * a.topk_ld + j] = composite_idx(sorted[j]);
    }
    if (a.params != nullptr && a.tokens != nullptr && (tid >> 5) == 0) {  // the draw: warp 0
      const int32_t tok = sample_sorted_warp(prm, sorted, want, ebuf);
      if (tid == 0) a.tokens[row] = tok;
    }
    __syncthreads();
  }
  pdl_launch_dependents();
}

}  // namespace

bool plan_merge(int K, int ntn, int dyn_max, int* capc, int* sortP, int* smem_bytes) {
  const int sp = next_pow2_host(K) > RANK_SORT_MAX ? next_pow2_host(K) : RANK_SORT_MAX;
  const int fixed = ntn * TC_LIST * 4 + sp * 8 + K * 8 + K * 4 + (3 * ntn + 1) * 4;
  // the candidate buffer holds the gathered elements and folds to the top K when full: sized for the
  // usual few hundred (ties in groups of a few) with room for K plus one saturated tile, small enough
  // for several rows' merges to share an SM
  int want = 4 * K + TC_N;
  if (want < 4096) want = 4096;  // room for ~20 rescanned tiles per pass
  want = (want + 3) & ~3;
  int cap = (dyn_max - fixed) / 8;
  cap &= ~3;
  if (cap > want) cap = want;
  if (cap < K + TC_N || cap < 2 * K) return false;
  *capc = cap;
  *sortP = sp;
  *smem_bytes = fixed + cap * 8;
  return true;
}

cudaError_t launch_merge(const MergeArgs& a, int grid, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MERGE_THREADS);
  cfg.dynamicSmemBytes = a.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, merge_lists_kernel, a);
}

cudaError_t prepare_tc(int max_smem_optin, int* merge_dyn_max) {
  cudaError_t e = prepare_tc_gemm(max_smem_optin);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, merge_lists_kernel);
  if (e != cudaSuccess) return e;
  // at most half the opt-in limit, so two rows' merges share an SM
  int dyn = (max_smem_optin - static_cast<int>(fa.sharedSizeBytes)) / 2 - 1024;
  e = cudaFuncSetAttribute(merge_lists_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  *merge_dyn_max = dyn;
  return cudaSuccess;
}

}  // namespace tail
