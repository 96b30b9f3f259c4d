// Global top-k and sampler of the tensor-core path ("GPT-OSS Tail Chunked
// Megakernel Kernel API Reference", section "Background" — stage-1 top-k per
// vocabulary chunk, then one top-k over the chunk results — and parameters `k`
// and `sampling_params`).
//
// One CTA per batch row.  Input: for every column tile the row's top TC_LIST
// composites (value desc, index asc), written by the tensor-core lm_head, and
// the row's fp32 logits.  The row's lists reach shared memory in one bulk copy.
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
//      is written out and the row's token is drawn from it (one warp).
#include "common.cuh"
#include "internal.h"
#include "sampler.cuh"
#include "select.cuh"
#include "tc_internal.h"

namespace tail {

namespace {

constexpr int MERGE_HEADS_PER_LANE = 48;  // list heads one warp holds in registers: up to 1536 tiles
constexpr int MERGE_LISTS_PB = 1;  // lists a thread takes per gather batch
constexpr int MERGE_ONEPASS_LPT = 6;  // lists a thread takes in the one-pass gather: up to 1536 tiles
constexpr int MERGE_SCAN_PT = 8;   // logits loads in flight per thread in the saturated-tile scan

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
  __shared__ uint32_t s_nc;  // candidates gathered
  __shared__ int s_fail;
  __shared__ __align__(8) uint64_t s_bar;  // the lists' bulk copy
  pdl_wait();  // lists and logits come from the lm_head kernel

  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31;
  const int K = a.K, ntn = a.ntn;
  const int nl = ntn * TC_LIST;  // list entries of a row
  const bool heads_bound = ntn >= K && ntn <= 32 * MERGE_HEADS_PER_LANE;
  uint64_t* ls = reinterpret_cast<uint64_t*>(smem);     // [nl]: the row's lists, copied in whole
  uint32_t* lk = reinterpret_cast<uint32_t*>(ls + nl);  // [nl] every entry's key, only for few tiles
  uint32_t* keys = lk + (heads_bound ? 0 : nl);         // [capc]: gathered candidates
  int32_t* idx = reinterpret_cast<int32_t*>(keys + a.capc);
  uint64_t* comp = reinterpret_cast<uint64_t*>(idx + a.capc);
  uint64_t* sorted = comp + a.sortP;
  float* ebuf = reinterpret_cast<float*>(sorted + K);
  int* sat = reinterpret_cast<int*>(ebuf + K);  // [ntn]: saturated lists
  const uint32_t bar = smem_u32(&s_bar);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // keeps the top K of keys/idx[0..n) (n > K), in place; returns K
  auto fold = [&](int n) {
    for (int j = tid; j < a.sortP; j += nt) comp[j] = 0ull;
    __syncthreads();
    block_top_composites(keys, idx, n, K, comp, s_red, s_list, s_misc);
    for (int j = tid; j < K; j += nt) {
      keys[j] = composite_key(comp[j]);
      idx[j] = composite_idx(comp[j]);
    }
    if (tid == 0) s_nc = static_cast<uint32_t>(K);
    __syncthreads();
    return K;
  };

  int parity = 0;
  for (int row = blockIdx.x; row < a.B; row += gridDim.x, parity ^= 1) {
    SampleParams prm = {};
    if (a.params != nullptr) prm = load_sample_params(a.params + static_cast<int64_t>(row) * a.ncols, a.ncols);
    const uint64_t* L = a.lists + static_cast<int64_t>(row) * ntn * TC_LIST;
    const float* lg = a.logits + static_cast<int64_t>(row) * a.ld;

    // ---- 1. the row's lists into shared memory: one bulk copy
    if (tid == 0) {
      s_nsat = 0;
      s_nc = 0u;
      s_fail = 0;
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nl) * 8u);
      bulk_g2s(smem_u32(ls), L, static_cast<uint32_t>(nl) * 8u, bar, policy_evict_first());
    }
    if (!mbar_wait_bounded(bar, static_cast<uint32_t>(parity), a.timeout_ns)) {
      raise_error(a.err, DEV_TIMEOUT_FULL);
      s_fail = 1;
    }
    __syncthreads();
    if (s_fail) break;  // uniform (the error flag is raised)

    // ---- 2. the bound x: K-th largest key of the list heads (distinct elements of the row), or of every
    // list entry when the tiles are fewer than K, or 0 when the entries are fewer than K (every list is
    // then saturated and all logits are scanned)
    uint32_t x;
    if (heads_bound) {
      // the heads into a compact array first (read 64 bytes apart they would share banks), in the
      // candidate buffer, which the gather only fills afterwards
      for (int j = tid; j < ntn; j += nt) keys[j] = composite_key(ls[j * TC_LIST]);
      __syncthreads();
      if (warp == 0) {
        uint32_t hk[MERGE_HEADS_PER_LANE];
#pragma unroll
        for (int i = 0; i < MERGE_HEADS_PER_LANE; ++i) {
          const int j = i * 32 + lane;
          hk[i] = j < ntn ? keys[j] : 0u;
        }
        const uint32_t b = warp_bound16_span_regs(hk, K);
        if (lane == 0) s_x = b;
      }
      __syncthreads();
      x = s_x;
    } else {
      for (int e = tid; e < nl; e += nt) lk[e] = composite_key(ls[e]);
      __syncthreads();
      x = nl >= K ? block_kth_key(lk, nl, K, s_red, s_list, s_misc).key : 0u;
    }

    // ---- 3. a list whose last entry is below x holds all of its tile's elements >= x (its first c
    // entries); a list whose last entry is >= x is saturated and its tile's logits are scanned below.
    // Batches of MERGE_LISTS_PB lists a thread, one reservation per warp; the buffer is folded to the
    // top K before a batch that might not fit.  A thread reads list j's entries starting at j mod 8
    // (the lists are 64 bytes apart: in entry order the lanes would share banks).
    int ncand = 0;
    // One pass when the candidates fit the buffer (the usual case: about K lists reach x, with one or
    // two entries each): every thread counts the candidates of its lists -- none below a head under x --
    // and one block-wide scan places them.  Otherwise (a buffer's worth of entries at or above x) the
    // batched gather below folds the buffer to the top K between batches.
    int cnt[MERGE_ONEPASS_LPT];
    int tot = 0;
#pragma unroll
    for (int r = 0; r < MERGE_ONEPASS_LPT; ++r) {
      const int j = tid + r * nt;
      cnt[r] = 0;
      if (j < ntn && composite_key(ls[j * TC_LIST]) >= x) {
        const uint64_t* lj = ls + static_cast<int64_t>(j) * TC_LIST;
        if (composite_key(lj[TC_LIST - 1]) >= x) {
          sat[atomicAdd(&s_nsat, 1)] = j;
        } else {
          int c = 1;
          while (composite_key(lj[c]) >= x) ++c;  // entries are in descending order; the last is below x
          cnt[r] = c;
        }
      }
      tot += cnt[r];
    }
    const bool onepass = ntn <= nt * MERGE_ONEPASS_LPT;
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_red[warp] = static_cast<uint32_t>(incl);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < nt / 32; ++w) {
      const int v = static_cast<int>(s_red[w]);
      before += w < warp ? v : 0;
      total += v;
    }
    if (onepass && total <= a.capc) {
      int pos = before + incl - tot;
#pragma unroll
      for (int r = 0; r < MERGE_ONEPASS_LPT; ++r) {
        const uint64_t* lj = ls + static_cast<int64_t>(tid + r * nt) * TC_LIST;
        for (int e = 0; e < cnt[r]; ++e, ++pos) {
          keys[pos] = composite_key(lj[e]);
          idx[pos] = composite_idx(lj[e]);
        }
      }
      if (tid == 0) s_nc = static_cast<uint32_t>(total);
    }
    __syncthreads();  // s_red and the saturated lists are complete; so are the candidates
    if (onepass && total <= a.capc) {
      ncand = total;
    } else {
      if (tid == 0) s_nsat = 0;  // the batched gather marks the saturated lists again
      __syncthreads();
    }
    for (int j0 = (onepass && total <= a.capc) ? ntn : 0; j0 < ntn; j0 += nt * MERGE_LISTS_PB) {
      if (ncand + nt * MERGE_LISTS_PB * TC_LIST > a.capc) ncand = fold(ncand);
      uint64_t le[MERGE_LISTS_PB][TC_LIST];
      int c[MERGE_LISTS_PB];
      int tot = 0;
#pragma unroll
      for (int r = 0; r < MERGE_LISTS_PB; ++r) {
        const int j = j0 + r * nt + tid;
        const uint64_t* lj = ls + static_cast<int64_t>(j < ntn ? j : 0) * TC_LIST;
#pragma unroll
        for (int e = 0; e < TC_LIST; ++e) {
          const int er = (e + j) & (TC_LIST - 1);
          const uint64_t v = lj[er];
#pragma unroll
          for (int t = 0; t < TC_LIST; ++t)  // le[r][er] = v, with er only known at run time
            if (t == er) le[r][t] = v;
        }
        c[r] = 0;
        if (j < ntn) {
          if (composite_key(le[r][TC_LIST - 1]) >= x) {
            sat[atomicAdd(&s_nsat, 1)] = j;
          } else {
#pragma unroll
            for (int e = 0; e < TC_LIST; ++e) c[r] += composite_key(le[r][e]) >= x ? 1 : 0;
          }
        }
        tot += c[r];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      uint32_t base = 0u;
      if (lane == 31 && incl > 0) base = atomicAdd(&s_nc, static_cast<uint32_t>(incl));
      int pos = static_cast<int>(__shfl_sync(0xffffffffu, base, 31)) + incl - tot;
#pragma unroll
      for (int r = 0; r < MERGE_LISTS_PB; ++r) {
#pragma unroll
        for (int e = 0; e < TC_LIST; ++e) {
          if (e < c[r]) {
            keys[pos] = composite_key(le[r][e]);
            idx[pos] = composite_idx(le[r][e]);
            ++pos;
          }
        }
      }
      __syncthreads();
      ncand = static_cast<int>(s_nc);
    }

    // ---- 4. saturated lists: scan their tiles' logits, as many tiles per pass as the buffer takes,
    // MERGE_SCAN_PT loads in flight per thread
    const int nsat = s_nsat;
    for (int s0 = 0; s0 < nsat;) {
      const int tn = a.tile_n;
      if (ncand + tn > a.capc) ncand = fold(ncand);
      const int ng = min(nsat - s0, (a.capc - ncand) / tn);  // >= 1 after the fold
      const int ne = ng * tn;
      for (int i0 = 0; i0 < ne; i0 += nt * MERGE_SCAN_PT) {  // warp-uniform trip counts
        uint32_t kv[MERGE_SCAN_PT];
        int ci[MERGE_SCAN_PT];
#pragma unroll
        for (int u = 0; u < MERGE_SCAN_PT; ++u) {
          const int i = i0 + u * nt + tid;
          ci[u] = i < ne ? sat[s0 + i / tn] * tn + i % tn : a.V;
          kv[u] = ci[u] < a.V ? float_key(__ldcg(lg + ci[u])) : 0u;
        }
#pragma unroll
        for (int u = 0; u < MERGE_SCAN_PT; ++u) {
          const bool take = ci[u] < a.V && kv[u] >= x;
          const uint32_t bt = __ballot_sync(0xffffffffu, take);
          if (bt != 0u) {
            uint32_t b0 = 0u;
            if (lane == 0) b0 = atomicAdd(&s_nc, static_cast<uint32_t>(__popc(bt)));
            b0 = __shfl_sync(0xffffffffu, b0, 0);
            if (take) {
              const int p = static_cast<int>(b0) + __popc(bt & lanemask_lt());
              keys[p] = kv[u];
              idx[p] = ci[u];
            }
          }
        }
      }
      __syncthreads();
      ncand = static_cast<int>(s_nc);
      s0 += ng;
    }

    // ---- 5. exact top K, sorted; tokens
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
  const int nl = ntn * TC_LIST;
  const bool heads_bound = ntn >= K && ntn <= 32 * MERGE_HEADS_PER_LANE;
  const int sp = next_pow2_host(K) > RANK_SORT_MAX ? next_pow2_host(K) : RANK_SORT_MAX;
  const int fixed = nl * 8 + (heads_bound ? 0 : nl * 4) + sp * 8 + K * 8 + K * 4 + ntn * 4;
  // the candidate buffer: the gathered elements, folded to the top K before a gather batch or a
  // saturated tile might not fit; sized for the usual few hundred with room for ~20 rescanned tiles
  int want = 4096;
  if (want < K + MERGE_THREADS * MERGE_LISTS_PB * TC_LIST) want = K + MERGE_THREADS * MERGE_LISTS_PB * TC_LIST;
  if (want < 2 * K) want = 2 * K;
  want = (want + 3) & ~3;
  if (fixed + want * 8 > dyn_max) return false;
  *capc = want;
  *sortP = sp;
  *smem_bytes = fixed + want * 8;
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
  // the whole opt-in limit; at the GPT-OSS shape (1048 tiles, k = 256) a row takes ~111 KB, so two
  // rows' merges still share an SM
  int dyn = max_smem_optin - static_cast<int>(fa.sharedSizeBytes);
  e = cudaFuncSetAttribute(merge_lists_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  *merge_dyn_max = dyn;
  return cudaSuccess;
}

}  // namespace tail
