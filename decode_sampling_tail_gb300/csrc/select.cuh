// Exact top-k selection by radix select on order-preserving 32-bit keys.
//
// Order: key descending, then position ascending.  Callers lay elements out in
// ascending vocabulary order, so "position ascending" is the page's tie-break
// (index ascending) for the global top-k ("GPT-OSS Tail Chunked Megakernel
// Kernel API Reference", section "Background" and parameter `k`).
//
// A selection returns (T, take_eq): every element with key > T is selected,
// plus the first take_eq elements (in position order) whose key equals T.
// The digits are 11, 11 and 10 bits wide, most significant first; a pass that
// finds its boundary bin exactly full stops early.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace tail {

struct Threshold {
  uint32_t key;
  int take_eq;   // elements equal to key that are taken (lowest positions first); -1: take all >= key
};

__device__ __forceinline__ int digit_shift(int pass) { return pass == 0 ? 21 : (pass == 1 ? 10 : 0); }
__device__ __forceinline__ int digit_bins(int pass) { return pass == 2 ? 1024 : 2048; }
__device__ __forceinline__ uint32_t digit_prefix_mask(int pass) {
  return pass == 0 ? 0u : (pass == 1 ? 0xFFE00000u : 0xFFFFFC00u);
}

// ------------------------------------------------------------------ warp-level
// One warp selects the top `want` of n keys given by get(i).  `hist` is this
// warp's private shared-memory histogram of HIST_BINS words.  Requires
// 1 <= want <= n.
template <typename GetKey>
__device__ Threshold warp_select(GetKey get, int n, int want, uint32_t* hist) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0;
  int need = want;
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = digit_shift(pass), nb = digit_bins(pass);
    const uint32_t pmask = digit_prefix_mask(pass);
    for (int i = lane; i < nb; i += 32) hist[i] = 0u;
    __syncwarp();
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      uint32_t d = 0xFFFFFFFFu;
      if (i < n) {
        const uint32_t k = get(i);
        if ((k & pmask) == prefix) d = (k >> shift) & static_cast<uint32_t>(nb - 1);
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (d != 0xFFFFFFFFu && lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
    }
    __syncwarp();
    // Lane l owns bins [nb - (l+1)*bpl, nb - l*bpl): lane 0 holds the largest digits.
    const int bpl = nb / 32;
    const int top = nb - lane * bpl;
    uint32_t s = 0;
    for (int j = 0; j < bpl; ++j) s += hist[top - 1 - j];
    uint32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const uint32_t excl = incl - s;
    const uint32_t hit = __ballot_sync(0xffffffffu, excl < static_cast<uint32_t>(need) &&
                                                        static_cast<uint32_t>(need) <= incl);
    const int L = __ffs(hit) - 1;
    // Lane L walks its bins from the top to find the boundary digit.
    uint32_t dstar = 0, gt = 0, cnt = 0;
    if (lane == L) {
      uint32_t c = excl;
      for (int j = 0; j < bpl; ++j) {
        const int bin = top - 1 - j;
        const uint32_t hb = hist[bin];
        if (c + hb >= static_cast<uint32_t>(need)) {
          dstar = static_cast<uint32_t>(bin);
          gt = c;
          cnt = hb;
          break;
        }
        c += hb;
      }
    }
    dstar = __shfl_sync(0xffffffffu, dstar, L);
    gt = __shfl_sync(0xffffffffu, gt, L);
    cnt = __shfl_sync(0xffffffffu, cnt, L);
    __syncwarp();
    need -= static_cast<int>(gt);
    prefix |= dstar << shift;
    if (cnt == static_cast<uint32_t>(need) && pass < 2) {
      // the whole boundary bin is taken: select every key whose high bits >= prefix
      return Threshold{prefix, -1};
    }
  }
  return Threshold{prefix, need};
}

// Emits, in position order, the elements a Threshold selects.  emit(pos, i, key)
// receives the output slot pos (0-based) and the element position i.
template <typename GetKey, typename Emit>
__device__ int warp_compact(GetKey get, int n, Threshold th, Emit emit) {
  const int lane = threadIdx.x & 31;
  int out = 0, eq_seen = 0;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    uint32_t k = 0;
    bool gt = false, eq = false;
    if (i < n) {
      k = get(i);
      if (th.take_eq < 0) {
        gt = k >= th.key;
      } else {
        gt = k > th.key;
        eq = k == th.key;
      }
    }
    const uint32_t beq = __ballot_sync(0xffffffffu, eq);
    const int eq_rank = eq_seen + __popc(beq & lanemask_lt());
    const bool take = gt || (eq && eq_rank < th.take_eq);
    const uint32_t bt = __ballot_sync(0xffffffffu, take);
    if (take) emit(out + __popc(bt & lanemask_lt()), i, k);
    out += __popc(bt);
    eq_seen += __popc(beq);
  }
  return out;
}

// ------------------------------------------------------------------ block-level
// All MERGE_THREADS threads select the top `want` of n keys held in shared
// memory (keys[0..n)).  `hist` holds HIST_BINS words; `scan` MERGE_THREADS words.
__device__ __forceinline__ Threshold block_select(const uint32_t* keys, int n, int want, uint32_t* hist,
                                  uint32_t* scan) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = MERGE_THREADS / 32;
  __shared__ uint32_t s_dstar, s_gt, s_cnt;
  uint32_t prefix = 0;
  int need = want;
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = digit_shift(pass), nb = digit_bins(pass);
    const uint32_t pmask = digit_prefix_mask(pass);
    for (int i = tid; i < nb; i += MERGE_THREADS) hist[i] = 0u;
    __syncthreads();
    for (int base = 0; base < n; base += MERGE_THREADS) {
      const int i = base + tid;
      uint32_t d = 0xFFFFFFFFu;
      if (i < n) {
        const uint32_t k = keys[i];
        if ((k & pmask) == prefix) d = (k >> shift) & static_cast<uint32_t>(nb - 1);
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (d != 0xFFFFFFFFu && lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
    }
    __syncthreads();
    // thread t owns bins [nb - (t+1)*bpt, nb - t*bpt), thread 0 the largest digits
    const int bpt = nb / MERGE_THREADS;
    const int top = nb - tid * bpt;
    uint32_t s = 0;
    for (int j = 0; j < bpt; ++j) s += hist[top - 1 - j];
    uint32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    uint32_t woff = 0;
    for (int w = 0; w < warp; ++w) woff += scan[w];
    incl += woff;
    const uint32_t excl = incl - s;
    if (excl < static_cast<uint32_t>(need) && static_cast<uint32_t>(need) <= incl) {
      uint32_t c = excl;
      for (int j = 0; j < bpt; ++j) {
        const int bin = top - 1 - j;
        const uint32_t hb = hist[bin];
        if (c + hb >= static_cast<uint32_t>(need)) {
          s_dstar = static_cast<uint32_t>(bin);
          s_gt = c;
          s_cnt = hb;
          break;
        }
        c += hb;
      }
    }
    __syncthreads();
    const uint32_t dstar = s_dstar, gt = s_gt, cnt = s_cnt;
    __syncthreads();  // s_* and scan are rewritten by the next pass
    need -= static_cast<int>(gt);
    prefix |= dstar << shift;
    if (cnt == static_cast<uint32_t>(need) && pass < 2) return Threshold{prefix, -1};
  }
  (void)NW;
  return Threshold{prefix, need};
}

// Block compaction in position order.  Thread t handles the contiguous chunk
// [t*E, (t+1)*E) with E = ceil(n / MERGE_THREADS).  `scan` holds 2*MERGE_THREADS words.
template <typename Emit>
__device__ int block_compact(const uint32_t* keys, int n, Threshold th, uint32_t* scan, Emit emit) {
  const int tid = threadIdx.x;
  const int E = (n + MERGE_THREADS - 1) / MERGE_THREADS;
  const int i0 = min(n, tid * E), i1 = min(n, i0 + E);
  uint32_t ngt = 0, neq = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t k = keys[i];
    if (th.take_eq < 0) {
      ngt += k >= th.key;
    } else {
      ngt += k > th.key;
      neq += k == th.key;
    }
  }
  scan[tid] = ngt;
  scan[MERGE_THREADS + tid] = neq;
  __syncthreads();
  // exclusive prefix (serial over warps' totals is fine at 256 threads)
  uint32_t gt_before = 0, eq_before = 0, gt_total = 0, eq_total = 0;
  {
    // every thread sums the entries below it; 256 adds, done once per merge
    for (int t = 0; t < MERGE_THREADS; ++t) {
      const uint32_t g = scan[t], e = scan[MERGE_THREADS + t];
      if (t < tid) {
        gt_before += g;
        eq_before += e;
      }
      gt_total += g;
      eq_total += e;
    }
  }
  const uint32_t take_eq = th.take_eq < 0 ? 0u : static_cast<uint32_t>(th.take_eq);
  uint32_t pos = gt_before + min(eq_before, take_eq);
  uint32_t eq_rank = eq_before;
  for (int i = i0; i < i1; ++i) {
    const uint32_t k = keys[i];
    bool take;
    if (th.take_eq < 0) {
      take = k >= th.key;
    } else if (k > th.key) {
      take = true;
    } else if (k == th.key) {
      take = eq_rank < take_eq;
      ++eq_rank;
    } else {
      take = false;
    }
    if (take) emit(static_cast<int>(pos++), i, k);
  }
  __syncthreads();
  return static_cast<int>(gt_total + min(eq_total, take_eq));
}

}  // namespace tail
