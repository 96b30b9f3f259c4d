// Exact top-k selection on order-preserving 32-bit keys.
//
// Order: key descending, then position ascending.  Callers lay elements out in
// ascending vocabulary order, so "position ascending" is the page's tie-break
// (index ascending) for the global top-k ("GPT-OSS Tail Chunked Megakernel
// Kernel API Reference", section "Background" and parameter `k`).
//
// A selection returns (T, take_eq): every element with key > T is selected,
// plus the first take_eq elements (in position order) whose key equals T.
//
// T, the want-th largest key, is the largest t with count(key >= t) >= want.
// It is built one bit at a time from the most significant bit; each step is a
// counting pass (compare + add, then a warp or block sum).  The first 12 bits
// run over every element; the remaining 20 run over the boundary bucket only
// (elements whose top 12 bits equal T's), which is small unless the input
// piles up on a few values, in which case the search simply continues over
// every element.  No atomics and no histograms: the cost does not depend on
// how the values are distributed.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace tail {

struct Threshold {
  uint32_t key;
  int take_eq;  // elements equal to key that are taken (lowest positions first)
};

constexpr int SEL_HI_BITS = 12;       // bits searched over every element
constexpr int SEL_BUCKET_MAX = 64;    // warp path: bucket held two keys per lane
constexpr int SEL_BLOCK_BUCKET_MAX = 256;

// Number of register keys >= c, summed over four independent chains.
template <int NPL>
__device__ __forceinline__ uint32_t count_ge(const uint32_t (&k)[NPL], uint32_t c) {
  uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
  for (int i = 0; i < NPL; i += 4) {
    a0 += k[i] >= c ? 1u : 0u;
    if (i + 1 < NPL) a1 += k[i + 1] >= c ? 1u : 0u;
    if (i + 2 < NPL) a2 += k[i + 2] >= c ? 1u : 0u;
    if (i + 3 < NPL) a3 += k[i + 3] >= c ? 1u : 0u;
  }
  return (a0 + a1) + (a2 + a3);
}

// ------------------------------------------------------------------ warp level, keys in registers
// Lane l holds the keys of positions l, l+32, l+64, ... in k[0..NPL); unused
// slots hold 0, which is below every non-NaN key.  `list` is per-warp shared
// scratch of SEL_BUCKET_MAX words.  Requires 1 <= want <= n.
template <int NPL>
__device__ __forceinline__ Threshold warp_select_regs(const uint32_t (&k)[NPL], int want, uint32_t* list) {
  const int lane = threadIdx.x & 31;
  uint32_t T = 0;
#pragma unroll 1
  for (int bit = 31; bit >= 32 - SEL_HI_BITS; --bit) {
    const uint32_t c = T | (1u << bit);
    if (__reduce_add_sync(0xffffffffu, count_ge(k, c)) >= static_cast<uint32_t>(want)) T = c;
  }
  // elements strictly above the bucket, and the bucket itself
  const uint32_t hi = T >> (32 - SEL_HI_BITS);
  uint32_t above = 0, inb = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const uint32_t h = k[i] >> (32 - SEL_HI_BITS);
    above += h > hi ? 1u : 0u;
    inb += h == hi ? 1u : 0u;
  }
  above = __reduce_add_sync(0xffffffffu, above);
  inb = __reduce_add_sync(0xffffffffu, inb);
  const int need = want - static_cast<int>(above);  // 1 <= need <= inb
  if (inb <= SEL_BUCKET_MAX) {
    // gather the bucket (order is irrelevant for the value search)
    int base = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const bool in = (k[i] >> (32 - SEL_HI_BITS)) == hi;
      const uint32_t b = __ballot_sync(0xffffffffu, in);
      if (in) list[base + __popc(b & lanemask_lt())] = k[i];
      base += __popc(b);
    }
    __syncwarp();
    const uint32_t l0 = lane < static_cast<int>(inb) ? list[lane] : 0u;
    const uint32_t l1 = lane + 32 < static_cast<int>(inb) ? list[lane + 32] : 0u;
    __syncwarp();
#pragma unroll 1
    for (int bit = 31 - SEL_HI_BITS; bit >= 0; --bit) {
      const uint32_t c = T | (1u << bit);
      const uint32_t cnt = (l0 >= c ? 1u : 0u) + (l1 >= c ? 1u : 0u);
      if (__reduce_add_sync(0xffffffffu, cnt) >= static_cast<uint32_t>(need)) T = c;
    }
  } else {
#pragma unroll 1
    for (int bit = 31 - SEL_HI_BITS; bit >= 0; --bit) {
      const uint32_t c = T | (1u << bit);
      if (__reduce_add_sync(0xffffffffu, count_ge(k, c)) >= static_cast<uint32_t>(want)) T = c;
    }
  }
  uint32_t gt = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) gt += k[i] > T ? 1u : 0u;
  gt = __reduce_add_sync(0xffffffffu, gt);
  return Threshold{T, want - static_cast<int>(gt)};
}

// A lower bound x for the want-th largest key (count(key >= x) >= want),
// exact in its top 16 bits: the search stops after 16 counting steps, so x is
// at most one 2^-7-octave step below the exact key.  Requires want <= the
// number of real (nonzero) keys.
template <int NPL>
__device__ __forceinline__ uint32_t warp_bound16_regs(const uint32_t (&k)[NPL], int want) {
  uint32_t T = 0;
#pragma unroll 1
  for (int bit = 31; bit >= 16; --bit) {
    const uint32_t c = T | (1u << bit);
    if (__reduce_add_sync(0xffffffffu, count_ge(k, c)) >= static_cast<uint32_t>(want)) T = c;
  }
  return T;
}

// warp_bound16_regs, starting below the bits all nonzero keys share: the bits
// above the highest one in which the smallest and largest nonzero key differ
// are those of the bound already, so only the bits below it (down to bit 16)
// take a counting step.  Same result, fewer steps for keys that span a
// narrow range.
template <int NPL>
__device__ __forceinline__ uint32_t warp_bound16_span_regs(const uint32_t (&k)[NPL], int want) {
  uint32_t kmx = 0u, kmn = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    kmx = max(kmx, k[i]);
    kmn = k[i] ? min(kmn, k[i]) : kmn;
  }
  kmx = __reduce_max_sync(0xffffffffu, kmx);
  kmn = __reduce_min_sync(0xffffffffu, kmn);
  uint32_t T = 0u;
  int top = 31;
  if (kmn <= kmx) {
    top = kmn == kmx ? 15 : 31 - __clz(kmn ^ kmx);
    T = top >= 31 ? 0u : (kmn & ~((2u << top) - 1u));
  }
#pragma unroll 1
  for (int bit = top; bit >= 16; --bit) {
    const uint32_t c = T | (1u << bit);
    if (__reduce_add_sync(0xffffffffu, count_ge(k, c)) >= static_cast<uint32_t>(want)) T = c;
  }
  return T;
}

// Emits, in position order, the elements a Threshold selects among the n
// register-held keys.  emit(pos, i, key): output slot pos, element position i.
template <int NPL, typename Emit>
__device__ __forceinline__ void warp_compact_regs(const uint32_t (&k)[NPL], int n, Threshold th, Emit emit) {
  const int lane = threadIdx.x & 31;
  int out = 0, eq_seen = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int pos = i * 32 + lane;
    const bool valid = pos < n;
    const bool gt = valid && k[i] > th.key;
    const bool eq = valid && k[i] == th.key;
    const uint32_t beq = __ballot_sync(0xffffffffu, eq);
    const int eq_rank = eq_seen + __popc(beq & lanemask_lt());
    const bool take = gt || (eq && eq_rank < th.take_eq);
    const uint32_t bt = __ballot_sync(0xffffffffu, take);
    if (take) emit(out + __popc(bt & lanemask_lt()), pos, k[i]);
    out += __popc(bt);
    eq_seen += __popc(beq);
  }
}

// ------------------------------------------------------------------ block level, keys in shared memory
// Every thread of the CTA takes part (any blockDim that is a multiple of 32,
// at most 1024).  `red` holds 64 words, `list` SEL_BLOCK_BUCKET_MAX words,
// `misc` 4 words, all in shared memory.
__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t* red, int parity) {
  const int nw = blockDim.x >> 5;
  v = __reduce_add_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) red[parity * 32 + (threadIdx.x >> 5)] = v;
  __syncthreads();
  uint32_t s = 0;
  for (int w = 0; w < nw; ++w) s += red[parity * 32 + w];
  return s;
}

// T = the want-th largest key of keys[0..n) (1 <= want <= n) and the number
// of keys strictly above it.
struct KthKey {
  uint32_t key;
  int above;
};

__device__ __forceinline__ KthKey block_kth_key(const uint32_t* keys, int n, int want, uint32_t* red, uint32_t* list,
                                                uint32_t* misc) {
  const int tid = threadIdx.x, nt = blockDim.x;
  int parity = 0;
  uint32_t T = 0;
#pragma unroll 1
  for (int bit = 31; bit >= 32 - SEL_HI_BITS; --bit) {
    const uint32_t c = T | (1u << bit);
    uint32_t cnt = 0;
    for (int i = tid; i < n; i += nt) cnt += keys[i] >= c ? 1u : 0u;
    if (block_sum(cnt, red, parity) >= static_cast<uint32_t>(want)) T = c;
    parity ^= 1;
  }
  const uint32_t hi = T >> (32 - SEL_HI_BITS);
  uint32_t above = 0, inb = 0;
  for (int i = tid; i < n; i += nt) {
    const uint32_t h = keys[i] >> (32 - SEL_HI_BITS);
    above += h > hi ? 1u : 0u;
    inb += h == hi ? 1u : 0u;
  }
  above = block_sum(above, red, parity);
  parity ^= 1;
  inb = block_sum(inb, red, parity);
  parity ^= 1;
  const int need = want - static_cast<int>(above);
  if (inb <= SEL_BLOCK_BUCKET_MAX) {
    if (tid == 0) misc[0] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += nt) {
      const uint32_t kv = keys[i];
      if ((kv >> (32 - SEL_HI_BITS)) == hi) list[atomicAdd(&misc[0], 1u)] = kv;
    }
    __syncthreads();
    if (tid < 32) {
      uint32_t l[SEL_BLOCK_BUCKET_MAX / 32];
#pragma unroll
      for (int j = 0; j < SEL_BLOCK_BUCKET_MAX / 32; ++j) {
        const int p = j * 32 + tid;
        l[j] = p < static_cast<int>(inb) ? list[p] : 0u;
      }
#pragma unroll 1
      for (int bit = 31 - SEL_HI_BITS; bit >= 0; --bit) {
        const uint32_t c = T | (1u << bit);
        uint32_t cnt = 0;
#pragma unroll
        for (int j = 0; j < SEL_BLOCK_BUCKET_MAX / 32; ++j) cnt += l[j] >= c ? 1u : 0u;
        if (__reduce_add_sync(0xffffffffu, cnt) >= static_cast<uint32_t>(need)) T = c;
      }
      if (tid == 0) misc[1] = T;
    }
    __syncthreads();
    T = misc[1];
  } else {
#pragma unroll 1
    for (int bit = 31 - SEL_HI_BITS; bit >= 0; --bit) {
      const uint32_t c = T | (1u << bit);
      uint32_t cnt = 0;
      for (int i = tid; i < n; i += nt) cnt += keys[i] >= c ? 1u : 0u;
      if (block_sum(cnt, red, parity) >= static_cast<uint32_t>(want)) T = c;
      parity ^= 1;
    }
  }
  uint32_t gt = 0;
  for (int i = tid; i < n; i += nt) gt += keys[i] > T ? 1u : 0u;
  gt = block_sum(gt, red, parity);
  __syncthreads();  // red is reused by the caller
  return KthKey{T, static_cast<int>(gt)};
}

// Composite sort key: descending order of it is (value desc, index asc).
__device__ __forceinline__ uint64_t composite(uint32_t key, int32_t idx) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}
__device__ __forceinline__ uint32_t composite_key(uint64_t c) { return static_cast<uint32_t>(c >> 32); }
__device__ __forceinline__ int32_t composite_idx(uint64_t c) {
  return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(c & 0xFFFFFFFFull));
}

// Keeps the top `want` of the n candidates (keys[i], idx[i]) in the order
// (key desc, vocabulary index asc), whatever order they sit in, and writes
// them as composites to out[0..want) in no particular order.  Ties at the
// boundary key are settled by a second bitwise search over the indices.
__device__ __forceinline__ void block_top_composites(const uint32_t* keys, const int32_t* idx, int n, int want,
                                                     uint64_t* out, uint32_t* red, uint32_t* list,
                                                     uint32_t* misc) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const KthKey kt = block_kth_key(keys, n, want, red, list, misc);
  const uint32_t T = kt.key;
  const int need_eq = want - kt.above;
  uint32_t neq = 0;
  for (int i = tid; i < n; i += nt) neq += keys[i] == T ? 1u : 0u;
  neq = block_sum(neq, red, 0);
  __syncthreads();
  // the need_eq-th smallest index among the keys equal to T (only when ties exceed the need)
  uint32_t cut = 0x7FFFFFFFu;
  if (static_cast<int>(neq) > need_eq) {
    uint32_t lo = 0;
    int parity = 1;
#pragma unroll 1
    for (int bit = 30; bit >= 0; --bit) {
      const uint32_t c = lo | (1u << bit);
      uint32_t cnt = 0;
      for (int i = tid; i < n; i += nt) cnt += (keys[i] == T && static_cast<uint32_t>(idx[i]) < c) ? 1u : 0u;
      if (block_sum(cnt, red, parity) < static_cast<uint32_t>(need_eq)) lo = c;
      parity ^= 1;
    }
    cut = lo;
    __syncthreads();
  }
  if (tid == 0) misc[2] = 0u;
  __syncthreads();
  for (int i = tid; i < n; i += nt) {
    const uint32_t kv = keys[i];
    if (kv > T || (kv == T && static_cast<uint32_t>(idx[i]) <= cut)) out[atomicAdd(&misc[2], 1u)] = composite(kv, idx[i]);
  }
  __syncthreads();
}

// Sorts comp[0..P) descending (P a power of two) with all threads of the CTA.
__device__ __forceinline__ void block_bitonic_desc(uint64_t* comp, int P) {
  const int nt = blockDim.x;
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P / 2; i += nt) {
        const int lo = (i / stride) * (2 * stride) + (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t x = comp[lo], y = comp[hi];
        if ((x < y) == desc) {
          comp[lo] = y;
          comp[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// sorted[0, want) = the largest `want` of the m distinct composites comp[0, m),
// in descending order, with every thread of the CTA.  comp must have room for
// m rounded up to a multiple of 32.  Each warp sorts runs of 32 in registers
// (bitonic network over the lanes); an element's position is then its place
// in its own run plus, for every other run, the number of its elements above
// it (a binary search of that sorted run).
__device__ __forceinline__ void sort_runs(uint64_t* comp, uint64_t* sorted, int m, int want) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int R = (m + 31) >> 5;
  for (int r = warp; r < R; r += nw) {
    const int i = r * 32 + lane;
    uint64_t v = i < m ? comp[i] : 0ull;  // 0 is below every composite
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
        // blocks with (lane & k) == 0 run descending; the lower lane of a pair keeps the larger
        const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
        v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
      }
    }
    comp[i] = v;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    const uint64_t v = comp[i];
    const int own = i >> 5;
    int pos = i & 31;
#pragma unroll 4
    for (int q = 0; q < R; ++q) {
      const uint64_t* run = comp + q * 32;
      int above = 0;  // elements of run q greater than v (the run is descending)
#pragma unroll
      for (int step = 16; step > 0; step >>= 1)
        if (run[above + step - 1] > v) above += step;
      if (run[above] > v) ++above;
      pos += q == own ? 0 : above;
    }
    if (pos < want) sorted[pos] = v;
  }
  __syncthreads();
}

}  // namespace tail
