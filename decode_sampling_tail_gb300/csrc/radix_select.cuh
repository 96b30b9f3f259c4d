// Block-wide radix selection of the want-th largest 32-bit key (with
// multiplicity) from keys in shared memory.
//
// The bits every key shares are found first (one min/max reduction); the
// remaining bits are resolved 8 at a time, each digit by a 256-bin histogram
// of the keys that match the digits fixed so far.  Three to four passes for
// keys that span a few binades, instead of one counting pass per bit.
#pragma once

#include "common.cuh"

namespace tail {

// keys[0..n), 1 <= want <= n.  Every thread of the CTA takes part; hist is 256
// words, red 64 words and misc 4 words of shared scratch.
__device__ __forceinline__ uint32_t block_kth_radix(const uint32_t* keys, int n, int want, uint32_t* hist,
                                                    uint32_t* red, uint32_t* misc) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  for (int i = tid; i < n; i += nt) {
    const uint32_t k = keys[i];
    mn = min(mn, k);
    mx = max(mx, k);
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    red[warp] = mn;
    red[32 + warp] = mx;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t a = red[0], b = red[32];
    for (int w = 1; w < nw; ++w) {
      a = min(a, red[w]);
      b = max(b, red[32 + w]);
    }
    misc[0] = a;
    misc[1] = b;
  }
  __syncthreads();
  mn = misc[0];
  mx = misc[1];
  __syncthreads();  // misc is rewritten below
  if (mn == mx) return mn;
  const int top = 31 - __clz(mn ^ mx);                 // highest bit in which the keys differ
  const uint32_t low = top == 31 ? 0xFFFFFFFFu : ((2u << top) - 1u);
  uint32_t pmask = ~low;                               // bits fixed so far
  uint32_t prefix = mn & pmask;
  uint32_t need = static_cast<uint32_t>(want);         // rank wanted among the keys matching prefix
  int shift = top + 1;
  while (shift > 0) {
    const int w = shift < 8 ? shift : 8;
    shift -= w;
    const uint32_t dmask = (1u << w) - 1u;
    for (int i = tid; i < 256; i += nt) hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += nt) {
      const uint32_t k = keys[i];
      if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & dmask], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins [8 (31 - l), +8): lane 0 the highest digits
      const int b0 = 8 * (31 - lane);
      uint32_t h[8], loc = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        h[j] = hist[b0 + j];
        loc += h[j];
      }
      uint32_t incl = loc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      uint32_t above = incl - loc;  // keys in higher digits than this lane's bins
      if (above < need && need <= incl) {
#pragma unroll
        for (int j = 7; j >= 0; --j) {
          if (above < need && need <= above + h[j]) {
            misc[2] = static_cast<uint32_t>(b0 + j);
            misc[3] = need - above;
          }
          above += h[j];
        }
      }
    }
    __syncthreads();
    prefix |= misc[2] << shift;
    need = misc[3];
    pmask |= dmask << shift;
    __syncthreads();  // hist and misc are reused by the next pass
  }
  return prefix;
}

}  // namespace tail
