// One-launch decode sampling tail for small problems, the latency path
// ("GPT-OSS Tail Chunked Megakernel Kernel API Reference": final RMSNorm,
// lm_head, global top-k with ties to the lower index and the sampler; section
// "Background" and parameters `deferred_rms`, `k` and `sampling_params`).
//
// CTA c of ceil(V / slab_cols) owns the vocabulary columns [c * slab_cols, ...):
//   1. it loads its first weight chunks and gamma before the dependency wait
//      (they are inputs of the step, not products of the previous kernel),
//      then every row's hidden state into shared memory;
//   2. rstd_b = 1 / sqrt(sum of x^2 over the row's active lanes / H_u + eps),
//      and the activations v = x * gamma (deferred form: rstd scales the sums)
//      or (x * rstd) * gamma (legacy form), kept in fp32;
//   3. the slab's logits: thread (g, ch) accumulates 8 columns of every row
//      over the k-rows g, g + G, ... with fp32 FMAs; the G partial sums of a
//      column are added by a fixed tree (T threads each add every T-th partial
//      in g order, then a butterfly over the T lanes; T and G depend on the
//      slab width only, not on the batch), and the logits go to
//      global memory (the caller's buffer or the handle's scratch); then the
//      CTA adds one to each row's arrival word (release);
//      Each slab also publishes, per row, the largest order key of its columns;
//   4. CTA b owns row b (and b + nslab, ... when the vocabulary is narrower than
//      the batch): it waits (bounded) until every slab has arrived.  A lower
//      bound x of the row's K-th largest key: with at least K slabs, the K-th
//      largest of the slabs' maxima (distinct elements of the row) cut to its
//      top 16 bits, found by one warp; else the largest key with its low 16
//      bits zero that at least K of the row's keys reach, found one bit at a
//      time over the whole row.  Every element of the top K has a key >= x, and
//      the keys >= x are few unless many share the bound's top 16 bits: they are
//      gathered as the logits are read and ranked in (value desc, index asc)
//      order (sorted runs of 32).  When more than the gather buffer holds reach
//      the bound, the search over the whole row, and past that the exact
//      selection over the whole row, take over.  The sorted top K is written
//      and the token drawn with the per-row sampler every path shares.
// CUDA-core arithmetic throughout: at these sizes a step is bound by latency,
// not by bytes or FLOPs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "sampler.cuh"
#include "select.cuh"
#include "small_internal.h"

namespace tail {

namespace {

__device__ __forceinline__ float small_load_x(const void* p, int dtype, int64_t i) {
  if (dtype == 0) return static_cast<const float*>(p)[i];
  if (dtype == 1) return __half2float(static_cast<const __half*>(p)[i]);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

// acc[b][j] += w_j * v[b][h] for the 8 bf16 columns of wv, every row b < B
__device__ __forceinline__ void small_fma_chunk(float (&acc)[SMALL_MAX_ROWS][8], uint4 wv, const float* act, int H,
                                                int h, int B) {
  const uint32_t u[4] = {wv.x, wv.y, wv.z, wv.w};
  float w[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    w[2 * q] = __uint_as_float(u[q] << 16);
    w[2 * q + 1] = __uint_as_float(u[q] & 0xffff0000u);
  }
#pragma unroll
  for (int b = 0; b < SMALL_MAX_ROWS; ++b) {
    if (b < B) {
      const float v = act[b * H + h];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[b][j] = fmaf(w[j], v, acc[b][j]);
    }
  }
}

// Sum of v over the CTA, returned to every thread: a warp sum, one shared word a warp, a warp sum of
// those.  Consecutive calls alternate `parity`, so a word is not rewritten while it may still be read.
__device__ __forceinline__ uint32_t small_block_sum(uint32_t v, uint32_t* red, int parity) {
  const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  v = __reduce_add_sync(0xffffffffu, v);
  if (lane == 0) red[parity * 32 + (threadIdx.x >> 5)] = v;
  __syncthreads();
  return __reduce_add_sync(0xffffffffu, lane < nw ? red[parity * 32 + lane] : 0u);
}

__global__ void __launch_bounds__(SMALL_THREADS, 1) small_tail_kernel(const SmallArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint32_t s_red[64];
  __shared__ uint32_t s_list[SEL_BLOCK_BUCKET_MAX];
  __shared__ uint32_t s_misc[4];
  __shared__ float s_rs[SMALL_MAX_ROWS];
  __shared__ uint32_t s_max[SMALL_MAX_ROWS];  // the slab's largest key of each row
  __shared__ int s_ok;
  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.B, H = a.H, V = a.V, SW = a.slab_cols;
  const int active_end = a.zero_pad ? H : a.Hu;
  const int c0 = blockIdx.x * SW;
  const int ncols = min(SW, V - c0);  // a multiple of 8: V and SW are
  const int nch_full = SW >> 3, nch = ncols >> 3;
  const int G = nt / nch_full;  // k-row groups
  const int g = tid / nch_full, ch = tid - g * nch_full;
  const bool active = g < G && ch < nch;
  const uint16_t* wcol = a.w + c0 + 8 * ch;

  // ---- 1. the first weight chunks of this thread (k-rows g, g + G, ...) and gamma, then the hidden rows
  float* act = reinterpret_cast<float*>(smem);  // [B][H]
  float* gam = act + B * H;                     // [H]
  float* part = gam + H;                        // [G][B][SW]
  for (int h = tid; h < H; h += nt) gam[h] = h < active_end ? a.gamma[h] : 0.f;
  if (tid < SMALL_MAX_ROWS) s_max[tid] = 0u;
  uint4 pf[SMALL_PREFETCH];
#pragma unroll
  for (int p = 0; p < SMALL_PREFETCH; ++p) {
    const int h = g + p * G;
    pf[p] = active && h < H ? __ldg(reinterpret_cast<const uint4*>(wcol + static_cast<int64_t>(h) * V))
                            : make_uint4(0u, 0u, 0u, 0u);
  }
  pdl_wait();  // the hidden state, and the previous step's use of the arrival words and outputs
  for (int i = tid; i < B * H; i += nt) {
    const int b = i / H, h = i - b * H;
    act[i] = h < active_end ? small_load_x(a.hidden, a.dtype, static_cast<int64_t>(b) * H + h) : 0.f;
  }
  __syncthreads();

  // ---- 2. rstd per row (warp b: lane-strided squares, then a butterfly), the activations in place
  if (warp < B) {
    float ss = 0.f;
    for (int h = lane; h < active_end; h += 32) {
      const float x = act[warp * H + h];
      ss = fmaf(x, x, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s_rs[warp] = 1.0f / sqrtf(ss / static_cast<float>(a.Hu) + a.eps);
  }
  __syncthreads();
  for (int i = tid; i < B * H; i += nt) {
    const int b = i / H, h = i - b * H;
    if (h < active_end) act[i] = a.deferred ? act[i] * gam[h] : (act[i] * s_rs[b]) * gam[h];
  }
  __syncthreads();

  // ---- 3. the slab's logits
  float acc[SMALL_MAX_ROWS][8];
#pragma unroll
  for (int b = 0; b < SMALL_MAX_ROWS; ++b)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[b][j] = 0.f;
  if (active) {
#pragma unroll
    for (int p = 0; p < SMALL_PREFETCH; ++p) {
      const int h = g + p * G;
      if (h < H) small_fma_chunk(acc, pf[p], act, H, h, B);
    }
#pragma unroll 4
    for (int h = g + SMALL_PREFETCH * G; h < H; h += G)
      small_fma_chunk(acc, __ldg(reinterpret_cast<const uint4*>(wcol + static_cast<int64_t>(h) * V)), act, H, h, B);
#pragma unroll
    for (int b = 0; b < SMALL_MAX_ROWS; ++b) {
      if (b < B) {
        float* dst = part + (g * B + b) * SW + 8 * ch;
        *reinterpret_cast<float4*>(dst) = make_float4(acc[b][0], acc[b][1], acc[b][2], acc[b][3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[b][4], acc[b][5], acc[b][6], acc[b][7]);
      }
    }
  }
  __syncthreads();
  {
    const int nout = B * ncols;
    // T = 2^lg2 threads an output, up to a warp, while the CTA covers the outputs of the largest batch
    // in one pass; T (hence every logit's order of additions) depends on the slab width only, so a
    // row's logits do not depend on the batch it runs in
    int lg2 = 0;
    while (lg2 < 5 && ((SMALL_MAX_ROWS * SW) << (lg2 + 1)) <= nt) ++lg2;
    const int T = 1 << lg2;
    for (int base = 0; base < (nout << lg2); base += nt) {  // every lane of a warp takes the same trips
      const int i = base + tid, o = i >> lg2, r = i & (T - 1);
      float s = 0.f;
      if (o < nout) {
        const int b = o / ncols, col = o - b * ncols;
#pragma unroll 8
        for (int q = r; q < G; q += T) s += part[(q * B + b) * SW + col];
      }
      for (int off = T >> 1; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (o < nout && r == 0) {
        const int b = o / ncols;
        const float logit = a.deferred ? s * s_rs[b] : s;
        a.logits[static_cast<int64_t>(b) * V + c0 + (o - b * ncols)] = logit;
        atomicMax(&s_max[b], float_key(logit));
      }
    }
  }
  __syncthreads();  // every thread's logits are stored: the release below orders them (cumulative)
  if (tid < B) {
    a.smax[tid * gridDim.x + blockIdx.x] = s_max[tid];
    __threadfence();
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(a.sync + tid), "l"(1ull) : "memory");
  }

  // ---- 4. the rows this CTA owns: exact top K of the row's logits, sorted, and the draw
  const int K = a.K;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);  // [V] (over the activations, no longer read)
  int32_t* idx = reinterpret_cast<int32_t*>(keys + V);  // [V], the whole-row selection only
  uint64_t* comp = reinterpret_cast<uint64_t*>(idx + V);  // [cap]: the gathered composites
  uint64_t* sorted = comp + a.cap;                         // [K]
  float* ebuf = reinterpret_cast<float*>(sorted + K);     // [K]
  for (int row = blockIdx.x; row < B; row += gridDim.x) {
    SampleParams prm = {};
    if (a.params != nullptr) prm = load_sample_params(a.params + static_cast<int64_t>(row) * a.ncols, a.ncols);
    if (tid == 0) {  // wait (bounded) until every slab has stored this row's logits
      unsigned long long v = 0;
      int ok = 1;
      const uint64_t t0 = global_timer_ns();
      while (true) {
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.sync + row) : "memory");
        if (v >= static_cast<unsigned long long>(gridDim.x)) break;
        if (global_timer_ns() - t0 > a.timeout_ns) {
          raise_error(a.err, DEV_TIMEOUT_BARRIER);
          ok = 0;
          break;
        }
      }
      if (ok) a.sync[row] = 0ull;  // every slab has arrived: ready for the next launch
      s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) break;  // uniform (the error flag is raised)
    const float* lg = a.logits + static_cast<int64_t>(row) * V;
    const int nslab = gridDim.x;
    int m = a.cap + 1;  // the gathered count; above cap: no gather yet, or one that overflowed
    if (nslab >= K) {  // the bound from the slabs' maxima, then one pass over the logits
      // warp 0 requests the maxima first; every thread then requests its logits (positions tid, tid + nt,
      // ...) and holds them as they arrive, while warp 0 forms the bound
      uint32_t mk[SMALL_MAX_SLABS / 32];
      if (warp == 0) {
#pragma unroll
        for (int i = 0; i < SMALL_MAX_SLABS / 32; ++i) {
          const int sl = i * 32 + lane;
          mk[i] = sl < nslab ? __ldcg(a.smax + row * nslab + sl) : 0u;
        }
      }
      float lv[SMALL_MAX_V / SMALL_THREADS];
#pragma unroll
      for (int u = 0; u < SMALL_MAX_V / SMALL_THREADS; ++u) {
        const int j = tid + u * nt;
        lv[u] = j < V ? __ldcg(lg + j) : 0.f;
      }
      if (warp == 0) {
        const uint32_t xb = warp_bound16_regs(mk, K);
        if (lane == 0) {
          s_misc[0] = 0u;
          s_misc[1] = xb;
        }
      }
      __syncthreads();
      const uint32_t xb = s_misc[1];
#pragma unroll
      for (int u = 0; u < SMALL_MAX_V / SMALL_THREADS; ++u) {
        const int j = tid + u * nt;
        const uint32_t kv = float_key(lv[u]);
        if (j < V && kv >= xb) {
          const unsigned pos = atomicAdd(&s_misc[0], 1u);
          if (pos < static_cast<unsigned>(a.cap)) comp[pos] = composite(kv, j);
        }
      }
      __syncthreads();
      m = static_cast<int>(s_misc[0]);
      __syncthreads();  // s_misc[0] is reset below before anyone could still read it
    }
    if (m > a.cap) {  // x over the whole row: bits 31 .. 16, each kept when at least K keys reach it
      for (int j = tid; j < V; j += nt) keys[j] = float_key(__ldcg(lg + j));
      if (tid == 0) s_misc[0] = 0u;
      __syncthreads();
      uint32_t x = 0;
      int parity = 0;
#pragma unroll 1
      for (int bit = 31; bit >= 16; --bit) {
        const uint32_t c = x | (1u << bit);
        uint32_t cnt = 0;
#pragma unroll 4
        for (int j = tid; j < V; j += nt) cnt += keys[j] >= c ? 1u : 0u;
        if (small_block_sum(cnt, s_red, parity) >= static_cast<uint32_t>(K)) x = c;
        parity ^= 1;
      }
      for (int j = tid; j < V; j += nt) {
        const uint32_t kv = keys[j];
        if (kv >= x) {
          const unsigned pos = atomicAdd(&s_misc[0], 1u);
          if (pos < static_cast<unsigned>(a.cap)) comp[pos] = composite(kv, j);
        }
      }
      __syncthreads();
      m = static_cast<int>(s_misc[0]);
    }
    const uint64_t* top = sorted;
    if (m <= a.cap) {
      sort_runs(comp, sorted, m, K);  // the composites are distinct (one index each)
    } else {  // many keys share the K-th's top 16 bits: the exact selection over the whole row (keys
      // are in shared memory: the whole-row search ran)
      for (int j = tid; j < V; j += nt) idx[j] = j;
      for (int j = tid; j < a.sortP; j += nt) comp[j] = 0ull;
      __syncthreads();
      block_top_composites(keys, idx, V, K, comp, s_red, s_list, s_misc);
      block_bitonic_desc(comp, a.sortP);  // the K composites first; the zero fill sorts last
      top = comp;
    }
    for (int j = tid; j < K; j += nt) {
      a.topk_val[static_cast<int64_t>(row) * a.topk_ld + j] = key_float(composite_key(top[j]));
      a.topk_idx[static_cast<int64_t>(row) * a.topk_ld + j] = composite_idx(top[j]);
    }
    if (a.params != nullptr && a.tokens != nullptr && warp == 0) {  // the draw: warp 0
      const int32_t tok = sample_sorted_warp(prm, top, K, ebuf);
      if (lane == 0) a.tokens[row] = tok;
    }
    __syncthreads();
  }
  pdl_launch_dependents();
}

}  // namespace

SmallPlan plan_small(int B, int H, int V, int K, int num_sms, int dyn_max) {
  SmallPlan p;
  if (B < 1 || B > SMALL_MAX_ROWS || H < 1 || H > SMALL_MAX_H || V < 8 || V > SMALL_MAX_V || V % 8 != 0 || K < 1 ||
      K > V || K > MAX_K || num_sms < 1)
    return p;
  const int groups = V / 8;  // 8-column groups of the vocabulary
  const int per = (groups + num_sms - 1) / num_sms;
  if (per > SMALL_THREADS) return p;
  p.slab_cols = per * 8;
  p.nslab = (V + p.slab_cols - 1) / p.slab_cols;
  if (p.nslab > SMALL_MAX_SLABS) return p;
  int sp = 1;
  while (sp < K) sp <<= 1;
  p.sortP = sp;
  // the gather buffer: twice K, at least 1024, a multiple of 32 (the run sort's granularity) and at
  // least sortP (the whole-row selection's buffer)
  int cap = 2 * K > 1024 ? 2 * K : 1024;
  cap = (cap + 31) & ~31;
  if (cap < sp) cap = sp;
  p.cap = cap;
  const int G = SMALL_THREADS / per;
  const int64_t gemv = static_cast<int64_t>(B) * H * 4 + static_cast<int64_t>(H) * 4 +
                       static_cast<int64_t>(G) * B * p.slab_cols * 4;
  const int64_t sel = static_cast<int64_t>(V) * 8 + static_cast<int64_t>(cap) * 8 + static_cast<int64_t>(K) * 12;
  const int64_t need = gemv > sel ? gemv : sel;
  p.smem_bytes = static_cast<int>(need);
  p.ok = need <= dyn_max;
  return p;
}

cudaError_t prepare_small(int max_smem_optin, int* dyn_max) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, small_tail_kernel);
  if (e != cudaSuccess) return e;
  const int dyn = max_smem_optin - static_cast<int>(fa.sharedSizeBytes);
  e = cudaFuncSetAttribute(small_tail_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  *dyn_max = dyn;
  return cudaSuccess;
}

cudaError_t launch_small(const SmallArgs& a, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nslab);
  cfg.blockDim = dim3(SMALL_THREADS);
  cfg.dynamicSmemBytes = a.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, small_tail_kernel, a);
}

}  // namespace tail
