// The lm_head projection and everything after it -- the global top-k and the
// sampler -- in one launch.
//
// Computes logit[b, v] = row_scale[b] * sum_h a[b, h] * W[h, v] for a batch of
// up to 64 rows ("GPT-OSS Tail Chunked Megakernel Kernel API Reference",
// parameters `lm_head_weight_t` and `deferred_rms`; `emit_logits` for the
// optional fp32 store), then the row's global top-K by (logit desc, index asc)
// (section "Background" and parameter `k`) and one sampled token per row
// (parameter `sampling_params`).
//
// Stream (one persistent CTA per SM):
//   * The vocabulary is split into nslab contiguous slabs of 16-column pairs,
//     balanced to one pair.  A CTA owns one slab and streams its columns of
//     W = [H, V] (bf16, V contiguous) exactly once.
//   * One producer thread fills a ring of shared-memory stages with bulk
//     asynchronous copies (cp.async.bulk, mbarrier transaction counts); a
//     stage holds kpb x 16 rows of W for the CTA's column block (each row one
//     contiguous segment, L2 evict-first) and the matching slices of the
//     packed activations.  The first stages are requested before the
//     dependency wait on the RMSNorm kernel, since W does not depend on it.
//   * Eight consumer warps run mma.sync m16n8k16 (bf16 inputs, fp32
//     accumulation): A is 8 batch rows' hi parts stacked on their lo parts
//     (the activation carried as two bf16 values), B a 16x8 W tile read with
//     ldmatrix.trans (row pitch an odd multiple of 16 bytes: no bank
//     conflicts).  Hi and lo products are summed in the epilogue.
//   * Every column's k-reduction runs through the same mma sequence wherever
//     the column sits, so duplicated W columns give bitwise-equal logits.
//
// Top-k and sampler, in two phases with one exchange between them (only the
// row owners wait, for the slabs' publications, and a slab publishes without
// waiting for anything, so the waits end whatever order the CTAs run in; each
// wait is bounded):
//   P  per (row, slab), no waiting: b = the 8th largest of the 32 lane maxima
//      of the slab's logits (8 distinct elements are >= b).  The slab
//      publishes every element >= b (typically ~10), b, and its 4 largest lane
//      maxima, then releases the row's arrival word.
//   O  CTA r, once all slabs have published row r: x = a lower bound of the
//      K-th largest of the nslab * 4 lane maxima (K distinct elements are
//      >= x); ranks the published candidates >= x; v = the K-th of them.  Only
//      a slab with b > v can hide a top-K element (in [v, b)); its row of the
//      global logits copy is rescanned.  Then the sorted top-k outputs and the
//      draw, with every thread of the CTA.
#include "common.cuh"
#include "internal.h"
#include "moe.cuh"
#include "sampler.cuh"
#include "select.cuh"
#include "tc_common.cuh"

namespace tail {

namespace {

constexpr int MAX_STAGES = 8;
constexpr int BAR_REGION = 256;  // ring barriers and control words at the start of shared memory
constexpr int MOE_HID_DEPTH = 6;  // producer step: stages of residual and slot columns in flight
constexpr int MOE_STAGE_BAR_OFF = 200;  // producer step: one mbarrier per staging slot
constexpr int NLEAD_L = SLAB_BOUND_KEYS * ((MAX_SLABS + 31) / 32);  // leader keys per lane of the owner's bound
constexpr int NGATHER = (MAX_SLABS * SLAB_CAND + GEMV_THREADS - 33) / (GEMV_THREADS - 32);  // slots per gatherer
static_assert(SLAB_BOUND_KEYS == 4 && SLAB_META_WORDS == 8, "a slab's publication is two 16-byte stores");
static_assert(SLAB_LEADERS >= SLAB_BOUND_KEYS && SLAB_LEADERS <= 32, "leaders are distinct lane maxima");
static_assert(GEMV_KPB <= 2, "the pack warp's 32 lanes cover one stage's k columns");
static_assert(MOE_FUSED_MAX_SLOTS == 8, "the activation warp reads a row's slot weights as two float4");
static_assert(MOE_STAGE_BAR_OFF >= 200 && MOE_STAGE_BAR_OFF + 8 * MOE_HID_DEPTH <= BAR_REGION,
              "the staging barriers sit after the ring barriers, the control words and the scale barrier");
static_assert(SLAB_CAND == 32 && (GEMV_THREADS - 32) % 32 == 0, "the owner's gather reads one slab per warp step");

__device__ __forceinline__ uint32_t bf16_bits_rn(float v) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(x), "r"(y) : "memory");
}

__device__ __forceinline__ void consumer_barrier() {
  asm volatile("bar.sync 1, %0;" ::"r"(GEMV_CONSUMER_WARPS * 32) : "memory");
}

// The post-stream phases.  They are inlined: a kernel that holds a real call
// (even one never taken) streams the weight markedly slower.

// ================================================================ phase P: publish the slab's leaders
// Per row: the SLAB_LEADERS largest lane maxima are distinct elements of the
// slab, so at least that many slab elements are >= b, the smallest of them.
// The slab publishes every element >= b (up to SLAB_CAND of them, else none,
// with b raised above every key), b, and its SLAB_BOUND_KEYS largest lane
// maxima -- distinct elements of the row, for the owner's global bound.  An
// unpublished element of the slab is below b.  Nothing waits here: a release
// on the row's arrival word hands the publication to the row's owner.
__device__ __forceinline__ void publish_rows(const GemvArgs& a, const float* slab_logits, int max_cols, int n,
                                         int64_t vbase, int c) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto load_row_keys = [&](int r, uint32_t (&k)[SEL_NPL]) {
    if (a.logits_in_smem) {  // explicit shared-memory loads (a generic pointer would not say so)
      const uint32_t src = smem_u32(slab_logits + r * max_cols) + 4u * lane;
#pragma unroll
      for (int i = 0; i < SEL_NPL; ++i) {
        uint32_t v = 0u;
        if (i * 32 + lane < n) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(src + 128u * i));
        k[i] = i * 32 + lane < n ? float_key(__uint_as_float(v)) : 0u;
      }
    } else {
      const float* src = a.logits_scratch + static_cast<int64_t>(r) * a.V + vbase;
#pragma unroll
      for (int i = 0; i < SEL_NPL; ++i) {
        const int pos = i * 32 + lane;
        k[i] = pos < n ? float_key(src[pos]) : 0u;
      }
    }
  };  for (int r = warp; r < a.B; r += GEMV_CONSUMER_WARPS) {
    uint32_t k[SEL_NPL];
    load_row_keys(r, k);
    uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
#pragma unroll
    for (int i = 0; i < SEL_NPL; i += 4) {
      m0 = max(m0, k[i]);
      m1 = max(m1, k[i + 1]);
      m2 = max(m2, k[i + 2]);
      m3 = max(m3, k[i + 3]);
    }
    // the 32 lane maxima sorted descending over the lanes (bitonic network): lane j then holds the
    // (j+1)-th largest, so lanes 0..3 are the leaders and lane SLAB_LEADERS-1 holds b
    uint32_t lm = max(max(m0, m1), max(m2, m3));
#pragma unroll
    for (int kb = 2; kb <= 32; kb <<= 1) {
#pragma unroll
      for (int j = kb >> 1; j > 0; j >>= 1) {
        const uint32_t o = __shfl_xor_sync(0xffffffffu, lm, j);
        lm = (((lane & j) == 0) == ((lane & kb) == 0)) ? max(lm, o) : min(lm, o);
      }
    }
    uint32_t lead[SLAB_BOUND_KEYS];
#pragma unroll
    for (int j = 0; j < SLAB_BOUND_KEYS; ++j) lead[j] = __shfl_sync(0xffffffffu, lm, j);
    const uint32_t b = __shfl_sync(0xffffffffu, lm, SLAB_LEADERS - 1);
    uint32_t mine = 0;
#pragma unroll
    for (int i = 0; i < SEL_NPL; ++i) mine += (i * 32 + lane < n && k[i] >= b) ? 1u : 0u;
    const uint32_t tot = __reduce_add_sync(0xffffffffu, mine);
    const bool fits = tot <= static_cast<uint32_t>(SLAB_CAND);
    if (fits) {
      uint32_t incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      uint64_t* dst = a.cand + (static_cast<int64_t>(r) * a.nslab + c) * SLAB_CAND;
      uint32_t o = incl - mine;
#pragma unroll
      for (int i = 0; i < SEL_NPL; ++i) {
        const int pos = i * 32 + lane;
        if (pos < n && k[i] >= b) dst[o++] = composite(k[i], static_cast<int32_t>(vbase + pos));
      }
    }
    if (lane == 0) {
      uint4* mp = reinterpret_cast<uint4*>(a.meta + (static_cast<int64_t>(r) * a.nslab + c) * SLAB_META_WORDS);
      mp[0] = make_uint4(lead[0], lead[1], lead[2], lead[3]);
      mp[1] = make_uint4(fits ? tot : 0u, fits ? b : 0xFFFFFFFFu, 0u, 0u);
    }
    // the warp barrier orders every lane's stores (and, through the CTA barriers above, the CTA's
    // global logits copy) before lane 0's release
    __syncwarp();
    if (lane == 0)
      asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(a.row_sync + r), "l"(1ull) : "memory");
  }
}

// sorted[0, min(K, m)) = the top of keys/idx[0, m) in (value desc, index asc)
// order, with every thread of the CTA; returns min(K, m).
__device__ __forceinline__ int rank_top(const GemvArgs& a, const uint32_t* keys, const int32_t* idx, uint64_t* comp,
                                        uint64_t* sorted, int m, uint32_t* s_red, uint32_t* s_list, uint32_t* s_misc) {
  const int want = min(a.K, m);
  if (m <= RANK_SORT_MAX) {
    for (int j = threadIdx.x; j < m; j += blockDim.x) comp[j] = composite(keys[j], idx[j]);
    __syncthreads();
    sort_runs(comp, sorted, m, want);
  } else {
    block_top_composites(keys, idx, m, want, comp, s_red, s_list, s_misc);
    sort_runs(comp, sorted, want, want);
  }
  return want;
}

// Appends to keys/idx[m, ...) the elements of row `row` in each listed slab
// s_bad[0, nbad) whose key is in [thr, b_s) -- the ones the slab did not
// publish that may reach the top K -- read from the global logits copy.  The
// buffer is folded to its top K whenever a slab might not fit.  Returns the
// new count.
__device__ __forceinline__ int rescan_slabs(const GemvArgs& a, int row, uint32_t thr, int nbad, const uint32_t* s_bad,
                                         const uint32_t* s_b, uint32_t* keys, int32_t* idx, uint64_t* comp, int m,
                                         uint32_t* s_red, uint32_t* s_list, uint32_t* s_misc, uint32_t* s_own) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const float* lsrc = a.logits_out ? a.logits_out + static_cast<int64_t>(row) * a.logits_out_ld
                                   : a.logits_scratch + static_cast<int64_t>(row) * a.V;
  for (int bi = 0; bi < nbad; ++bi) {
    const int s = static_cast<int>(s_bad[bi]);
    const int64_t c0 = slab_pair_lo(a.npairs, a.nslab, s) * 16;
    const int w = static_cast<int>(slab_pair_lo(a.npairs, a.nslab, s + 1) * 16 - c0);
    if (m + w > a.capc) {  // keep the top K so far
      for (int j = tid; j < a.sortP; j += nt) comp[j] = 0ull;
      __syncthreads();
      block_top_composites(keys, idx, m, a.K, comp, s_red, s_list, s_misc);
      for (int j = tid; j < a.K; j += nt) {
        keys[j] = composite_key(comp[j]);
        idx[j] = composite_idx(comp[j]);
      }
      if (tid == 0) s_own[1] = static_cast<uint32_t>(a.K);
      __syncthreads();
      m = a.K;
    }
    const uint32_t bs = s_b[s];
    for (int j = tid; j < w; j += nt) {
      const uint32_t kv = float_key(__ldcg(lsrc + c0 + j));
      if (kv >= thr && kv < bs) {
        const uint32_t p = atomicAdd(&s_own[1], 1u);
        keys[p] = kv;
        idx[p] = static_cast<int32_t>(c0 + j);
      }
    }
    __syncthreads();
    m = static_cast<int>(s_own[1]);
  }
  return m;
}

// ================================================================ phase O: the row owner
// CTA c owns rows c, c + nslab, ...  Once every slab has published row r:
//   x = a lower bound of the K-th largest published leader key: at least K
//       distinct elements are >= x, so every top-K element is >= x;
//   F = the published candidates >= x, ranked by (value desc, index asc);
//   v = the K-th of them (x when F holds fewer than K).  A slab whose b is
//       above v may hold unpublished elements in [v, b): its logits row is
//       rescanned for them.  Any other unpublished element is below its
//       slab's b <= v, so the top K of F and the rescans is the exact top K.
__device__ __forceinline__ void own_rows(const GemvArgs& a, uint8_t* ring, int c, uint32_t* s_red, uint32_t* s_list,
                                     uint32_t* s_misc, uint32_t* s_own) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nt = blockDim.x;
  uint32_t* keys = reinterpret_cast<uint32_t*>(ring);
  int32_t* idx = reinterpret_cast<int32_t*>(keys + a.capc);
  uint64_t* comp = reinterpret_cast<uint64_t*>(idx + a.capc);
  uint64_t* sorted = comp + a.sortP;
  float* ebuf = reinterpret_cast<float*>(sorted + a.K);
  uint32_t* s_cnt = reinterpret_cast<uint32_t*>(ebuf + a.K);  // slab counts, then the rescan list
  uint32_t* s_b = s_cnt + a.nslab;
  const int nflat = a.nslab * SLAB_CAND;
  // rescans read the slabs' logits copies (written after the publications) unless the caller's logits
  const bool copied = a.logits_in_smem && !a.logits_out;
  auto wait_copies = [&](int row) {  // bounded wait until every slab's copy of the row is written
    if (tid == 0) {
      unsigned long long v = 0;
      int ok = 1;
      const uint64_t t0 = global_timer_ns();
      while (true) {
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.row_copy + row) : "memory");
        if (v >= static_cast<unsigned long long>(a.nslab)) break;
        if (global_timer_ns() - t0 > a.timeout_ns) {
          raise_error(a.err, DEV_TIMEOUT_BARRIER);
          ok = 0;
          break;
        }
      }
      s_own[2] = ok ? 0u : 1u;
    }
    __syncthreads();
    return s_own[2] == 0u;
  };
  for (int row = c; row < a.B; row += a.nslab) {
    SampleParams prm = {};
    if (a.params != nullptr) prm = load_sample_params(a.params + static_cast<int64_t>(row) * a.ncols, a.ncols);
    // wait (bounded) until every slab has published this row
    if (tid == 0) {
      unsigned long long v = 0;
      int ok = 1;
      const uint64_t t0 = global_timer_ns();
      while (true) {
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.row_sync + row) : "memory");
        if (v >= static_cast<unsigned long long>(a.nslab)) break;
        if (global_timer_ns() - t0 > a.timeout_ns) {
          raise_error(a.err, DEV_TIMEOUT_BARRIER);
          ok = 0;
          break;
        }
      }
      if (ok) a.row_sync[row] = 0ull;  // every slab has arrived: ready for the next run
      s_own[2] = ok ? 0u : 1u;
      s_own[1] = 0u;  // F's size
      s_own[3] = 0u;  // slabs to rescan
    }
    __syncthreads();
    if (s_own[2] != 0u) break;  // uniform: a slab never published (the error flag is raised)
    const uint32_t* meta = a.meta + static_cast<int64_t>(row) * a.nslab * SLAB_META_WORDS;
    const uint64_t* cand = a.cand + static_cast<int64_t>(row) * nflat;
    uint64_t cr[NGATHER];
    const int tg = tid - 32, ntg = nt - 32;
    if (warp == 0) {
      // the leaders, for the bound; every slab's count and b
      uint32_t pk[NLEAD_L];
#pragma unroll
      for (int j = 0; j < NLEAD_L / SLAB_BOUND_KEYS; ++j) {
        const int s = j * 32 + lane;
        uint4 l = make_uint4(0u, 0u, 0u, 0u);
        if (s < a.nslab) {
          l = __ldcg(reinterpret_cast<const uint4*>(meta + s * SLAB_META_WORDS));
          const uint2 cb = __ldcg(reinterpret_cast<const uint2*>(meta + s * SLAB_META_WORDS + 4));
          s_cnt[s] = cb.x;
          s_b[s] = cb.y;
        }
        pk[4 * j] = l.x;
        pk[4 * j + 1] = l.y;
        pk[4 * j + 2] = l.z;
        pk[4 * j + 3] = l.w;
      }
      const uint32_t x = a.nslab * SLAB_BOUND_KEYS >= a.K ? warp_bound16_span_regs(pk, a.K) : 0u;
      if (lane == 0) s_own[0] = x;
    } else {
      // the candidate slots, loaded blind; the empty ones are dropped below
#pragma unroll
      for (int q = 0; q < NGATHER; ++q) {
        const int f = q * ntg + tg;
        cr[q] = f < nflat ? __ldcg(cand + f) : 0ull;
      }
    }
    __syncthreads();
    const uint32_t x = s_own[0];
    if (warp != 0) {
      // a warp's 32 slots of one step are one slab's (SLAB_CAND == 32, ntg a multiple of 32); the
      // warp counts its kept slots by ballots, reserves room once, then writes them
      uint32_t bm[NGATHER];
      uint32_t cnt = 0u;
#pragma unroll
      for (int q = 0; q < NGATHER; ++q) {
        const int f = q * ntg + tg;
        const bool take = f < nflat && static_cast<uint32_t>(lane) < s_cnt[min(f, nflat - 1) / SLAB_CAND] &&
                          composite_key(cr[q]) >= x;
        bm[q] = __ballot_sync(0xffffffffu, take);
        cnt += static_cast<uint32_t>(__popc(bm[q]));
      }
      uint32_t base = 0u;
      if (lane == 0 && cnt != 0u) base = atomicAdd(&s_own[1], cnt);
      base = __shfl_sync(0xffffffffu, base, 0);
      const uint32_t below = lanemask_lt();
#pragma unroll
      for (int q = 0; q < NGATHER; ++q) {
        if (bm[q] & (1u << lane)) {
          const uint32_t p = base + static_cast<uint32_t>(__popc(bm[q] & below));
          keys[p] = composite_key(cr[q]);
          idx[p] = composite_idx(cr[q]);
        }
        base += static_cast<uint32_t>(__popc(bm[q]));
      }
    }
    __syncthreads();
    int m = static_cast<int>(s_own[1]);
    int want = rank_top(a, keys, idx, comp, sorted, m, s_red, s_list, s_misc);
    // slabs whose unpublished elements may reach the top K
    const uint32_t thr = want >= a.K ? composite_key(sorted[a.K - 1]) : x;
    for (int s = tid; s < a.nslab; s += nt)
      if (s_b[s] > thr) s_cnt[atomicAdd(&s_own[3], 1u)] = static_cast<uint32_t>(s);
    __syncthreads();
    const int nbad = static_cast<int>(s_own[3]);
    if (nbad > 0) {
      if (copied && !wait_copies(row)) break;  // uniform: a copy never arrived (the error flag is raised)
      m = rescan_slabs(a, row, thr, nbad, s_cnt, s_b, keys, idx, comp, m, s_red, s_list, s_misc, s_own);
      want = rank_top(a, keys, idx, comp, sorted, m, s_red, s_list, s_misc);
    }
    for (int j = tid; j < want; j += nt) {
      a.topk_val[static_cast<int64_t>(row) * a.topk_ld + j] = key_float(composite_key(sorted[j]));
      a.topk_idx[static_cast<int64_t>(row) * a.topk_ld + j] = composite_idx(sorted[j]);
    }
    if (a.params != nullptr && a.tokens != nullptr && warp == 0) {  // the draw: warp 0
      const int32_t tok = sample_sorted_warp(prm, sorted, want, ebuf);
      if (lane == 0) a.tokens[row] = tok;
    }
    __syncthreads();
    if (copied) {  // every copy of the row has landed by now, normally: clear the word for the next run
      if (!wait_copies(row)) break;
      if (tid == 0) a.row_copy[row] = 0ull;
    }
  }
}

// ================================================================ activations with the producer step
// The activation warp of the fused form when the hidden state is formed in
// the kernel from the bf16 residual and up to MOE_FUSED_MAX_SLOTS expert
// slots (moe.cuh).  Per ring stage (k columns [32 js, 32 js + 32)):
//   * two tensor copies (TMA) bring the stage's columns of every residual row
//     and of every row's slots into a staging slot (MOE_HID_DEPTH slots in
//     flight, one mbarrier each): the copy engine's path, as for W, with two
//     requests a stage.  The slot box always spans MOE_FUSED_MAX_SLOTS slots;
//     those past S read as zeros and their weights are zero, so the chains
//     run over all of them (fma(+0, +0, acc) is acc: a chain from +0 never
//     holds -0), with the routed-slot count as a compile-time constant;
//   * the combine: lane (g, q) forms h = bf16(x + bf16(r + sh)) for columns
//     [4q, 4q + 4) of rows g, g + 4, ... (vector loads of four columns, the
//     routed and shared fma chains per column), writes h over the residual
//     row in the staging slot, and CTA 0 also writes it to the caller's buffer;
//   * then the plain fused form on h, lane j on column j as without the
//     producer step (the same order of the squares' sums, so rstd is the one
//     the tail computes on h given as its input): x^2 into the row's sum,
//     a = h * gamma split into hi + lo, stored in A-fragment order and released
//     by the lane's arrival on the stage's full barrier.
template <int MT, int SZ, int NR>
__device__ __forceinline__ void moe_combine_stage(const GemvArgs& a, uint8_t* slot, int ncols, int64_t c0,
                                                  const float (&wl)[MT * 2][MOE_FUSED_MAX_SLOTS]) {
  constexpr int NS = MOE_FUSED_MAX_SLOTS;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 3, q = lane & 7;
  uint8_t* xq = slot + q * 8;
  const uint8_t* yq = slot + moe_y_offset(a.B) + q * 4 * SZ;
#pragma unroll
  for (int p = 0; p < MT * 2; ++p) {
    const int r = g + 4 * p;
    if (r < a.B) {
      float y[NS][4];
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const uint8_t* e = yq + (r * NS + s) * 32 * SZ;
        if constexpr (SZ == 4) {
          const float4 v = *reinterpret_cast<const float4*>(e);
          y[s][0] = v.x; y[s][1] = v.y; y[s][2] = v.z; y[s][3] = v.w;
        } else {
          const uint2 v = *reinterpret_cast<const uint2*>(e);
          y[s][0] = __uint_as_float(v.x << 16); y[s][1] = __uint_as_float(v.x & 0xffff0000u);
          y[s][2] = __uint_as_float(v.y << 16); y[s][3] = __uint_as_float(v.y & 0xffff0000u);
        }
      }
      const uint2 xv = *reinterpret_cast<const uint2*>(xq + r * 64);
      // slots past S are zero rows of zero weight: fma(+0, +0, acc) leaves acc (never -0) as it is
      float rr[4] = {0.f, 0.f, 0.f, 0.f}, sh[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < NR; ++s)
#pragma unroll
        for (int j = 0; j < 4; ++j) rr[j] = __fmaf_rn(wl[p][s], y[s][j], rr[j]);
#pragma unroll
      for (int s = NR; s < NS; ++s)
#pragma unroll
        for (int j = 0; j < 4; ++j) sh[j] = __fmaf_rn(wl[p][s], y[s][j], sh[j]);
      const uint32_t h0 = moe_finish(xv.x & 0xffffu, rr[0], sh[0]), h1 = moe_finish(xv.x >> 16, rr[1], sh[1]);
      const uint32_t h2 = moe_finish(xv.y & 0xffffu, rr[2], sh[2]), h3 = moe_finish(xv.y >> 16, rr[3], sh[3]);
      const uint2 hv = make_uint2(h0 | (h1 << 16), h2 | (h3 << 16));
      *reinterpret_cast<uint2*>(xq + r * 64) = hv;
      if (a.moe.h_out != nullptr && blockIdx.x == 0 && q * 4 < ncols)
        *reinterpret_cast<uint2*>(a.moe.h_out + static_cast<int64_t>(r) * a.H + c0 + q * 4) = hv;
    }
  }
}

// moe_combine_stage with the routed-slot count as a constant (the chains then carry no branch)
template <int MT, int SZ>
__device__ __forceinline__ void moe_combine_stage_nr(const GemvArgs& a, uint8_t* slot, int ncols, int64_t c0,
                                                     const float (&wl)[MT * 2][MOE_FUSED_MAX_SLOTS]) {
  switch (a.moe.n_routed) {
    case 0: moe_combine_stage<MT, SZ, 0>(a, slot, ncols, c0, wl); break;
    case 1: moe_combine_stage<MT, SZ, 1>(a, slot, ncols, c0, wl); break;
    case 2: moe_combine_stage<MT, SZ, 2>(a, slot, ncols, c0, wl); break;
    case 3: moe_combine_stage<MT, SZ, 3>(a, slot, ncols, c0, wl); break;
    case 4: moe_combine_stage<MT, SZ, 4>(a, slot, ncols, c0, wl); break;
    case 5: moe_combine_stage<MT, SZ, 5>(a, slot, ncols, c0, wl); break;
    case 6: moe_combine_stage<MT, SZ, 6>(a, slot, ncols, c0, wl); break;
    case 7: moe_combine_stage<MT, SZ, 7>(a, slot, ncols, c0, wl); break;
    default: moe_combine_stage<MT, SZ, 8>(a, slot, ncols, c0, wl); break;
  }
}

template <int MT>
__device__ __forceinline__ void moe_activation_warp(const GemvArgs& a, uint8_t* smem, uint32_t full0, uint32_t empty0,
                                                    uint32_t scale_bar, volatile int* s_abort, float* s_scale,
                                                    int total, int spb) {
  constexpr int NS = MOE_FUSED_MAX_SLOTS;
  constexpr int ROWS = MT * MTILE_ROWS;
  constexpr int DEPTH = MOE_HID_DEPTH;
  const int lane = threadIdx.x & 31;
  const int KPB = a.kpb, NST = a.nstages;
  const int active_end = a.zero_pad ? a.H : a.Hu;
  const int kc = lane & (KSTEP - 1), ksub = lane >> 4;  // a stage is at most two k-steps: 32 columns
  const int col = ksub * KSTEP + kc;
  const int S = a.moe.S;
  const int sesz = a.moe.slot_dtype == 0 ? 4 : 2;
  const int slot_bytes = a.hid_slot_bytes;
  const int stg_off = BAR_REGION + NST * a.stage_bytes;  // the staging ring, after the weight ring
  const uint32_t stg = smem_u32(smem) + static_cast<uint32_t>(stg_off);
  const uint32_t sbar0 = smem_u32(smem + MOE_STAGE_BAR_OFF);
  const uint32_t ring_u32 = smem_u32(smem + BAR_REGION);
  const uint32_t xbytes = static_cast<uint32_t>(a.B) * 32u * 2u;
  const uint32_t ybytes = S > 0 ? static_cast<uint32_t>(a.B) * NS * 32u * static_cast<uint32_t>(sesz) : 0u;
  if (S == 0)  // no slot copy ever lands: the slot rows read as zeros in every staging slot
    for (int d = 0; d < DEPTH; ++d) {
      float* yrow = reinterpret_cast<float*>(smem + stg_off + d * slot_bytes + moe_y_offset(a.B));
      for (int i = lane; i < a.B * NS * 32; i += 32) yrow[i] = 0.f;
    }
  pdl_wait();  // the residual, the slots and their weights may come from the previous kernel
  float wl[MT * 2][NS];  // the weights of this lane's rows of the combine: g, g + 4, ...
#pragma unroll
  for (int p = 0; p < MT * 2; ++p) {
    const int r = (lane >> 3) + 4 * p;
#pragma unroll
    for (int sl = 0; sl < NS; ++sl) wl[p][sl] = (r < a.B && sl < S) ? a.moe.w[r * S + sl] : 0.f;
  }
  __syncwarp();
  const uint64_t pol = policy_evict_last();  // every CTA reads the same rows
  auto issue = [&](int it) {
    if (it >= total || lane != 0) return;
    const int c0 = (it % spb) * KPB * KSTEP;
    const uint32_t slot = stg + static_cast<uint32_t>((it % DEPTH) * slot_bytes);
    const uint32_t bar = sbar0 + 8u * static_cast<uint32_t>(it % DEPTH);
    mbar_arrive_expect_tx(bar, xbytes + ybytes);
    tma_load_2d(slot, &a.moe_map_x, c0, 0, bar, pol);
    if (S > 0) tma_load_3d(slot + static_cast<uint32_t>(moe_y_offset(a.B)), &a.moe_map_y, c0, 0, 0, bar, pol);
  };
  float ss[ROWS];
#pragma unroll
  for (int r = 0; r < ROWS; ++r) ss[r] = 0.f;
  for (int p = 0; p < DEPTH - 1; ++p) issue(p);
  int issued = min(DEPTH - 1, total);
  int it = 0;
  for (; it < total; ++it) {
    issue(it + DEPTH - 1);  // into the slot the previous iteration finished reading
    if (it + DEPTH - 1 < total) issued = it + DEPTH;
    const bool landed = __all_sync(0xffffffffu, mbar_wait_bounded(sbar0 + 8u * static_cast<uint32_t>(it % DEPTH),
                                                                   static_cast<uint32_t>(it / DEPTH) & 1u,
                                                                   a.timeout_ns));
    if (!landed) {
      if (lane == 0) {
        raise_error(a.err, DEV_TIMEOUT_FULL);
        *s_abort = 1;
      }
      break;
    }
    const int js = it % spb;
    const int kn = min(KPB, a.ksteps - js * KPB);
    const int h = (js * KPB + ksub) * KSTEP + kc;
    const bool in = ksub < kn;
    const float gc = in && h < active_end ? a.gamma[h] : 0.f;
    uint8_t* slot = smem + stg_off + (it % DEPTH) * slot_bytes;
    if (sesz == 4)
      moe_combine_stage_nr<MT, 4>(a, slot, kn * KSTEP, static_cast<int64_t>(js) * KPB * KSTEP, wl);
    else
      moe_combine_stage_nr<MT, 2>(a, slot, kn * KSTEP, static_cast<int64_t>(js) * KPB * KSTEP, wl);
    fence_proxy_async_smem();  // h's stores, before a later tensor copy refills the slot
    __syncwarp();  // h of every row is in the staging slot
    float xc[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
      xc[r] = (in && h < active_end && r < a.B)
                  ? __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(slot + r * 64 + col * 2)) << 16)
                  : 0.f;
    __syncwarp();  // the slot is refilled by the next iteration's copies
    if (*s_abort) break;
    if (it >= NST && !__all_sync(0xffffffffu, mbar_wait_bounded(empty0 + 8 * (it % NST),
                                                                 static_cast<uint32_t>((it / NST) - 1) & 1u,
                                                                 a.timeout_ns))) {
      if (lane == 0) {
        raise_error(a.err, DEV_TIMEOUT_EMPTY);
        *s_abort = 1;
      }
      break;
    }
    const uint32_t wbase = ring_u32 + static_cast<uint32_t>((it % NST) * a.stage_bytes + KPB * KSTEP * a.pitch +
                                                            ksub * MT * APACK_TILE_BYTES + ((kc & 7) >> 1) * 16 +
                                                            (kc < 8 ? 0 : 8));
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      ss[r] = fmaf(xc[r], xc[r], ss[r]);
      const float v = xc[r] * gc;
      const uint32_t hi = bf16_bits_rn(v);
      const uint32_t lo = bf16_bits_rn(v - __uint_as_float(hi << 16));
      const uint32_t hi1 = __shfl_down_sync(0xffffffffu, hi, 1);
      const uint32_t lo1 = __shfl_down_sync(0xffffffffu, lo, 1);
      if (in && (kc & 1) == 0)
        st_shared_v2(wbase + static_cast<uint32_t>(((r >> 3) * 32 + (r & 7) * 4) * 16), hi | (hi1 << 16),
                     lo | (lo1 << 16));
    }
    mbar_arrive(full0 + 8 * (it % NST));  // each lane releases its own stores
  }
  // no copy may land after the warp moves on: wait (bounded) for the staging slots still in flight
  for (int j = it; j < issued; ++j)
    if (!mbar_wait_bounded(sbar0 + 8u * static_cast<uint32_t>(j % DEPTH), static_cast<uint32_t>(j / DEPTH) & 1u,
                           DEFAULT_TIMEOUT_NS)) {
      if (lane == 0) raise_error(a.err, DEV_TIMEOUT_DRAIN);
      break;
    }
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    float t = ss[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) s_scale[r] = r < a.B ? 1.0f / sqrtf(t / static_cast<float>(a.Hu) + a.eps) : 0.f;
  }
  if (lane == 0) mbar_arrive(scale_bar);
}

template <int MT, int PW, bool MOE>
__global__ void __launch_bounds__(GEMV_THREADS, 1) lmhead_tail_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t s_red[64];
  __shared__ uint32_t s_list[SEL_BLOCK_BUCKET_MAX];
  __shared__ uint32_t s_misc[4];
  __shared__ uint32_t s_own[4];  // owner: x, |F|, wait failed, slabs to rescan
  __shared__ float s_scale[MAX_ROWS_PER_PASS];  // fused: the rows' rstd
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + MAX_STAGES);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + 2 * MAX_STAGES * 8);
  int* s_consumed_min = reinterpret_cast<int*>(smem + 2 * MAX_STAGES * 8 + 4);
  int* s_issued = reinterpret_cast<int*>(smem + 2 * MAX_STAGES * 8 + 8);
  const uint32_t scale_bar = smem_u32(smem + 192);  // fused: s_scale is ready
  uint8_t* ring = smem + BAR_REGION;
  const uint32_t ring_u32 = smem_u32(ring);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const int64_t pair_lo = slab_pair_lo(a.npairs, a.nslab, c);
  const int64_t pair_hi = slab_pair_lo(a.npairs, a.nslab, c + 1);
  const int slab_pairs = static_cast<int>(pair_hi - pair_lo);
  const int nblk = (slab_pairs + a.cb_pairs - 1) / a.cb_pairs;
  const int KPB = a.kpb;                       // k-steps (16 rows each) per ring stage
  const int spb = (a.ksteps + KPB - 1) / KPB;  // ring stages per column block
  const int total = nblk * spb;
  const int NST = a.nstages;
  const int max_cols = a.max_slab_cols;
  float* slab_logits = reinterpret_cast<float*>(ring);

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full0 + 8 * s, a.fused ? 33 : 1);  // fused: the producer and the pack warp's 32 lanes
      mbar_init(empty0 + 8 * s, GEMV_CONSUMER_WARPS);
    }
    mbar_init(scale_bar, 1);
    if constexpr (MOE)
      for (int d = 0; d < MOE_HID_DEPTH; ++d) mbar_init(smem_u32(smem + MOE_STAGE_BAR_OFF) + 8 * d, 1);
    *s_abort = 0;
    *s_consumed_min = total;
    *s_issued = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == GEMV_PRODUCER_WARP) {
    // ================================================================ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      const uint32_t abytes = a.fused ? 0u : static_cast<uint32_t>(MT * APACK_TILE_BYTES);
      auto stage_of = [&](int it) { return ring_u32 + static_cast<uint32_t>((it % NST) * a.stage_bytes); };
      auto issue_w = [&](int it) {
        const int blk = it / spb, js = it % spb;
        const int kn = min(KPB, a.ksteps - js * KPB);
        const int64_t bp0 = pair_lo + static_cast<int64_t>(blk) * a.cb_pairs;
        const int npb = static_cast<int>(min(static_cast<int64_t>(a.cb_pairs), pair_hi - bp0));
        const uint32_t row_bytes = static_cast<uint32_t>(npb) * 32u;
        const uint32_t bar = full0 + 8 * (it % NST);
        const uint32_t st = stage_of(it);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kn) * (KSTEP * row_bytes + abytes));
        const uint16_t* src = a.w + static_cast<int64_t>(js) * KPB * KSTEP * a.V + bp0 * 16;
#pragma unroll 4
        for (int r = 0; r < kn * KSTEP; ++r)
          bulk_g2s(st + static_cast<uint32_t>(r * a.pitch), src + static_cast<int64_t>(r) * a.V, row_bytes, bar,
                   pol_w);
      };
      auto issue_a = [&](int it) {
        const int js = it % spb;
        const int kn = min(KPB, a.ksteps - js * KPB);
        bulk_g2s(stage_of(it) + static_cast<uint32_t>(KPB * KSTEP * a.pitch),
                 a.apack + static_cast<int64_t>(js) * KPB * abytes, static_cast<uint32_t>(kn) * abytes,
                 full0 + 8 * (it % NST), pol_a);
      };
      const int npre = min(NST, total);
      for (int it = 0; it < npre; ++it)
        if (it != a.drop_iter) issue_w(it);
      if (!a.fused) {
        pdl_wait();  // the packed activations come from the RMSNorm kernel
        for (int it = 0; it < npre; ++it)
          if (it != a.drop_iter) issue_a(it);
      }
      int issued = npre;
      for (int it = npre; it < total; ++it) {
        if (*s_abort) break;
        const uint32_t par = static_cast<uint32_t>((it / NST) - 1) & 1u;
        if (!mbar_wait_bounded(empty0 + 8 * (it % NST), par, a.timeout_ns)) {
          raise_error(a.err, DEV_TIMEOUT_EMPTY);
          *s_abort = 1;
          break;
        }
        if (it != a.drop_iter) {
          issue_w(it);
          if (!a.fused) issue_a(it);
        }
        issued = it + 1;
      }
      *s_issued = issued;
    }
  } else if (warp == GEMV_PACK_WARP) {
    // ================================================================ activations (fused RMSNorm)
    // Deferred form: a = x * gamma feeds the GEMM and rstd scales its output, so
    // stage it needs only k columns [32 js, 32 js + 32) of every row.  Lane j
    // widens x[r][32 js + j] exactly, adds x^2 to row r's running sum, splits
    // a = hi + lo into two bf16 values and writes them in the mma.sync
    // A-fragment order the RMSNorm kernel uses; its arrival on the stage's full
    // barrier releases them.  After the last stage, rstd = 1 / sqrt(ss / H_u +
    // eps) per row (fixed order: lane sums, then an xor butterfly).
    if constexpr (MOE) {  // the same, with the hidden state formed from the residual and the slots
      if (a.fused) moe_activation_warp<MT>(a, smem, full0, empty0, scale_bar, s_abort, s_scale, total, spb);
    } else {
    if constexpr (MT <= FUSED_MAX_MT) {  // larger batches take the RMSNorm kernel (registers)
    if (a.fused) {
      pdl_wait();  // hidden may come from the previous kernel
      const int active_end = a.zero_pad ? a.H : a.Hu;
      const int kc = lane & (KSTEP - 1), ksub = lane >> 4;  // a stage is at most two k-steps: 32 columns
      const int esz = a.dtype == 0 ? 4 : 2;
      const uint32_t stg = ring_u32 + static_cast<uint32_t>(NST * a.stage_bytes);  // hidden staging ring
      const char* hid = static_cast<const char*>(a.hidden);
      // stage `it`'s k columns of every row -> staging slot it % HID_DEPTH, 16-byte async copies
      auto issue_hidden = [&](int it) {
        if (it < total) {
          const int js = it % spb;
          const int kn = min(KPB, a.ksteps - js * KPB);
          const int cpr = kn * KSTEP * esz / 16;  // 16-byte chunks per row
          const uint32_t slot = stg + static_cast<uint32_t>((it % HID_DEPTH) * HID_SLOT_BYTES);
          for (int q = lane; q < a.B * cpr; q += 32) {
            const int r = q / cpr, c = q - r * cpr;
            const char* src = hid + (static_cast<int64_t>(r) * a.H + js * KPB * KSTEP) * esz + c * 16;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(slot + r * HID_ROW_BYTES + c * 16),
                         "l"(src) : "memory");
          }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      };
      float ss[MT * MTILE_ROWS];
#pragma unroll
      for (int r = 0; r < MT * MTILE_ROWS; ++r) ss[r] = 0.f;
      for (int p = 0; p < HID_DEPTH - 1; ++p) issue_hidden(p);
      for (int it = 0; it < total; ++it) {
        issue_hidden(it + HID_DEPTH - 1);
        asm volatile("cp.async.wait_group %0;" ::"n"(HID_DEPTH - 1) : "memory");
        __syncwarp();
        const int js = it % spb;
        const int kn = min(KPB, a.ksteps - js * KPB);
        const int h = (js * KPB + ksub) * KSTEP + kc;
        const bool act = ksub < kn && h < active_end;
        const float gc = act ? a.gamma[h] : 0.f;
        const uint8_t* srow = smem + BAR_REGION + NST * a.stage_bytes + (it % HID_DEPTH) * HID_SLOT_BYTES +
                              (ksub * KSTEP + kc) * esz;
        float xc[MT * MTILE_ROWS];
#pragma unroll
        for (int r = 0; r < MT * MTILE_ROWS; ++r) {
          float x = 0.f;
          if (act && r < a.B) {
            const uint8_t* e = srow + r * HID_ROW_BYTES;
            x = a.dtype == 0 ? *reinterpret_cast<const float*>(e)
                : a.dtype == 1 ? __half2float(*reinterpret_cast<const __half*>(e))
                               : __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(e));
          }
          xc[r] = x;
        }
        __syncwarp();  // the slot is refilled by the next iteration's copies
        if (*s_abort) break;
        if (it >= NST && !mbar_wait_bounded(empty0 + 8 * (it % NST), static_cast<uint32_t>((it / NST) - 1) & 1u,
                                            a.timeout_ns)) {
          raise_error(a.err, DEV_TIMEOUT_EMPTY);
          *s_abort = 1;
          break;
        }
        const uint32_t wbase = ring_u32 + static_cast<uint32_t>((it % NST) * a.stage_bytes + KPB * KSTEP * a.pitch +
                                                                ksub * MT * APACK_TILE_BYTES + ((kc & 7) >> 1) * 16 +
                                                                (kc < 8 ? 0 : 8));
#pragma unroll
        for (int r = 0; r < MT * MTILE_ROWS; ++r) {
          ss[r] = fmaf(xc[r], xc[r], ss[r]);
          const float v = xc[r] * gc;
          const uint32_t hi = bf16_bits_rn(v);
          const uint32_t lo = bf16_bits_rn(v - __uint_as_float(hi << 16));
          const uint32_t hi1 = __shfl_down_sync(0xffffffffu, hi, 1);
          const uint32_t lo1 = __shfl_down_sync(0xffffffffu, lo, 1);
          if (ksub < kn && (kc & 1) == 0)
            st_shared_v2(wbase + static_cast<uint32_t>(((r >> 3) * 32 + (r & 7) * 4) * 16), hi | (hi1 << 16),
                         lo | (lo1 << 16));
        }
        mbar_arrive(full0 + 8 * (it % NST));  // each lane releases its own stores
      }
      asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy lands after the warp moves on
#pragma unroll
      for (int r = 0; r < MT * MTILE_ROWS; ++r) {
        float t = ss[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) s_scale[r] = r < a.B ? 1.0f / sqrtf(t / static_cast<float>(a.Hu) + a.eps) : 0.f;
      }
      if (lane == 0) mbar_arrive(scale_bar);
    }
    }
    }
  } else {
    // ================================================================ consumers
    pdl_wait();  // row_scale (RMSNorm kernel) is read and outputs are written only after the previous kernel
    const int g = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3;  // ldmatrix: this lane addresses a row of matrix mi
    const uint32_t lrow_off = static_cast<uint32_t>(((mi & 1) * 8 + (lane & 7)) * a.pitch + (mi >> 1) * 16);
    bool ok = true;
    int it = 0;
    float acc[MT][PW][2][4];

    // hi + lo, row scale, optional fp32 store, and staging of one column block's logits
    auto block_epilogue = [&](int64_t bp0, int npb) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int r = m * MTILE_ROWS + g;
        if (r >= a.B) continue;
        const float sc = a.fused ? s_scale[r] : a.row_scale[r];
#pragma unroll
        for (int q = 0; q < PW; ++q) {
          const int pr = warp + GEMV_CONSUMER_WARPS * q;
          if (pr >= npb) continue;
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            const int64_t col = (bp0 + pr) * 16 + n * 8 + 2 * tq;
            float2 v;
            v.x = (acc[m][q][n][0] + acc[m][q][n][2]) * sc;
            v.y = (acc[m][q][n][1] + acc[m][q][n][3]) * sc;
            if (a.logits_out) *reinterpret_cast<float2*>(a.logits_out + r * a.logits_out_ld + col) = v;
            if (a.logits_in_smem)
              *reinterpret_cast<float2*>(slab_logits + r * max_cols + (col - pair_lo * 16)) = v;
            else  // the slab's logits live in global memory
              *reinterpret_cast<float2*>(a.logits_scratch + static_cast<int64_t>(r) * a.V + col) = v;
          }
        }
      }
    };

    int64_t last_bp0 = pair_lo;
    int last_npb = 0;
    for (int blk = 0; blk < nblk && ok; ++blk) {
      const int64_t bp0 = pair_lo + static_cast<int64_t>(blk) * a.cb_pairs;
      const int npb = static_cast<int>(min(static_cast<int64_t>(a.cb_pairs), pair_hi - bp0));
      last_bp0 = bp0;
      last_npb = npb;
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int q = 0; q < PW; ++q)
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[m][q][n][r] = 0.f;

      for (int js = 0; js < spb; ++js, ++it) {
        const int s = it % NST;
        const uint32_t par = static_cast<uint32_t>(it / NST) & 1u;
        if (!mbar_wait_bounded(full0 + 8 * s, par, a.timeout_ns)) {
          raise_error(a.err, DEV_TIMEOUT_FULL);
          *s_abort = 1;
          ok = false;
          break;
        }
        const uint32_t st = ring_u32 + static_cast<uint32_t>(s * a.stage_bytes);
        const int kn = min(KPB, a.ksteps - js * KPB);
#pragma unroll 1
        for (int kk = 0; kk < kn; ++kk) {
          const uint32_t wst = st + static_cast<uint32_t>(kk * KSTEP * a.pitch);
          const uint32_t abase =
              st + static_cast<uint32_t>(KPB * KSTEP * a.pitch + kk * MT * APACK_TILE_BYTES) + lane * 16;
          uint32_t af[MT][4];
#pragma unroll
          for (int m = 0; m < MT; ++m) lds128(abase + m * APACK_TILE_BYTES, af[m][0], af[m][1], af[m][2], af[m][3]);
#pragma unroll
          for (int q = 0; q < PW; ++q) {
            const int pr = warp + GEMV_CONSUMER_WARPS * q;
            if (pr < npb) {
              uint32_t b0, b1, b2, b3;
              ldsm_x4_trans(wst + lrow_off + static_cast<uint32_t>(pr * 32), b0, b1, b2, b3);
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                mma_bf16_16816(acc[m][q][0], af[m][0], af[m][1], af[m][2], af[m][3], b0, b1);
                mma_bf16_16816(acc[m][q][1], af[m][0], af[m][1], af[m][2], af[m][3], b2, b3);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
      }
      // global staging: every block's logits leave registers right away
      if (ok && !a.logits_in_smem) block_epilogue(bp0, npb);
    }
    atomicMin(s_consumed_min, it);

    // Every consumer warp reaches both barriers whatever happened above; the
    // abort decision is read once, after the first of them.
    consumer_barrier();  // all stages consumed: the ring may now hold the slab logits
    bool aborted_c = *s_abort != 0;
    if (!aborted_c && a.fused && !mbar_wait_bounded(scale_bar, 0u, a.timeout_ns)) {
      raise_error(a.err, DEV_TIMEOUT_FULL);
      aborted_c = true;
    }
    if (!aborted_c && a.logits_in_smem) block_epilogue(last_bp0, last_npb);
    __threadfence_block();
    consumer_barrier();
  }

  // ================================================================ drain
  // No copy may still be landing when the ring is reused or the CTA leaves.
  __syncthreads();
  if (warp == GEMV_CONSUMER_WARPS && lane == 0) {
    const int issued = *s_issued;
    for (int it = *s_consumed_min; it < issued; ++it) {
      if (it == a.drop_iter) continue;  // never issued
      const uint32_t par = static_cast<uint32_t>(it / NST) & 1u;
      if (!mbar_wait_bounded(full0 + 8 * (it % NST), par, DEFAULT_TIMEOUT_NS)) {
        raise_error(a.err, DEV_TIMEOUT_DRAIN);
        break;
      }
    }
  }
  __syncthreads();
  const bool aborted = *s_abort != 0;
  const int n = slab_pairs * 16;
  const int64_t vbase = pair_lo * 16;


  if (!aborted && warp < GEMV_CONSUMER_WARPS) publish_rows(a, slab_logits, max_cols, n, vbase, c);
  if (!aborted && a.logits_in_smem && !a.logits_out) {
    // a global copy of the slab's logits for the row owners' rescans, written after the publication
    // so that its release does not wait for these stores; counted per row on its own word
    const int n4 = n / 4;
    for (int q = tid; q < a.B * n4; q += blockDim.x) {
      const int r = q / n4, i = q - r * n4;
      reinterpret_cast<float4*>(a.logits_scratch + static_cast<int64_t>(r) * a.V + vbase)[i] =
          reinterpret_cast<const float4*>(slab_logits + r * max_cols)[i];
    }
    __syncthreads();
    if (tid < a.B) {
      __threadfence();
      asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(a.row_copy + tid), "l"(1ull) : "memory");
    }
  }
  if (!aborted) own_rows(a, ring, c, s_red, s_list, s_misc, s_own);
  pdl_launch_dependents();
}

template <int MT, int PW, bool MOE>
cudaError_t launch_t(const GemvArgs& a, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nslab);
  cfg.blockDim = dim3(GEMV_THREADS);
  cfg.dynamicSmemBytes = a.smem_bytes;
  cfg.stream = stream;
  // A plain launch: no CTA waits for one that has not started (slabs publish without waiting; only
  // the row owners wait, for the publications), so the grid needs no co-residency guarantee.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, lmhead_tail_kernel<MT, PW, MOE>, a);
}

int mt_template(int B) {
  const int mt = (B + MTILE_ROWS - 1) / MTILE_ROWS;
  return mt <= 1 ? 1 : mt <= 2 ? 2 : mt <= 4 ? 4 : 8;
}

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

GemvPlan plan_gemv(int B, int H, int V, int K, int nslab, int max_smem, int kpb, int max_stages, int moe_slots,
                   int moe_slot_bytes) {
  (void)H;
  GemvPlan p = {};
  p.mt = mt_template(B);
  p.pw = p.mt == 1 ? 12 : p.mt == 2 ? 6 : p.mt == 4 ? 3 : 1;
  p.cb_pairs = GEMV_CONSUMER_WARPS * p.pw;
  const int64_t npairs = V / 16;
  const int max_slab_pairs = static_cast<int>((npairs + nslab - 1) / nslab);
  const int cb_eff = max_slab_pairs < p.cb_pairs ? max_slab_pairs : p.cb_pairs;
  p.pitch = cb_eff * 32 + 16;  // odd multiple of 16 bytes: conflict-free ldmatrix rows
  p.kpb = kpb;
  p.stage_bytes = ((kpb * (KSTEP * p.pitch + p.mt * APACK_TILE_BYTES)) + 127) & ~127;
  const int budget = max_smem - BAR_REGION;
  // fused: hidden staging after the ring (with the producer step: the residual rows, then
  // MOE_FUSED_MAX_SLOTS slot rows per batch row)
  p.hid_slot_bytes = moe_slots >= 0 ? moe_slot_bytes_for(B) : HID_SLOT_BYTES;
  const int hid = p.mt <= FUSED_MAX_MT ? (moe_slots >= 0 ? MOE_HID_DEPTH : HID_DEPTH) * p.hid_slot_bytes : 0;
  const bool moe_ok = moe_slots < 0 || (moe_slots <= MOE_FUSED_MAX_SLOTS && (moe_slot_bytes == 4 || moe_slot_bytes == 2) &&
                                        p.mt <= FUSED_MAX_MT);
  p.nstages = (budget - hid) / p.stage_bytes;
  if (p.nstages > max_stages) p.nstages = max_stages;
  if (p.nstages > MAX_STAGES) p.nstages = MAX_STAGES;
  p.max_slab_cols = max_slab_pairs * 16;
  const int nblk = (max_slab_pairs + p.cb_pairs - 1) / p.cb_pairs;
  const int smem_logits = (B * p.max_slab_cols * 4 + 127) & ~127;
  const int ring = p.nstages * p.stage_bytes + hid;
  p.logits_in_smem = (nblk == 1 && smem_logits <= budget) ? 1 : 0;
  // owner phase: candidate buffer (capc keys + ids), sort buffer, sampler scratch, slab counts and bounds
  // composite buffer: the top-K selection writes up to K entries, the direct rank sort up to RANK_SORT_MAX
  p.sortP = next_pow2(K) > RANK_SORT_MAX ? next_pow2(K) : RANK_SORT_MAX;
  const int fixed_c = p.sortP * 8 + K * 8 + K * 4 + (2 * nslab + 8) * 4;
  // every published slot of a row, or K kept candidates plus one slab's rescan
  const int need_capc = nslab * SLAB_CAND > K + p.max_slab_cols ? nslab * SLAB_CAND : K + p.max_slab_cols;
  const int want_capc = ((need_capc > 2 * K ? need_capc : 2 * K) + 3) & ~3;
  int epi = p.logits_in_smem ? smem_logits : 0;
  const int phase_c = want_capc * 8 + fixed_c;
  if (phase_c > epi) epi = phase_c;
  p.smem_bytes = BAR_REGION + (ring > epi ? ring : epi);
  if (p.smem_bytes > max_smem) p.smem_bytes = max_smem;
  p.capc = ((p.smem_bytes - BAR_REGION - fixed_c) / 8) & ~3;
  if (p.capc > want_capc) p.capc = want_capc;
  p.ok = moe_ok && p.nstages >= 2 && p.capc >= 2 * K && p.capc >= need_capc && nslab <= MAX_SLABS &&
         BAR_REGION + ring <= max_smem &&
         (!p.logits_in_smem || BAR_REGION + smem_logits <= max_smem);
  return p;
}

cudaError_t prepare_gemv(int max_smem_optin, int* max_dynamic) {
  const void* fns[] = {reinterpret_cast<const void*>(lmhead_tail_kernel<1, 12, false>),
                       reinterpret_cast<const void*>(lmhead_tail_kernel<2, 6, false>),
                       reinterpret_cast<const void*>(lmhead_tail_kernel<4, 3, false>),
                       reinterpret_cast<const void*>(lmhead_tail_kernel<8, 1, false>),
                       reinterpret_cast<const void*>(lmhead_tail_kernel<1, 12, true>),
                       reinterpret_cast<const void*>(lmhead_tail_kernel<2, 6, true>)};
  int dyn = max_smem_optin;
  for (const void* fn : fns) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    const int d = max_smem_optin - static_cast<int>(fa.sharedSizeBytes);
    if (d < dyn) dyn = d;
  }
  for (const void* fn : fns) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    if (e != cudaSuccess) return e;
  }
  *max_dynamic = dyn;
  return cudaSuccess;
}

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t stream, bool pdl) {
  if (a.use_moe) {  // the producer step inside the activation warp: fused form only
    if (!a.fused) return cudaErrorInvalidValue;
    switch (a.mt) {
      case 1: return launch_t<1, 12, true>(a, stream, pdl);
      case 2: return launch_t<2, 6, true>(a, stream, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.mt) {
    case 1: return launch_t<1, 12, false>(a, stream, pdl);
    case 2: return launch_t<2, 6, false>(a, stream, pdl);
    case 4: return launch_t<4, 3, false>(a, stream, pdl);
    case 8: return launch_t<8, 1, false>(a, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tail
