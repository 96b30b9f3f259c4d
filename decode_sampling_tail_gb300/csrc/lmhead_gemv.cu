// lm_head projection with the stage-1 chunked top-k fused into its epilogue.
//
// Computes logit[b, v] = row_scale[b] * sum_h a[b, h] * W[h, v] for a batch of
// up to 64 rows ("GPT-OSS Tail Chunked Megakernel Kernel API Reference",
// parameters `lm_head_weight_t` and `deferred_rms`; `emit_logits` for the
// optional fp32 store), then keeps, per row and per vocabulary slab, the
// slab's top K by (logit desc, index asc) -- the first stage of the page's
// `chunked_topk` ("Background": global top-k computed locally over the full
// vocabulary).
//
// Structure (one persistent CTA per SM):
//   * The vocabulary is split into nslab contiguous slabs of 16-column pairs,
//     balanced to one pair.  A CTA owns one slab and streams its columns of
//     W = [H, V] (bf16, V contiguous) exactly once.
//   * One producer thread fills a ring of shared-memory stages with bulk
//     asynchronous copies (cp.async.bulk, mbarrier transaction counts); a
//     stage holds 16 rows of W for the CTA's current column block (each row
//     one contiguous segment, L2 evict-first) plus the 16-k slice of the packed
//     activations.  The first stages are requested before the dependency wait
//     on the RMSNorm kernel, since W does not depend on it.
//   * Eight consumer warps run mma.sync m16n8k16 (bf16 inputs, fp32
//     accumulation): the A operand is 8 batch rows' hi parts stacked on their
//     lo parts (the activation carried as two bf16 values), the B operand is a
//     16x8 W tile read with ldmatrix.trans (the row pitch is an odd multiple of
//     16 bytes, so the eight row addresses of a matrix hit distinct banks).
//     Hi and lo products are summed in the epilogue.
//   * Every column's k-reduction runs through the same sequence of mma
//     instructions wherever the column sits, so duplicated W columns give
//     bitwise-equal logits and exact ties survive into the top-k.
//   * After the last stage, the CTA keeps its slab's logits in shared memory
//     (or, when they do not fit, in a global staging buffer) and each warp
//     radix-selects the slab top-K of its rows, writing (key, index) pairs in
//     index order.
// Every wait is bounded (global timer); a wait that runs out raises the error
// flag, stops the producer, drains copies in flight and returns.
#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace tail {

namespace {

constexpr int MAX_STAGES = 8;
constexpr int BAR_REGION = 256;  // barriers and control words at the start of shared memory

__device__ __forceinline__ void consumer_barrier() {
  asm volatile("bar.sync 1, %0;" ::"r"(GEMV_CONSUMER_WARPS * 32) : "memory");
}

template <int MT, int PW>
__global__ void __launch_bounds__(GEMV_THREADS, 1) lmhead_gemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + MAX_STAGES);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + 2 * MAX_STAGES * 8);
  int* s_consumed_min = reinterpret_cast<int*>(smem + 2 * MAX_STAGES * 8 + 4);
  int* s_issued = reinterpret_cast<int*>(smem + 2 * MAX_STAGES * 8 + 8);
  uint8_t* ring = smem + BAR_REGION;
  const uint32_t ring_u32 = smem_u32(ring);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const int64_t pair_lo = slab_pair_lo(a.npairs, a.nslab, c);
  const int64_t pair_hi = slab_pair_lo(a.npairs, a.nslab, c + 1);
  const int slab_pairs = static_cast<int>(pair_hi - pair_lo);
  const int nblk = (slab_pairs + a.cb_pairs - 1) / a.cb_pairs;
  const int total = nblk * a.ksteps;
  const int NST = a.nstages;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, GEMV_CONSUMER_WARPS);
    }
    *s_abort = 0;
    *s_consumed_min = total;
    *s_issued = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == GEMV_CONSUMER_WARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      const uint32_t abytes = static_cast<uint32_t>(MT * APACK_TILE_BYTES);
      auto stage_of = [&](int it) { return ring_u32 + static_cast<uint32_t>((it % NST) * a.stage_bytes); };
      auto issue_w = [&](int it) {
        const int blk = it / a.ksteps, ks = it % a.ksteps;
        const int64_t bp0 = pair_lo + static_cast<int64_t>(blk) * a.cb_pairs;
        const int npb = static_cast<int>(min(static_cast<int64_t>(a.cb_pairs), pair_hi - bp0));
        const uint32_t row_bytes = static_cast<uint32_t>(npb) * 32u;
        const uint32_t bar = full0 + 8 * (it % NST);
        const uint32_t st = stage_of(it);
        mbar_arrive_expect_tx(bar, KSTEP * row_bytes + abytes);
        const uint16_t* src = a.w + static_cast<int64_t>(ks) * KSTEP * a.V + bp0 * 16;
#pragma unroll 4
        for (int r = 0; r < KSTEP; ++r)
          bulk_g2s(st + static_cast<uint32_t>(r * a.pitch), src + static_cast<int64_t>(r) * a.V, row_bytes,
                   bar, pol_w);
      };
      auto issue_a = [&](int it) {
        const int ks = it % a.ksteps;
        bulk_g2s(stage_of(it) + static_cast<uint32_t>(KSTEP * a.pitch),
                 a.apack + static_cast<int64_t>(ks) * abytes, abytes, full0 + 8 * (it % NST), pol_a);
      };
      const int npre = min(NST, total);
      for (int it = 0; it < npre; ++it) issue_w(it);
      pdl_wait();  // the packed activations come from the RMSNorm kernel
      for (int it = 0; it < npre; ++it) issue_a(it);
      int issued = npre;
      for (int it = npre; it < total; ++it) {
        if (*s_abort) break;
        const uint32_t par = static_cast<uint32_t>((it / NST) - 1) & 1u;
        if (!mbar_wait_bounded(empty0 + 8 * (it % NST), par, a.timeout_ns)) {
          raise_error(a.err, DEV_TIMEOUT_EMPTY);
          *s_abort = 1;
          break;
        }
        issue_w(it);
        issue_a(it);
        issued = it + 1;
      }
      *s_issued = issued;
    }
  } else {
    // ------------------------------------------------------------ consumers
    pdl_wait();  // row_scale is read and outputs are written only after the RMSNorm kernel
    const int g = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3;  // ldmatrix: this lane addresses a row of matrix mi
    const uint32_t lrow_off = static_cast<uint32_t>(((mi & 1) * 8 + (lane & 7)) * a.pitch + (mi >> 1) * 16);
    const int max_cols = a.max_slab_cols;
    float* slab_logits = reinterpret_cast<float*>(ring);
    bool ok = true;
    int it = 0;
    float acc[MT][PW][2][4];

    // hi + lo, row scale, optional fp32 store, and staging of one column block's logits
    auto block_epilogue = [&](int64_t bp0, int npb) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int r = m * MTILE_ROWS + g;
        if (r >= a.B) continue;
        const float sc = a.row_scale[r];
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
            if (a.logits_in_smem) {
              *reinterpret_cast<float2*>(slab_logits + r * max_cols + (col - pair_lo * 16)) = v;
            } else {
              *reinterpret_cast<float2*>(a.logits_scratch + static_cast<int64_t>(r) * a.V + col) = v;
            }
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

      for (int ks = 0; ks < a.ksteps; ++ks, ++it) {
        const int s = it % NST;
        const uint32_t par = static_cast<uint32_t>(it / NST) & 1u;
        if (!mbar_wait_bounded(full0 + 8 * s, par, a.timeout_ns)) {
          raise_error(a.err, DEV_TIMEOUT_FULL);
          *s_abort = 1;
          ok = false;
          break;
        }
        const uint32_t st = ring_u32 + static_cast<uint32_t>(s * a.stage_bytes);
        const uint32_t abase = st + static_cast<uint32_t>(KSTEP * a.pitch) + lane * 16;
        uint32_t af[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m) lds128(abase + m * APACK_TILE_BYTES, af[m][0], af[m][1], af[m][2], af[m][3]);
#pragma unroll
        for (int q = 0; q < PW; ++q) {
          const int pr = warp + GEMV_CONSUMER_WARPS * q;
          if (pr < npb) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(st + lrow_off + static_cast<uint32_t>(pr * 32), b0, b1, b2, b3);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              mma_bf16_16816(acc[m][q][0], af[m][0], af[m][1], af[m][2], af[m][3], b0, b1);
              mma_bf16_16816(acc[m][q][1], af[m][0], af[m][1], af[m][2], af[m][3], b2, b3);
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

    // Every consumer warp reaches both barriers below whatever happened above,
    // and the abort decision is read once, after the first of them.
    consumer_barrier();  // all stages consumed: the ring may now hold the slab logits
    const bool aborted = *s_abort != 0;
    if (!aborted && a.logits_in_smem) block_epilogue(last_bp0, last_npb);
    __threadfence_block();
    consumer_barrier();

    // ---------------- stage-1 top-k of each (row, slab)
    if (!aborted) {
      const int n = slab_pairs * 16;
      const int want = min(a.K, n);
      const int64_t vbase = pair_lo * 16;
      uint8_t* hist_base = a.logits_in_smem
                               ? ring + ((static_cast<size_t>(a.B) * max_cols * 4 + 127) & ~size_t(127))
                               : ring;
      uint32_t* hist = reinterpret_cast<uint32_t*>(hist_base) + warp * HIST_BINS;
      for (int r = warp; r < a.B; r += GEMV_CONSUMER_WARPS) {
        const float* src = a.logits_in_smem ? slab_logits + r * max_cols
                                            : a.logits_scratch + static_cast<int64_t>(r) * a.V + vbase;
        auto get = [&](int i) { return float_key(src[i]); };
        const int64_t obase = (static_cast<int64_t>(r) * a.nslab + c) * a.K;
        auto emit = [&](int pos, int i, uint32_t k) {
          a.cand_key[obase + pos] = k;
          a.cand_idx[obase + pos] = static_cast<int32_t>(vbase + i);
        };
        Threshold th;
        if (want == n) {
          th.key = 0u;
          th.take_eq = -1;  // the whole slab
        } else {
          th = warp_select(get, n, want, hist);
        }
        warp_compact(get, n, th, emit);
        __syncwarp();
      }
    }
  }

  // ---------------- drain: no copy may still be landing when the CTA leaves
  __syncthreads();
  if (warp == GEMV_CONSUMER_WARPS && lane == 0) {
    const int issued = *s_issued;
    for (int it = *s_consumed_min; it < issued; ++it) {
      const uint32_t par = static_cast<uint32_t>(it / NST) & 1u;
      if (!mbar_wait_bounded(full0 + 8 * (it % NST), par, DEFAULT_TIMEOUT_NS)) {
        raise_error(a.err, DEV_TIMEOUT_DRAIN);
        break;
      }
    }
  }
  pdl_launch_dependents();
}

template <int MT, int PW>
cudaError_t launch_t(const GemvArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nslab);
  cfg.blockDim = dim3(GEMV_THREADS);
  cfg.dynamicSmemBytes = a.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lmhead_gemv_kernel<MT, PW>, a);
}

int mt_template(int B) {
  const int mt = (B + MTILE_ROWS - 1) / MTILE_ROWS;
  return mt <= 1 ? 1 : mt <= 2 ? 2 : mt <= 4 ? 4 : 8;
}

}  // namespace

GemvPlan plan_gemv(int B, int H, int V, int K, int nslab, int max_smem) {
  (void)H;
  (void)K;
  GemvPlan p = {};
  p.mt = mt_template(B);
  p.pw = p.mt == 1 ? 12 : p.mt == 2 ? 6 : p.mt == 4 ? 3 : 1;
  p.cb_pairs = GEMV_CONSUMER_WARPS * p.pw;
  const int64_t npairs = V / 16;
  const int max_slab_pairs = static_cast<int>((npairs + nslab - 1) / nslab);
  const int cb_eff = max_slab_pairs < p.cb_pairs ? max_slab_pairs : p.cb_pairs;
  p.pitch = cb_eff * 32 + 16;  // odd multiple of 16 bytes: conflict-free ldmatrix rows
  p.stage_bytes = ((KSTEP * p.pitch + p.mt * APACK_TILE_BYTES) + 127) & ~127;
  const int budget = max_smem - BAR_REGION;
  p.nstages = budget / p.stage_bytes;
  if (p.nstages > MAX_STAGES) p.nstages = MAX_STAGES;
  p.max_slab_cols = max_slab_pairs * 16;
  const int nblk = (max_slab_pairs + p.cb_pairs - 1) / p.cb_pairs;
  const int hist_bytes = GEMV_CONSUMER_WARPS * HIST_BINS * 4;
  const int smem_logits = ((B * p.max_slab_cols * 4 + 127) & ~127) + hist_bytes;
  const int ring = p.nstages * p.stage_bytes;
  p.logits_in_smem = (nblk == 1 && smem_logits <= budget) ? 1 : 0;
  const int epi = p.logits_in_smem ? smem_logits : hist_bytes;
  p.smem_bytes = BAR_REGION + (ring > epi ? ring : epi);
  p.ok = p.nstages >= 2 && p.smem_bytes <= max_smem;
  return p;
}

cudaError_t prepare_gemv(int max_smem) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(lmhead_gemv_kernel<1, 12>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem)))
    return e;
  if ((e = cudaFuncSetAttribute(lmhead_gemv_kernel<2, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem)))
    return e;
  if ((e = cudaFuncSetAttribute(lmhead_gemv_kernel<4, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem)))
    return e;
  return cudaFuncSetAttribute(lmhead_gemv_kernel<8, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t stream) {
  switch (a.mt) {
    case 1: return launch_t<1, 12>(a, stream);
    case 2: return launch_t<2, 6>(a, stream);
    case 4: return launch_t<4, 3>(a, stream);
    case 8: return launch_t<8, 1>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tail
