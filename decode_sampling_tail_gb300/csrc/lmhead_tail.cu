// The lm_head projection and everything after it -- the global top-k and the
// sampler -- in one cooperative launch.
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
// Top-k and sampler, in three phases separated by a grid barrier (the launch
// is cooperative, so every CTA is resident; each wait is bounded):
//   A  per (row, slab): publish the 4 largest of the 32 lane maxima of the
//      slab's logits.  They are 4 distinct elements of the row.
//   B  per row: x = the K-th largest of the nslab * 4 published keys.  At
//      least K elements of the row are >= x, so the row's K-th largest key is
//      >= x and every global top-K element is >= x.  Each CTA emits its slab
//      elements >= x (its exact slab top-K if more than K pass) -- a handful
//      per slab instead of K.
//   C  CTA r gathers row r's candidates, keeps the top K (ties at the
//      boundary settled by index), sorts them, writes the top-k outputs and
//      runs the sampler on warp 0.
#include "common.cuh"
#include "internal.h"
#include "sampler.cuh"
#include "select.cuh"

namespace tail {

namespace {

constexpr int MAX_STAGES = 8;
constexpr int BAR_REGION = 256;  // ring barriers and control words at the start of shared memory
constexpr int PUB = TAIL_PUB_PER_SLAB;
constexpr int NPUB_L = (PUB * MAX_SLABS + 31) / 32;  // published keys per lane in phase B
constexpr int GATHER_PT = 4;                           // candidate loads in flight per thread in phase C

__device__ __forceinline__ void consumer_barrier() {
  asm volatile("bar.sync 1, %0;" ::"r"(GEMV_CONSUMER_WARPS * 32) : "memory");
}

// Grid-wide barrier over the co-resident CTAs of a cooperative launch.  The
// counter only grows (each barrier adds gridDim.x), so generations never
// collide.  Returns false, after raising the error flag, if the wait ran out.
__device__ __forceinline__ bool grid_barrier(unsigned long long* counter, uint64_t limit_ns, int* err,
                                             volatile int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned long long nb = gridDim.x;
    const unsigned long long old = atomicAdd(counter, 1ull);
    const unsigned long long target = (old / nb + 1) * nb;
    int ok = 1;
    const uint64_t t0 = global_timer_ns();
    while (true) {
      unsigned long long cur;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(cur) : "l"(counter) : "memory");
      if (cur >= target) break;
      if (global_timer_ns() - t0 > limit_ns) {
        raise_error(err, DEV_TIMEOUT_BARRIER);
        ok = 0;
        break;
      }
    }
    __threadfence();
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

template <int MT, int PW>
__global__ void __launch_bounds__(GEMV_THREADS, 1) lmhead_tail_kernel(const GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t s_red[64];
  __shared__ uint32_t s_list[SEL_BLOCK_BUCKET_MAX];
  __shared__ uint32_t s_misc[4];
  __shared__ int s_rows[1];
  __shared__ int s_flag;
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
  const int KPB = a.kpb;                       // k-steps (16 rows each) per ring stage
  const int spb = (a.ksteps + KPB - 1) / KPB;  // ring stages per column block
  const int total = nblk * spb;
  const int NST = a.nstages;
  const int max_cols = a.max_slab_cols;
  float* slab_logits = reinterpret_cast<float*>(ring);

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
    // ================================================================ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      const uint32_t abytes = static_cast<uint32_t>(MT * APACK_TILE_BYTES);
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
      pdl_wait();  // the packed activations come from the RMSNorm kernel
      for (int it = 0; it < npre; ++it)
        if (it != a.drop_iter) issue_a(it);
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
          issue_a(it);
        }
        issued = it + 1;
      }
      *s_issued = issued;
    }
  } else {
    // ================================================================ consumers
    pdl_wait();  // row_scale is read and outputs are written only after the RMSNorm kernel
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
    const bool aborted_c = *s_abort != 0;
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
  uint32_t* wlist = reinterpret_cast<uint32_t*>(
                        ring + (a.logits_in_smem ? ((static_cast<size_t>(a.B) * max_cols * 4 + 127) & ~size_t(127)) : 0)) +
                    warp * SEL_BUCKET_MAX;
  auto load_row_keys = [&](int r, uint32_t (&k)[SEL_NPL]) {
    const float* src = a.logits_in_smem ? slab_logits + r * max_cols
                                        : a.logits_scratch + static_cast<int64_t>(r) * a.V + vbase;
#pragma unroll
    for (int i = 0; i < SEL_NPL; ++i) {
      const int pos = i * 32 + lane;
      k[i] = pos < n ? float_key(src[pos]) : 0u;
    }
  };

  // ================================================================ phase A: publish lane maxima
  if (!aborted && warp < GEMV_CONSUMER_WARPS) {
    for (int r = warp; r < a.B; r += GEMV_CONSUMER_WARPS) {
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
      uint32_t lm = max(max(m0, m1), max(m2, m3));
      uint32_t* dst = a.pub + (static_cast<int64_t>(r) * a.nslab + c) * PUB;
#pragma unroll
      for (int j = 0; j < PUB; ++j) {
        const uint32_t best = __reduce_max_sync(0xffffffffu, lm);
        const uint32_t who = __ballot_sync(0xffffffffu, lm == best);
        if (lane == 0) dst[j] = best;
        if (lane == __ffs(who) - 1) lm = 0u;  // each lane maximum is published once
      }
    }
  }
  const bool ok1 = grid_barrier(a.bar, a.timeout_ns, a.err, &s_flag);

  // ================================================================ phase B: emit the slab's elements >= x
  if (!aborted && ok1 && warp < GEMV_CONSUMER_WARPS) {
    const int npub = a.nslab * PUB;
    for (int r = warp; r < a.B; r += GEMV_CONSUMER_WARPS) {
      uint32_t x = 0u;  // below every key: no bound when too few keys are published
      if (npub >= a.K) {
        uint32_t pk[NPUB_L];
        const uint32_t* srcp = a.pub + static_cast<int64_t>(r) * npub;
#pragma unroll
        for (int i = 0; i < NPUB_L; ++i) {
          const int pos = i * 32 + lane;
          pk[i] = pos < npub ? __ldcg(srcp + pos) : 0u;
        }
        x = warp_bound16_span_regs(pk, a.K);
      }
      uint32_t k[SEL_NPL];
      load_row_keys(r, k);
      uint32_t mine = 0;
#pragma unroll
      for (int i = 0; i < SEL_NPL; ++i) mine += (i * 32 + lane < n && k[i] >= x) ? 1u : 0u;
      const uint32_t tot = __reduce_add_sync(0xffffffffu, mine);
      // reserve room in the row's packed candidate array, emit, then count this slab as arrived
      const uint32_t take = tot <= static_cast<uint32_t>(a.K) ? tot : static_cast<uint32_t>(a.K);
      uint32_t off = 0;
      if (lane == 0) off = static_cast<uint32_t>(atomicAdd(a.row_sync + r, static_cast<unsigned long long>(take)));
      off = __shfl_sync(0xffffffffu, off, 0);
      const int64_t obase = static_cast<int64_t>(r) * a.nslab * a.K + off;
      if (tot <= static_cast<uint32_t>(a.K)) {
        uint32_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        uint32_t o = incl - mine;
#pragma unroll
        for (int i = 0; i < SEL_NPL; ++i) {
          const int pos = i * 32 + lane;
          if (pos < n && k[i] >= x) {
            a.cand_key[obase + o] = k[i];
            a.cand_idx[obase + o] = static_cast<int32_t>(vbase + pos);
            ++o;
          }
        }
      } else {
        // more than K pass: the slab's exact top-K (ties by index) covers its share of the global top-K
        const Threshold th = warp_select_regs(k, a.K, wlist);
        warp_compact_regs(k, n, th, [&](int pos, int i, uint32_t kv) {
          a.cand_key[obase + pos] = kv;
          a.cand_idx[obase + pos] = static_cast<int32_t>(vbase + i);
        });
      }
      // the warp barrier orders every lane's candidate stores before lane 0's release of the arrival
      __syncwarp();
      if (lane == 0)
        asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(a.row_sync + r), "l"(1ull << 32) : "memory");
    }
  }

  // ================================================================ phase C: final top-K, sort, sampler
  if (!aborted && ok1) {
    const int nt = blockDim.x, nw = nt >> 5;
    uint32_t* keys = reinterpret_cast<uint32_t*>(ring);
    int32_t* idx = reinterpret_cast<int32_t*>(keys + a.capc);
    uint64_t* comp = reinterpret_cast<uint64_t*>(idx + a.capc);
    uint64_t* sorted = comp + a.sortP;
    float* ebuf = reinterpret_cast<float*>(sorted + a.K);
    // keeps the top K of the m > K candidates, in place
    auto fold = [&](int m) {
      for (int j = tid; j < a.sortP; j += nt) comp[j] = 0ull;
      __syncthreads();
      block_top_composites(keys, idx, m, a.K, comp, s_red, s_list, s_misc);
      for (int j = tid; j < a.K; j += nt) {
        keys[j] = composite_key(comp[j]);
        idx[j] = composite_idx(comp[j]);
      }
      __syncthreads();
      return a.K;
    };
    for (int row = c; row < a.B; row += a.nslab) {
      SampleParams prm = {};
      if (a.params != nullptr) prm = load_sample_params(a.params + static_cast<int64_t>(row) * a.ncols, a.ncols);
      // wait (bounded) until every slab has emitted its candidates of this row
      if (tid == 0) {
        unsigned long long v = 0;
        const uint64_t t0 = global_timer_ns();
        while (true) {
          asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.row_sync + row) : "memory");
          if ((v >> 32) >= static_cast<unsigned long long>(a.nslab)) break;
          if (global_timer_ns() - t0 > a.timeout_ns) {
            raise_error(a.err, DEV_TIMEOUT_BARRIER);
            v = ~0ull;
            break;
          }
        }
        s_rows[0] = v == ~0ull ? -1 : static_cast<int>(v & 0xFFFFFFFFull);
      }
      __syncthreads();
      const int total_c = s_rows[0];
      if (total_c < 0) break;  // uniform: a slab never arrived (the error flag is raised)
      const int64_t cbase = static_cast<int64_t>(row) * a.nslab * a.K;
      // gather the packed candidates; when they exceed the buffer, fold it to its top K between runs
      int ncand = 0;
      for (int base = 0; base < total_c;) {
        const int take = min(total_c - base, a.capc - ncand);
        for (int i0 = 0; i0 < take; i0 += GATHER_PT * nt) {  // loads first, then stores
          uint32_t kr[GATHER_PT];
          int32_t ir[GATHER_PT];
#pragma unroll
          for (int q = 0; q < GATHER_PT; ++q) {
            const int i = i0 + q * nt + tid;
            kr[q] = i < take ? __ldcg(a.cand_key + cbase + base + i) : 0u;
            ir[q] = i < take ? __ldcg(a.cand_idx + cbase + base + i) : 0;
          }
#pragma unroll
          for (int q = 0; q < GATHER_PT; ++q) {
            const int i = i0 + q * nt + tid;
            if (i < take) {
              keys[ncand + i] = kr[q];
              idx[ncand + i] = ir[q];
            }
          }
        }
        ncand += take;
        base += take;
        __syncthreads();
        if (base < total_c) ncand = fold(ncand);
      }
      if (tid == 0) a.row_sync[row] = 0ull;  // ready for the next run
      const int want = min(a.K, ncand);
      // candidates to rank: all of them when few, else the top `want` found by a selection
      int nr = ncand;
      if (ncand <= RANK_SORT_MAX) {
        for (int j = tid; j < ncand; j += nt) comp[j] = composite(keys[j], idx[j]);
        __syncthreads();
      } else {
        block_top_composites(keys, idx, ncand, want, comp, s_red, s_list, s_misc);
        nr = want;
      }
      // rank sort: the composites are distinct, so rank(i) = #{j : comp[j] > comp[i]} is the
      // position of candidate i in (value desc, index asc) order
      for (int i = tid; i < nr; i += nt) {
        const uint64_t ci = comp[i];
        int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
        int j = 0;
        const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(comp);  // comp is 16-byte aligned
        for (; j + 4 <= nr; j += 4) {
          const ulonglong2 p = c2[j >> 1], q = c2[(j >> 1) + 1];
          r0 += p.x > ci;
          r1 += p.y > ci;
          r2 += q.x > ci;
          r3 += q.y > ci;
        }
        for (; j < nr; ++j) r0 += comp[j] > ci;
        const int rank = (r0 + r1) + (r2 + r3);
        if (rank < want) sorted[rank] = ci;
      }
      __syncthreads();
      for (int j = tid; j < want; j += nt) {
        a.topk_val[static_cast<int64_t>(row) * a.topk_ld + j] = key_float(composite_key(sorted[j]));
        a.topk_idx[static_cast<int64_t>(row) * a.topk_ld + j] = composite_idx(sorted[j]);
      }
      if (a.params != nullptr && a.tokens != nullptr) {  // every thread takes part in the draw
        const int32_t tok = sample_sorted_row(prm, sorted, want, ebuf,
                                              reinterpret_cast<float*>(s_red));
        if (tid == 0) a.tokens[row] = tok;
      }
      __syncthreads();
    }
  }
  pdl_launch_dependents();
}

template <int MT, int PW>
cudaError_t launch_t(const GemvArgs& a, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nslab);
  cfg.blockDim = dim3(GEMV_THREADS);
  cfg.dynamicSmemBytes = a.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, lmhead_tail_kernel<MT, PW>, a);
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

GemvPlan plan_gemv(int B, int H, int V, int K, int nslab, int max_smem, int kpb, int max_stages) {
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
  p.nstages = budget / p.stage_bytes;
  if (p.nstages > max_stages) p.nstages = max_stages;
  if (p.nstages > MAX_STAGES) p.nstages = MAX_STAGES;
  p.max_slab_cols = max_slab_pairs * 16;
  const int nblk = (max_slab_pairs + p.cb_pairs - 1) / p.cb_pairs;
  const int list_bytes = GEMV_CONSUMER_WARPS * SEL_BUCKET_MAX * 4;
  const int smem_logits = ((B * p.max_slab_cols * 4 + 127) & ~127) + list_bytes;
  const int ring = p.nstages * p.stage_bytes;
  p.logits_in_smem = (nblk == 1 && smem_logits <= budget) ? 1 : 0;
  // phase C: candidate buffer (capc keys + ids), sort buffer, sampler scratch, slab counts and offsets
  // composite buffer: the top-K selection writes up to K entries, the direct rank sort up to RANK_SORT_MAX
  p.sortP = next_pow2(K) > RANK_SORT_MAX ? next_pow2(K) : RANK_SORT_MAX;
  const int fixed_c = p.sortP * 8 + K * 8 + K * 4 + (2 * nslab + 8) * 4;
  const int want_capc = nslab * K < PHASE_C_CAP ? ((nslab * K + 3) & ~3) : PHASE_C_CAP;
  int epi = p.logits_in_smem ? smem_logits : list_bytes;
  const int phase_c = want_capc * 8 + fixed_c;
  if (phase_c > epi) epi = phase_c;
  p.smem_bytes = BAR_REGION + (ring > epi ? ring : epi);
  if (p.smem_bytes > max_smem) p.smem_bytes = max_smem;
  p.capc = ((p.smem_bytes - BAR_REGION - fixed_c) / 8) & ~3;
  if (p.capc > PHASE_C_CAP) p.capc = PHASE_C_CAP;
  p.ok = p.nstages >= 2 && p.capc >= 2 * K && BAR_REGION + ring <= max_smem &&
         (!p.logits_in_smem || BAR_REGION + smem_logits <= max_smem);
  return p;
}

cudaError_t prepare_gemv(int max_smem_optin, int* max_dynamic) {
  const void* fns[] = {reinterpret_cast<const void*>(lmhead_tail_kernel<1, 12>),
                       reinterpret_cast<const void*>(lmhead_tail_kernel<2, 6>),
                       reinterpret_cast<const void*>(lmhead_tail_kernel<4, 3>),
                       reinterpret_cast<const void*>(lmhead_tail_kernel<8, 1>)};
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
  switch (a.mt) {
    case 1: return launch_t<1, 12>(a, stream, pdl);
    case 2: return launch_t<2, 6>(a, stream, pdl);
    case 4: return launch_t<4, 3>(a, stream, pdl);
    case 8: return launch_t<8, 1>(a, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tail
