// Tensor-core lm_head of the tail for batches above 8 rows ("GPT-OSS Tail
// Chunked Megakernel Kernel API Reference", parameters `lm_head_weight_t`,
// `deferred_rms`, `emit_logits`, and section "Background": a stage-1 top-k
// per vocabulary chunk feeding one global top-k).
//
// logit[b][v] = row_scale[b] * sum_h (hi[b][h] + lo[b][h]) * W[h][v], with
// hi + lo the two-bf16 split of the RMSNorm output, on tcgen05 tensor cores
// with fp32 accumulation in tensor memory.
//
// Persistent kernel, one CTA per SM, 7 warps:
//   warp 0     weight producer: per ring stage the 64 x N weight slice
//              (N / 64 boxes of 64 x 64, 128-byte swizzle; N = 192 columns
//              when hi and lo share a tile, else 256), requested up to NW
//              stages ahead: one TMA tensor-tile load per box, or, from the
//              prepared weight (weight_pack.cu), one bulk copy per stage.
//   warp 6     activation producer: the matching 64-wide k slice of the
//              activation tile (hi and lo: two 128 x 64 tiles, or one tile
//              holding both when the batch fits in 64 rows), NA stages ahead,
//              by one bulk copy of the split kernel's pre-swizzled image: the
//              copy engine then spends its per-row request rate on the
//              weight alone.
//   warp 1     tensor-memory owner and MMA issuer: M = 128, N, K = 16
//              per instruction, A K-major, B (the weight, V contiguous)
//              MN-major; two accumulators of 256 columns so the epilogue of
//              one tile overlaps the MMAs of the next.
//   warps 2-5  epilogue, one batch row per thread (tensor-memory lane): row
//              scale, the fp32 logits (32 x 32 blocks staged in shared
//              memory and written by TMA tensor stores), and the tile's top
//              TC_LIST candidates (value desc, index asc) for the merge.
//              When hi and lo share a tile, the two warps holding a row's
//              hi and lo parts each take half of the columns.
// Tiles are (column tile n, m-block m) pairs taken round robin by the CTAs,
// m varying fastest, so the CTAs that share a weight tile run it together and
// the weight is read from HBM once.
//
// Every wait is bounded (the error flag is raised and the CTA winds down:
// no copy or MMA is left in flight and the tensor memory is released).
#include "common.cuh"
#include "internal.h"
#include "select.cuh"
#include "tc_common.cuh"
#include "tc_internal.h"

namespace tail {

namespace {

constexpr int TC_THREADS = 224;  // warp 0 weight producer, 1 MMA, 2-5 epilogue, 6 activation producer
constexpr uint32_t TC_ACC_COLS = 256;               // tensor-memory columns per accumulator
constexpr uint32_t TC_TMEM_COLS = 2 * TC_ACC_COLS;  // two accumulators
constexpr uint32_t W_BOX_BYTES = 64 * 64 * 2;
constexpr uint32_t A_BOX_BYTES = 128 * 64 * 2;
constexpr int XHALF_PITCH = 17;                     // floats per row of a half-chunk hand-over (16 + 1)
constexpr int XHALF = 64 * XHALF_PITCH;              // floats of one direction's hand-over (64 rows)

// Shared memory: the activation ring (NA stages), the weight ring (NW stages), the
// stacked hi/lo exchange, the logits store boxes and the barriers.  The two
// rings are separate so that the weight, streamed from HBM, can be requested
// further ahead than the L2-resident activations.
template <bool STACKED>
struct TcGeom {
  static constexpr int N = STACKED ? TC_N_STACKED : TC_N_SEPARATE;  // vocabulary columns of a tile
  static_assert(N % 64 == 0 && N <= static_cast<int>(TC_ACC_COLS), "tile width: whole 64-column boxes, one accumulator");
  static constexpr int CHUNKS = N / 32;  // 32-column blocks of the epilogue
  static constexpr int WBOX = N / 64;    // 64-column weight boxes per stage
  static constexpr uint32_t A_BYTES = STACKED ? A_BOX_BYTES : 2 * A_BOX_BYTES;  // one activation stage
  static constexpr uint32_t W_BYTES = WBOX * W_BOX_BYTES;                     // one weight stage
  static constexpr int TBUF_N = STACKED ? 1 : 2;  // 32 x 32 fp32 store boxes per epilogue warp
  static constexpr uint32_t TBUF_BYTES = 4 * TBUF_N * 4096;
  static constexpr uint32_t XBUF_BYTES = STACKED ? (2 * XHALF * 4 + 1023) / 1024 * 1024 : 0;
  static_assert(!STACKED || 64 * 2 * TC_LIST * 4 <= 2 * XHALF * 4, "the list hand-over fits the exchange buffer");
  static constexpr uint32_t CTL_BYTES = 256;
  static constexpr int NA = 3;
  static constexpr int NW_FIT =
      static_cast<int>((227 * 1024 - 1024 - XBUF_BYTES - TBUF_BYTES - CTL_BYTES - NA * A_BYTES) / W_BYTES);
  static constexpr int NW = NW_FIT < 8 ? NW_FIT : 8;
  static constexpr uint32_t SMEM = 1024 /* alignment slack */ + NA * A_BYTES + NW * W_BYTES + XBUF_BYTES +
                                   TBUF_BYTES + CTL_BYTES;
};

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void fail(int* err, int code, volatile int* abort_flag) {
  if (!*abort_flag) raise_error(err, code);
  *abort_flag = 1;
}

// A tile's candidate list per row is kept as TC_LIST composites in registers: key
// in the high word, ~column in the low word (0 for an empty slot), in descending
// order -- (value desc, index asc) -- the layout the merge reads.  It is updated
// per chunk with fixed comparator networks (no data-dependent loops).

// a >= b afterwards
__device__ __forceinline__ void cas_desc(uint64_t& a, uint64_t& b) {
  const uint64_t x = a, y = b;
  a = x > y ? x : y;
  b = x > y ? y : x;
}

// v[O, O + 8) into descending order (bitonic network, 24 comparators)
template <int O, int N>
__device__ __forceinline__ void sort8_desc(uint64_t (&v)[N]) {
#pragma unroll
  for (int k = 2; k <= 8; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int l = i ^ j;
        if (l > i) {
          if ((i & k) == 0) cas_desc(v[O + i], v[O + l]);
          else cas_desc(v[O + l], v[O + i]);
        }
      }
}

// t[0, 8) bitonic -> descending (half-cleaners, 12 comparators)
__device__ __forceinline__ void bitonic_merge8_desc(uint64_t (&t)[TC_LIST]) {
#pragma unroll
  for (int j = 4; j > 0; j >>= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i ^ j) > i) cas_desc(t[i], t[i ^ j]);
}

// a = the top 8 of a and b (both descending): the element-wise maximum of a and reversed b holds
// them as a bitonic sequence
__device__ __forceinline__ void merge_top8(uint64_t (&a)[TC_LIST], const uint64_t (&b)[TC_LIST]) {
#pragma unroll
  for (int i = 0; i < TC_LIST; ++i) a[i] = a[i] > b[TC_LIST - 1 - i] ? a[i] : b[TC_LIST - 1 - i];
  bitonic_merge8_desc(a);
}

// out = the top 8 of c[O, O + 16), descending (c is reordered)
template <int O, int N>
__device__ __forceinline__ void top8_of16(uint64_t (&c)[N], uint64_t (&out)[TC_LIST]) {
  sort8_desc<O>(c);
  sort8_desc<O + 8>(c);
#pragma unroll
  for (int i = 0; i < TC_LIST; ++i) out[i] = c[O + i] > c[O + 15 - i] ? c[O + i] : c[O + 15 - i];
  bitonic_merge8_desc(out);
}

__device__ __forceinline__ uint64_t cand_composite(bool ok, float v, int col) {
  return ok ? (static_cast<uint64_t>(float_key(v)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(col)) : 0ull;
}

// Inserts composite c into the descending list L.  Every slot takes its new entry from the old list in
// parallel (no serial bubble chain); a composite at or below the last entry leaves L unchanged.
__device__ __forceinline__ void list_push(uint64_t (&L)[TC_LIST], uint64_t c) {
  bool gt[TC_LIST];
#pragma unroll
  for (int i = 0; i < TC_LIST; ++i) gt[i] = c > L[i];
#pragma unroll
  for (int i = TC_LIST - 1; i > 0; --i) L[i] = gt[i - 1] ? L[i - 1] : (gt[i] ? c : L[i]);
  L[0] = gt[0] ? c : L[0];
}

// Pushes the chunk columns marked in `cand` (bit j: column col0 + j, its value at float j of this
// lane's 128-byte-swizzled row of the store box), each lane its own: once the list has filled, a
// chunk holds few columns above its last entry, and only those can enter.
__device__ __forceinline__ void push_candidates(uint64_t (&L)[TC_LIST], uint32_t cand, uint32_t box, int col0) {
  const int lane = threadIdx.x & 31;
  const uint32_t row = box + static_cast<uint32_t>(lane * 128);
  while (cand != 0u) {
    const int j = __ffs(cand) - 1;
    cand &= cand - 1u;
    float val;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(val) : "r"(row + ((((j >> 2) ^ (lane & 7)) << 4) | ((j & 3) << 2))));
    list_push(L, cand_composite(true, val, col0 + j));
  }
}

template <bool STACKED>
__global__ void __launch_bounds__(TC_THREADS, 1)
    lmhead_tc_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapL,
                     const TcArgs a) {
  using G = TcGeom<STACKED>;
  constexpr int NA = G::NA, NW = G::NW;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base_u = (raw_u + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base_u - raw_u);
  const uint32_t ringA_u = base_u;
  const uint32_t ringW_u = base_u + NA * G::A_BYTES;
  const uint32_t rings = NA * G::A_BYTES + NW * G::W_BYTES;
  float* xbuf = reinterpret_cast<float*>(sm + rings);
  float* tbuf = reinterpret_cast<float*>(sm + rings + G::XBUF_BYTES);
  uint8_t* ctl = sm + rings + G::XBUF_BYTES + G::TBUF_BYTES;
  const uint32_t ctl_u = base_u + rings + G::XBUF_BYTES + G::TBUF_BYTES;
  auto fullA_bar = [&](int s) { return ctl_u + 8u * s; };
  auto emptyA_bar = [&](int s) { return ctl_u + 8u * (NA + s); };
  auto fullW_bar = [&](int s) { return ctl_u + 8u * (2 * NA + s); };
  auto emptyW_bar = [&](int s) { return ctl_u + 8u * (2 * NA + NW + s); };
  auto tfull_bar = [&](int acc) { return ctl_u + 8u * (2 * NA + 2 * NW + acc); };
  auto tempty_bar = [&](int acc) { return ctl_u + 8u * (2 * NA + 2 * NW + 2 + acc); };
  const uint32_t done_bar = ctl_u + 8u * (2 * NA + 2 * NW + 4);
  int* cw = reinterpret_cast<int*>(ctl + 8 * (2 * NA + 2 * NW + 5));
  volatile int* s_abort = cw;
  volatile int* s_go = cw + 1;  // [2]: epilogue go flags, by tile parity
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(cw + 3);
  int* s_issued_w = cw + 4;
  int* s_issued_a = cw + 5;
  int* s_consumed = cw + 6;
  static_assert(8 * (2 * G::NA + 2 * G::NW + 5) + 7 * 4 <= G::CTL_BYTES, "barrier region");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = a.ntn * a.n_mb;
  const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  const int total_it = my_tiles * a.kblocks;

  if (tid == 0) {
    for (int s = 0; s < NA; ++s) {
      mbar_init(fullA_bar(s), 1);
      mbar_init(emptyA_bar(s), 1);
    }
    for (int s = 0; s < NW; ++s) {
      mbar_init(fullW_bar(s), 1);
      mbar_init(emptyW_bar(s), 1);
    }
    for (int acc = 0; acc < 2; ++acc) {
      mbar_init(tfull_bar(acc), 1);
      mbar_init(tempty_bar(acc), 4);
    }
    mbar_init(done_bar, 1);
    *s_abort = 0;
    s_go[0] = 0;
    s_go[1] = 0;
    *s_issued_w = 0;
    *s_issued_a = 0;
    *s_consumed = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), TC_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  auto tile_coords = [&](int tile_i, int& n, int& m) {
    const int t = static_cast<int>(blockIdx.x) + tile_i * static_cast<int>(gridDim.x);
    n = t / a.n_mb;
    m = t - n * a.n_mb;
  };

  if (warp == 0) {
    // ================================================================ weight producer
    if (lane == 0) {
      const bool packed = a.w_packed != nullptr;
      if (!packed) tma_prefetch_map(&mapW);
      const uint64_t pol_w = policy_evict_first();
      auto issue_w = [&](int it) {
        int n, m;
        tile_coords(it / a.kblocks, n, m);
        const int kb = it % a.kblocks;
        const int s = it % NW;
        const uint32_t st = ringW_u + static_cast<uint32_t>(s) * G::W_BYTES;
        if (packed) {
          // the stage's boxes are adjacent blocks of the prepared weight: one bulk copy
          const int g0 = n * G::WBOX;
          const int nbox = min(G::WBOX, a.w_groups - g0);  // >= 1: the tile starts below V
          const uint32_t bytes = static_cast<uint32_t>(nbox) * W_BOX_BYTES;
          mbar_arrive_expect_tx(fullW_bar(s), bytes);
          bulk_g2s(st, a.w_packed + (static_cast<int64_t>(kb) * a.w_groups + g0) * W_BOX_BYTES, bytes, fullW_bar(s),
                   pol_w);
          return;
        }
        const int x0 = n * G::N;
        int nbox = 0;
#pragma unroll
        for (int j = 0; j < G::WBOX; ++j) nbox += (x0 + 64 * j < a.V) ? 1 : 0;  // >= 1: x0 < V
        mbar_arrive_expect_tx(fullW_bar(s), static_cast<uint32_t>(nbox) * W_BOX_BYTES);
        for (int j = 0; j < nbox; ++j)
          tma_load_2d(st + j * W_BOX_BYTES, &mapW, x0 + 64 * j, kb * TC_KB, fullW_bar(s), pol_w);
      };
      // stages in flight: the whole ring unless fewer are asked for (stage it is issued once stage
      // it - ahead has been consumed, which also frees its slot, as ahead <= NW)
      const int ahead = (a.w_ahead > 0 && a.w_ahead < NW) ? a.w_ahead : NW;
      // the weight does not depend on the split kernel: the first stages go out before its wait
      const int npre = min(ahead, total_it);
      for (int it = 0; it < npre; ++it) issue_w(it);
      int issued = npre;
      for (int it = npre; it < total_it; ++it) {
        if (*s_abort) break;
        const int prev = it - ahead;
        if (!wait_or_abort(emptyW_bar(prev % NW), static_cast<uint32_t>(prev / NW) & 1u, a.timeout_ns, s_abort)) {
          fail(a.err, DEV_TIMEOUT_EMPTY, s_abort);
          break;
        }
        issue_w(it);
        issued = it + 1;
      }
      *s_issued_w = issued;
    }
  } else if (warp == 6) {
    // ================================================================ activation producer
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();
      pdl_wait();  // the activations come from the split kernel
      int issued = 0;
      for (int it = 0; it < total_it; ++it) {
        if (*s_abort) break;
        const int s = it % NA;
        if (it >= NA &&
            !wait_or_abort(emptyA_bar(s), static_cast<uint32_t>((it / NA) - 1) & 1u, a.timeout_ns, s_abort)) {
          fail(a.err, DEV_TIMEOUT_EMPTY, s_abort);
          break;
        }
        int n, m;
        tile_coords(it / a.kblocks, n, m);
        const int kb = it % a.kblocks;
        const uint32_t st = ringA_u + static_cast<uint32_t>(s) * G::A_BYTES;
        const int64_t img = STACKED ? static_cast<int64_t>(kb) * G::A_BYTES
                                    : (static_cast<int64_t>(m) * a.kblocks + kb) * G::A_BYTES;
        mbar_arrive_expect_tx(fullA_bar(s), G::A_BYTES);
        bulk_g2s(st, a.act_img + img, G::A_BYTES, fullA_bar(s), pol_a);
        issued = it + 1;
      }
      *s_issued_a = issued;
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(TC_M, G::N);
      int it = 0;
      bool ok = true;
      for (int tile_i = 0; tile_i < my_tiles && ok; ++tile_i) {
        const int acc = tile_i & 1, use = tile_i >> 1;
        if (use >= 1 && !wait_or_abort(tempty_bar(acc), static_cast<uint32_t>(use - 1) & 1u, a.timeout_ns, s_abort)) {
          fail(a.err, DEV_TIMEOUT_EMPTY, s_abort);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc) * TC_ACC_COLS;
        for (int kb = 0; kb < a.kblocks; ++kb, ++it) {
          const int sa = it % NA, sw = it % NW;
          if (!wait_or_abort(fullA_bar(sa), static_cast<uint32_t>(it / NA) & 1u, a.timeout_ns, s_abort) ||
              !wait_or_abort(fullW_bar(sw), static_cast<uint32_t>(it / NW) & 1u, a.timeout_ns, s_abort)) {
            fail(a.err, DEV_TIMEOUT_FULL, s_abort);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sta = ringA_u + static_cast<uint32_t>(sa) * G::A_BYTES;
          const uint32_t stw = ringW_u + static_cast<uint32_t>(sw) * G::W_BYTES;
#pragma unroll
          for (int ks = 0; ks < TC_KB / 16; ++ks) {
            const uint64_t bd = sdesc_sw128(stw + ks * 2048u, W_BOX_BYTES, 1024u);
            const uint64_t ah = sdesc_sw128(sta + ks * 32u, 16u, 1024u);
            tc_mma(d, ah, bd, idesc, (kb | ks) != 0 ? 1u : 0u);
            if (!STACKED) {
              const uint64_t al = sdesc_sw128(sta + A_BOX_BYTES + ks * 32u, 16u, 1024u);
              tc_mma(d, al, bd, idesc, 1u);
            }
          }
          tc_commit(emptyA_bar(sa));  // the stages are free once these MMAs have read them
          tc_commit(emptyW_bar(sw));
        }
        if (ok) tc_commit(tfull_bar(acc));
      }
      *s_consumed = it;
      // nothing of ours may still run on the tensor cores when the memory is released
      tc_commit(done_bar);
      if (!mbar_wait_bounded(done_bar, 0u, DEFAULT_TIMEOUT_NS)) raise_error(a.err, DEV_TIMEOUT_DRAIN);
    }
  } else {
    // ================================================================ epilogue (128 threads)
    pdl_wait();  // row_scale comes from the split kernel
    const int et = tid - 64;
    const int wq = warp & 3;  // tensor-memory lane quarter this warp may read
    const uint32_t tbuf_u = smem_u32(tbuf);
    const uint64_t pol_l = policy_evict_first();
    int store_n = 0;  // boxes this warp has stored (selects the double buffer)
    if (lane == 0) tma_prefetch_map(&mapL);
    for (int tile_i = 0; tile_i < my_tiles; ++tile_i) {
      const int acc = tile_i & 1, use = tile_i >> 1;
      if (et == 0) {
        bool ok = wait_or_abort(tfull_bar(acc), static_cast<uint32_t>(use) & 1u, a.timeout_ns, s_abort);
        if (!ok) fail(a.err, DEV_TIMEOUT_FULL, s_abort);
        s_go[tile_i & 1] = ok ? 1 : 0;
      }
      named_sync(1, 128);
      if (!s_go[tile_i & 1]) break;  // uniform across the epilogue warps
      tc_fence_after();
      int n, m;
      tile_coords(tile_i, n, m);
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * wq) << 16) + static_cast<uint32_t>(acc) * TC_ACC_COLS;
      // stacked: warps wq and wq + 2 hold the hi and the lo parts of the same 32 batch rows
      const int row = STACKED ? 32 * (wq & 1) + lane : m * TC_M + 32 * wq + lane;
      const bool valid = row < a.B;
      const float rs = valid ? a.row_scale[row] : 0.f;
      uint64_t L[TC_LIST];  // this tile's top TC_LIST candidates of the row (composites, descending)
#pragma unroll
      for (int i = 0; i < TC_LIST; ++i) L[i] = 0ull;
      const int rbase = row - lane;  // first row of this warp's 32
      if constexpr (STACKED) {
        // Each warp of a pair forms hi + lo for one half of every 32-column chunk (the hi warp columns
        // 0-15, the lo warp 16-31, after handing the other half over through xbuf), keeps its own
        // list of that half, and both write their half into the pair's store box.  The lists are
        // merged at the tile's end.
        const bool hi_part = wq < 2;
        const int pair = wq & 1;
        const int xr = 32 * pair + lane;
        float* xo = xbuf + (hi_part ? 0 : XHALF) + xr * XHALF_PITCH;        // this warp's half for its partner
        const float* xi = xbuf + (hi_part ? XHALF : 0) + xr * XHALF_PITCH;  // the partner's half
#pragma unroll 1
        for (int c = 0; c < G::CHUNKS; ++c) {
          float v[32];
          tmem_ld32(taddr + 32u * c, v);
          const int col0 = n * G::N + 32 * c;
          const bool live = col0 < a.V;  // uniform across the epilogue
          // the pair's box this chunk reuses has been read by the store two chunks back
          const uint32_t box = tbuf_u + static_cast<uint32_t>(pair * 2 + (store_n & 1)) * 4096u;
          if (hi_part && lane == 0 && live) tma_store_wait_read<1>();
          if (hi_part) {
#pragma unroll
            for (int j = 0; j < 16; ++j) xo[j] = v[16 + j];
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) xo[j] = v[j];
          }
          named_sync(2, 128);
          float h[16];  // hi + lo of this warp's half, row-scaled
          if (hi_part) {
#pragma unroll
            for (int j = 0; j < 16; ++j) h[j] = (v[j] + xi[j]) * rs;
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) h[j] = (xi[j] + v[16 + j]) * rs;
          }
          if (live) {
            const int qb = hi_part ? 0 : 4;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t dst = box + static_cast<uint32_t>(lane * 128 + (((qb + q) ^ (lane & 7)) << 4));
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "f"(h[4 * q]), "f"(h[4 * q + 1]),
                           "f"(h[4 * q + 2]), "f"(h[4 * q + 3])
                           : "memory");
            }
            fence_proxy_async_smem();
          }
          named_sync(2, 128);  // both halves are in the box; xbuf is free for the next chunk
          if (live) {
            // the logits: the pair's 32 rows x 32 columns, one TMA store (rows past B and columns past V
            // are clipped by the tensor map)
            if (hi_part && lane == 0) {
              tma_store_2d(&mapL, col0, rbase, box, pol_l);
              tma_store_commit();
            }
            ++store_n;
            const int cb = col0 + (hi_part ? 0 : 16);
            const int nv = a.V - cb;  // columns of this half inside V: >= 16, or <= 0 (V is a multiple of 16)
            uint64_t c16[16];
            uint64_t cmax = 0ull;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              c16[j] = cand_composite(valid && j < nv, h[j], cb + j);
              cmax = c16[j] > cmax ? c16[j] : cmax;
            }
            if (__any_sync(0xffffffffu, cmax > L[TC_LIST - 1])) {  // the list can change
              uint64_t t8[TC_LIST];
              top8_of16<0>(c16, t8);
              merge_top8(L, t8);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(acc));
        // the lo warp's list joins the hi warp's (xbuf is free: every chunk ended with a barrier, and
        // the next tile's first write to it follows the next tile's start barrier)
        uint64_t* xl = reinterpret_cast<uint64_t*>(xbuf) + xr * TC_LIST;
        if (!hi_part) {
#pragma unroll
          for (int i = 0; i < TC_LIST; ++i) xl[i] = L[i];
        }
        named_sync(2, 128);
        if (hi_part) {
          uint64_t o[TC_LIST];
#pragma unroll
          for (int i = 0; i < TC_LIST; ++i) o[i] = xl[i];
          merge_top8(L, o);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < G::CHUNKS; ++c) {
          float v[32];
          tmem_ld32(taddr + 32u * c, v);
          const int col0 = n * G::N + 32 * c;
          if (col0 < a.V) {  // uniform across the epilogue
            const int nv = min(32, a.V - col0);  // 16 or 32: V is a multiple of 16
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= rs;
            // the logits: this warp's 32 rows x 32 columns as one 128-byte-swizzled box, stored by TMA
            // (rows past B and columns past V are clipped by the tensor map)
            const uint32_t box = tbuf_u + static_cast<uint32_t>(wq * G::TBUF_N + store_n % G::TBUF_N) * 4096u;
            if (lane == 0) {  // the box this store reuses has been read by its previous store
              if (G::TBUF_N == 2) tma_store_wait_read<1>(); else tma_store_wait_read<0>();
            }
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint32_t dst = box + static_cast<uint32_t>(lane * 128 + ((q ^ (lane & 7)) << 4));
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "f"(v[4 * q]), "f"(v[4 * q + 1]),
                           "f"(v[4 * q + 2]), "f"(v[4 * q + 3])
                           : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&mapL, col0, rbase, box, pol_l);
              tma_store_commit();
            }
            ++store_n;
            // this tile's top TC_LIST candidates of the row: the first chunk fills the list through the
            // networks; later chunks push only their columns above its last entry
            if (c == 0) {
              uint64_t c32[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) c32[j] = cand_composite(valid && j < nv, v[j], col0 + j);
              uint64_t u8[TC_LIST];
              top8_of16<0>(c32, L);
              top8_of16<16>(c32, u8);
              merge_top8(L, u8);
            } else {
              uint32_t cand = 0u;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                cand |= cand_composite(valid && j < nv, v[j], col0 + j) > L[TC_LIST - 1] ? (1u << j) : 0u;
              push_candidates(L, cand, box, col0);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(acc));
      }
      if (valid && (!STACKED || wq < 2)) {
        ulonglong2* dst = reinterpret_cast<ulonglong2*>(a.lists + (static_cast<int64_t>(row) * a.ntn + n) * TC_LIST);
#pragma unroll
        for (int i = 0; i < TC_LIST / 2; ++i) dst[i] = make_ulonglong2(L[2 * i], L[2 * i + 1]);
      }
    }
    if (lane == 0) tma_store_wait_all();  // the logits are in global memory before the CTA leaves
  }

  // ================================================================ wind down
  __syncthreads();
  if ((warp == 0 || warp == 6) && lane == 0) {
    // copies issued for stages the MMA warp never consumed must land before the CTA leaves
    const bool w = warp == 0;
    const int nst = w ? NW : NA;
    const int issued = w ? *s_issued_w : *s_issued_a;
    for (int it = *s_consumed; it < issued; ++it) {
      const uint32_t bar = w ? fullW_bar(it % nst) : fullA_bar(it % nst);
      if (!mbar_wait_bounded(bar, static_cast<uint32_t>(it / nst) & 1u, DEFAULT_TIMEOUT_NS)) {
        raise_error(a.err, DEV_TIMEOUT_DRAIN);
        break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, TC_TMEM_COLS);
  }
  pdl_launch_dependents();
}

template <bool STACKED>
cudaError_t launch_tc_t(const TcArgs& a, const CUtensorMap& mapW, const CUtensorMap& mapL,
                        int grid, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = TcGeom<STACKED>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, lmhead_tc_kernel<STACKED>, mapW, mapL, a);
}

}  // namespace

cudaError_t launch_tc(const TcArgs& a, const CUtensorMap& mapW, const CUtensorMap& mapL,
                      int stacked, int grid, cudaStream_t stream, bool pdl) {
  return stacked ? launch_tc_t<true>(a, mapW, mapL, grid, stream, pdl)
                 : launch_tc_t<false>(a, mapW, mapL, grid, stream, pdl);
}

cudaError_t prepare_tc_gemm(int max_smem_optin) {
  if (static_cast<int>(TcGeom<false>::SMEM) > max_smem_optin || static_cast<int>(TcGeom<true>::SMEM) > max_smem_optin)
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(lmhead_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(TcGeom<false>::SMEM));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(lmhead_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(TcGeom<true>::SMEM));
}

}  // namespace tail
