// C ABI of the decode sampling tail: handle lifetime, argument validation,
// scratch ownership and the launch sequence of one step
//   [rms_rows ->] lm_head + global top-k + sampler (one launch),
// on the caller's stream, chained with programmatic dependent launch.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include <cuda.h>

#include <mutex>

#include "../../include/tail.h"
#include "abi_common.h"
#include "internal.h"
#include "moe_internal.h"
#include "small_internal.h"
#include "taps_internal.h"
#include "tc_internal.h"

using namespace tail;

struct tail_s {
  tail_config cfg;
  int device;
  int num_sms;
  int max_smem;
  int nslab;
  int rows_pass;  // rows per lm_head pass
  int tc_min;     // batches of at least this many rows take the tensor-core path; 0: none do
  int pdl_ok;     // 0 once a launch with programmatic serialization was refused
  int64_t scratch_bytes;
  // device scratch
  uint32_t* apack;
  float* row_scale;
  uint64_t* cand;
  float* logit_scratch;
  uint32_t* meta;
  unsigned long long* row_sync;
  float* topk_val;
  int32_t* topk_idx;
  int* err;
  // tensor-core path (gbs >= tc_min)
  uint8_t* tc_act;      // the activation image of the largest batch (tc_act_image_bytes)
  float* tc_rs;         // [gbs_max] row scales
  uint64_t* tc_lists;   // [gbs_max][tc_ntn_max][TC_LIST]
  float* tc_logits;     // [gbs_max][V] fp32 logits when the caller passes none
  int tc_ntn_max;       // column tiles of the narrower tile width (the most lists a row can have)
  uint8_t* tc_wpack;    // the prepared copy of the weight (tail_prepare_weight), or null
  int64_t tc_wpack_bytes;
  const void* tc_wpack_src;  // the w_t it was prepared from: runs with this pointer read the copy
  int merge_dyn;
  int merge_capc, merge_sortP, merge_smem;
  const void* tc_map_w_ptr;  // tensor maps cached for (w_t pointer, logits pointer, batch rows)
  const void* tc_map_l_ptr;
  int tc_map_rows;
  CUtensorMap tc_map_w;
  CUtensorMap tc_map_l;
  // one-launch small path (cfg.path TAIL_PATH_SMALL): every batch
  int small;
  int small_dyn;                 // the kernel's dynamic shared memory limit
  float* sm_logits;              // [gbs_max][V] fp32 logits when the caller passes none
  unsigned long long* sm_sync;   // [gbs_max] per-row arrival words, zero between launches
  uint32_t* sm_smax;             // [gbs_max][SMALL_MAX_SLABS] the slabs' largest keys of each row
  // staging of tail_run_host
  void* st_hidden;
  float* st_params;
  int32_t* st_tokens;
  int32_t* st_tokens_mapped;  // pinned, mapped host memory [gbs_max]: the kernels write the tokens there
  float* st_logits;
  // wait bound of the kernels and the dropped-stage test hook
  uint64_t wait_limit_ns;
  int drop_iter;
  // per-kernel profiling
  int prof_on;
  int prof_n;
  cudaEvent_t* prof_ev;  // [PROF_MAX][PROF_EV]
};

static constexpr int PROF_MAX = 256;
static constexpr int PROF_EV = 4;  // before the RMSNorm kernel, after it, after the lm_head, after the merge

namespace tail {

static thread_local char g_last_error[256] = "";

int cuda_fail(cudaError_t e, const char* what) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", what, cudaGetErrorString(e), static_cast<int>(e));
  cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? TAIL_ERR_OOM : TAIL_ERR_CUDA;
}

void set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

int validate_config(const tail_config* c) {
  if (!c) return TAIL_ERR_INVALID_ARG;
  const int Hu = c->hidden_actual <= 0 ? c->H : c->hidden_actual;
  if (c->H <= 0 || c->V <= 0 || Hu < 1 || Hu > c->H) return TAIL_ERR_INVALID_ARG;
  if (c->k < 1 || c->k > MAX_K || c->k > c->V) return TAIL_ERR_INVALID_ARG;
  if (c->gbs_max < 1 || c->gbs_max > 4096) return TAIL_ERR_INVALID_ARG;
  if (c->hidden_dtype < TAIL_F32 || c->hidden_dtype > TAIL_BF16) return TAIL_ERR_INVALID_ARG;
  if (!(c->eps >= 0.0f)) return TAIL_ERR_INVALID_ARG;
  if (c->H % KSTEP != 0 || c->V % 16 != 0) return TAIL_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(c->H) * c->V >= (int64_t(1) << 40)) return TAIL_ERR_UNSUPPORTED;
  return TAIL_OK;
}

}  // namespace tail

namespace {

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

template <typename T>
cudaError_t dalloc(T** p, size_t n, int64_t* total) {
  *p = nullptr;
  if (n == 0) return cudaSuccess;
  *total += static_cast<int64_t>(n * sizeof(T));
  return cudaMalloc(reinterpret_cast<void**>(p), n * sizeof(T));
}

void free_all(tail_t* h) {
  void* ptrs[] = {h->apack,    h->row_scale, h->cand,      h->logit_scratch, h->meta,
                  h->row_sync, h->topk_val,  h->topk_idx,  h->err,           h->st_hidden,
                  h->st_params, h->st_tokens, h->st_logits, h->tc_act,   h->tc_rs,         h->tc_lists,
                  h->tc_logits, h->tc_wpack, h->sm_logits, h->sm_sync, h->sm_smax};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  if (h->st_tokens_mapped) cudaFreeHost(h->st_tokens_mapped);
}

// cuTensorMapEncodeTiled, reached through the runtime (the library links no driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  });
  return fn;
}

// 2-D tensor [rows][cols] (cols contiguous) of bf16 or fp32, box box_cols x box_rows, 128-byte swizzle,
// zero fill outside on loads, clipped stores.
bool encode_2d(CUtensorMap* map, const void* base, bool fp32, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (fp32 ? 4 : 2)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of one producer-step pass of B rows (the lm_head kernel's activation warp loads a
// stage's 32 columns of every row with one copy each): the residual [B][H] bf16, box 32 x B, and
// the slots [B][S][H], box 32 x MOE_FUSED_MAX_SLOTS x B (slots past S read as zeros).  No swizzle:
// the boxes land as plain rows.
bool encode_moe_maps(GemvArgs& ga, const MoeIn& m, int B, int H) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  const cuuint64_t xdims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t xstr[1] = {static_cast<cuuint64_t>(H) * 2};
  const cuuint32_t xbox[2] = {32, static_cast<cuuint32_t>(B)};
  if (fn(&ga.moe_map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(m.x), xdims, xstr, xbox, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  if (m.S == 0) return true;
  const cuuint64_t esz = m.slot_dtype == 0 ? 4 : 2;
  const cuuint64_t ydims[3] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(m.S), static_cast<cuuint64_t>(B)};
  const cuuint64_t ystr[2] = {static_cast<cuuint64_t>(H) * esz, static_cast<cuuint64_t>(m.S) * H * esz};
  const cuuint32_t ybox[3] = {32, MOE_FUSED_MAX_SLOTS, static_cast<cuuint32_t>(B)};
  return fn(&ga.moe_map_y, m.slot_dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(m.slots), ydims, ystr, ybox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

const char* tail_last_error(void) { return g_last_error; }

const char* tail_status_string(int s) {
  switch (s) {
    case TAIL_OK: return "ok";
    case TAIL_ERR_INVALID_ARG: return "invalid argument";
    case TAIL_ERR_UNSUPPORTED: return "unsupported shape, dtype or device";
    case TAIL_ERR_CUDA: return "CUDA runtime error";
    case TAIL_ERR_OOM: return "out of device memory";
    case TAIL_ERR_DEVICE: return "device-side error flag raised (bounded wait ran out)";
    default: return "unknown status";
  }
}

int tail_create(const tail_config* cfg, int device, tail_t** out) {
  if (!out) return TAIL_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc) return rc;
  if (cfg->path < TAIL_PATH_AUTO || cfg->path > TAIL_PATH_SMALL) return TAIL_ERR_INVALID_ARG;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return TAIL_ERR_INVALID_ARG;
  DeviceGuard guard(device);
  if (!guard.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
  cudaDeviceProp prop;
  cudaError_t pe = cudaGetDeviceProperties(&prop, device);
  if (pe != cudaSuccess) return cuda_fail(pe, "cudaGetDeviceProperties");
  if (prop.major != 10 || prop.minor != 3) return TAIL_ERR_UNSUPPORTED;  // built for sm_103a only

  tail_t* h = new (std::nothrow) tail_t();
  if (!h) return TAIL_ERR_OOM;
  memset(h, 0, sizeof(*h));
  h->cfg = *cfg;
  if (h->cfg.hidden_actual <= 0) h->cfg.hidden_actual = h->cfg.H;
  h->device = device;
  h->num_sms = prop.multiProcessorCount;
  h->max_smem = static_cast<int>(prop.sharedMemPerBlockOptin);
  const int64_t npairs = cfg->V / 16;
  h->nslab = slab_count(npairs, h->num_sms, MAX_SLABS);
  // the tensor-core path, when the merge can be planned for k and V: batches of
  // TC_MIN_ROWS rows or more always take it; narrow vocabularies take it for
  // every batch (the mma.sync kernel's per-row bulk copies make it no faster there)
  h->tc_ntn_max = tc_col_tiles(cfg->V, TC_N_STACKED);
  cudaError_t te = prepare_tc(static_cast<int>(prop.sharedMemPerBlockOptin), &h->merge_dyn);
  if (te != cudaSuccess) {
    delete h;
    return cuda_fail(te, "cudaFuncSetAttribute (tensor-core kernels)");
  }
  // one merge plan for both tile widths: the candidate buffers do not depend on the tile count,
  // the shared memory for the lists does, so the larger of the two requirements is kept
  int capc2 = 0, sortP2 = 0, smem2 = 0;
  const bool tc_ok =
      encode_tiled() &&
      plan_merge(cfg->k, h->tc_ntn_max, h->merge_dyn, &h->merge_capc, &h->merge_sortP, &h->merge_smem) &&
      plan_merge(cfg->k, tc_col_tiles(cfg->V, TC_N_SEPARATE), h->merge_dyn, &capc2, &sortP2, &smem2) &&
      capc2 == h->merge_capc && sortP2 == h->merge_sortP;
  if (smem2 > h->merge_smem) h->merge_smem = smem2;
  if (cfg->path == TAIL_PATH_SMALL) {  // one launch for every batch, when the problem fits its limits
    cudaError_t se = prepare_small(static_cast<int>(prop.sharedMemPerBlockOptin), &h->small_dyn);
    if (se != cudaSuccess) {
      delete h;
      return cuda_fail(se, "cudaFuncSetAttribute (small tail kernel)");
    }
    if (!plan_small(cfg->gbs_max, cfg->H, cfg->V, cfg->k, h->num_sms, h->small_dyn).ok) {
      delete h;
      return TAIL_ERR_UNSUPPORTED;
    }
    h->small = 1;
    h->tc_min = cfg->gbs_max + 1;  // no batch reaches the tensor-core path
  } else if (cfg->path == TAIL_PATH_TENSOR)
    h->tc_min = 1;
  else if (cfg->path == TAIL_PATH_AUTO && cfg->V <= TAIL_TC_ALL_ROWS_MAX_V && tc_ok)
    h->tc_min = 1;
  else
    h->tc_min = TC_MIN_ROWS;
  const bool use_tc = cfg->gbs_max >= h->tc_min;
  if (use_tc && !tc_ok) {
    delete h;
    return TAIL_ERR_UNSUPPORTED;
  }
  if (!use_tc) h->tc_min = 0;
  // smaller batches run on the mma.sync lm_head, up to TC_MIN_ROWS - 1 rows a pass
  h->rows_pass = (h->tc_min == 1 || h->small) ? 0 : cfg->gbs_max < TC_MIN_ROWS - 1 ? cfg->gbs_max : TC_MIN_ROWS - 1;
  int max_dyn = 0;
  cudaError_t pe2 = prepare_gemv(h->max_smem, &max_dyn);
  if (pe2 != cudaSuccess) {
    delete h;
    return cuda_fail(pe2, "cudaFuncSetAttribute (shared memory opt-in)");
  }
  h->max_smem = max_dyn;
  // every row count the passes can use must have a shared-memory plan
  for (int B = 1; B <= h->rows_pass; ++B) {
    if (!plan_gemv(B, cfg->H, cfg->V, cfg->k, h->nslab, h->max_smem).ok) {
      delete h;
      return TAIL_ERR_UNSUPPORTED;
    }
  }
  // the slab selects hold a slab row in registers: at most SEL_NPL keys per lane
  if (h->rows_pass > 0 && (npairs + h->nslab - 1) / h->nslab * 16 > 32 * SEL_NPL) {
    delete h;
    return TAIL_ERR_UNSUPPORTED;
  }
  h->pdl_ok = 1;

  const int R = h->rows_pass;
  const int Rpad = ((R + 7) / 8) * 8 < 8 ? 8 : ((R + 7) / 8) * 8;
  const int mt_max = Rpad / 8 <= 1 ? 1 : Rpad / 8 <= 2 ? 2 : Rpad / 8 <= 4 ? 4 : 8;
  const size_t ksteps = cfg->H / KSTEP;
  const size_t K = cfg->k;
  int64_t tot = 0;
  cudaError_t e = cudaSuccess;
  e = e ? e : dalloc(&h->apack, ksteps * mt_max * APACK_TILE_BYTES / 4, &tot);
  e = e ? e : dalloc(&h->row_scale, static_cast<size_t>(mt_max) * 8, &tot);
  e = e ? e : dalloc(&h->cand, static_cast<size_t>(R) * h->nslab * SLAB_CAND, &tot);
  e = e ? e : dalloc(&h->logit_scratch, static_cast<size_t>(R) * cfg->V, &tot);
  e = e ? e : dalloc(&h->meta, static_cast<size_t>(R) * h->nslab * SLAB_META_WORDS, &tot);
  e = e ? e : dalloc(&h->row_sync, static_cast<size_t>(2 * R), &tot);  // arrivals, then copies
  e = e ? e : dalloc(&h->topk_val, static_cast<size_t>(cfg->gbs_max) * K, &tot);
  e = e ? e : dalloc(&h->topk_idx, static_cast<size_t>(cfg->gbs_max) * K, &tot);
  e = e ? e : dalloc(&h->err, 1, &tot);
  e = e ? e : dalloc(reinterpret_cast<uint8_t**>(&h->st_hidden),
                     static_cast<size_t>(cfg->gbs_max) * cfg->H * elem_bytes(cfg->hidden_dtype), &tot);
  e = e ? e : dalloc(&h->st_params, static_cast<size_t>(cfg->gbs_max) * 4, &tot);
  e = e ? e : dalloc(&h->st_tokens, static_cast<size_t>(cfg->gbs_max), &tot);
  if (use_tc) {
    const size_t G = static_cast<size_t>(cfg->gbs_max);
    // the separate-tile layout of gbs_max rows covers the stacked one of any smaller batch
    const size_t act_bytes = static_cast<size_t>(tc_act_image_bytes(cfg->gbs_max, cfg->H));
    e = e ? e : dalloc(&h->tc_act, act_bytes, &tot);
    e = e ? e : dalloc(&h->tc_rs, G, &tot);
    e = e ? e : dalloc(&h->tc_lists, G * h->tc_ntn_max * TC_LIST, &tot);
    e = e ? e : dalloc(&h->tc_logits, G * cfg->V, &tot);
    // rows of the activation image past a batch's rows still feed the MMA: keep them finite
    if (e == cudaSuccess) e = cudaMemset(h->tc_act, 0, act_bytes);
  }
  if (h->small) {
    e = e ? e : dalloc(&h->sm_logits, static_cast<size_t>(cfg->gbs_max) * cfg->V, &tot);
    e = e ? e : dalloc(&h->sm_sync, static_cast<size_t>(cfg->gbs_max), &tot);
    e = e ? e : dalloc(&h->sm_smax, static_cast<size_t>(cfg->gbs_max) * SMALL_MAX_SLABS, &tot);
    if (e == cudaSuccess) e = cudaMemset(h->sm_sync, 0, static_cast<size_t>(cfg->gbs_max) * sizeof(unsigned long long));
  }
  if (e == cudaSuccess) e = cudaMemset(h->err, 0, sizeof(int));
  if (e == cudaSuccess && R > 0) e = cudaMemset(h->row_sync, 0, static_cast<size_t>(2 * R) * sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(h->apack, 0, ksteps * mt_max * APACK_TILE_BYTES);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_all(h);
    delete h;
    return cuda_fail(e, "scratch allocation");
  }
  h->scratch_bytes = tot;
  h->wait_limit_ns = DEFAULT_TIMEOUT_NS;
  h->drop_iter = -1;
  *out = h;
  return TAIL_OK;
}

// Launches with programmatic dependent launch while the handle's runtime takes it.  A launch that
// fails with the attribute is retried once without it; only when that retry succeeds (the attribute
// was what the runtime refused) does the handle stop using it.  Any other failure is returned as it is.
}  // extern "C"

template <typename Launch>
static cudaError_t launch_pdl(tail_t* h, Launch launch) {
  if (!h->pdl_ok) return launch(false);
  cudaError_t e = launch(true);
  if (e == cudaSuccess) return e;
  cudaGetLastError();  // a refused launch leaves a (non-sticky) error behind
  const cudaError_t e2 = launch(false);
  if (e2 == cudaSuccess) h->pdl_ok = 0;
  return e2 == cudaSuccess ? e2 : e;
}

extern "C" {

// The small path: one launch forms the activations, the logits, the top k and the tokens of every row.
static int run_small(tail_t* h, const void* hidden, const float* gamma, const uint16_t* w_t, const float* params,
                     int32_t ncols, int32_t gbs, int32_t* out_tokens, float* out_logits, float* out_topk_vals,
                     int32_t* out_topk_idx, cudaStream_t stream) {
  const tail_config& c = h->cfg;
  const SmallPlan plan = plan_small(gbs, c.H, c.V, c.k, h->num_sms, h->small_dyn);
  if (!plan.ok) return TAIL_ERR_UNSUPPORTED;  // not reached: the plan of gbs_max rows held at create
  cudaEvent_t* ev = (h->prof_on && h->prof_n < PROF_MAX) ? h->prof_ev + h->prof_n * PROF_EV : nullptr;
  if (ev) {
    ++h->prof_n;
    cudaEventRecord(ev[0], stream);
    cudaEventRecord(ev[1], stream);  // no RMSNorm kernel: the launch forms the activations
  }
  SmallArgs a;
  a.hidden = hidden;
  a.dtype = c.hidden_dtype;
  a.gamma = gamma;
  a.w = w_t;
  a.logits = out_logits ? out_logits : h->sm_logits;
  a.topk_val = out_topk_vals ? out_topk_vals : h->topk_val;
  a.topk_idx = out_topk_idx ? out_topk_idx : h->topk_idx;
  a.topk_ld = c.k;
  a.params = params;
  a.ncols = ncols;
  a.tokens = params ? out_tokens : nullptr;
  a.sync = h->sm_sync;
  a.smax = h->sm_smax;
  a.err = h->err;
  a.timeout_ns = h->wait_limit_ns;
  a.B = gbs;
  a.H = c.H;
  a.Hu = c.hidden_actual;
  a.V = c.V;
  a.K = c.k;
  a.zero_pad = c.zero_interleaved_pad ? 1 : 0;
  a.deferred = c.deferred_rms ? 1 : 0;
  a.eps = c.eps;
  a.slab_cols = plan.slab_cols;
  a.nslab = plan.nslab;
  a.sortP = plan.sortP;
  a.cap = plan.cap;
  a.smem_bytes = plan.smem_bytes;
  const cudaError_t e = launch_pdl(h, [&](bool pdl) { return launch_small(a, stream, pdl); });
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch (small tail)");
  if (ev) {
    cudaEventRecord(ev[2], stream);
    cudaEventRecord(ev[3], stream);  // the top k and the draw run inside the same launch
  }
  return TAIL_OK;
}

// Batches of tc_min rows or more: split -> tensor-core lm_head -> merge + sampler, one pass.
static int run_tc(tail_t* h, const void* hidden, const float* gamma, const uint16_t* w_t, const float* params,
                  int32_t ncols, int32_t gbs, int32_t* out_tokens, float* out_logits, float* out_topk_vals,
                  int32_t* out_topk_idx, cudaStream_t stream, const MoeIn* moe) {
  const tail_config& c = h->cfg;
  const int stacked = tc_stacked(gbs);
  const int n_mb = tc_mblocks(gbs);
  const int tile_n = tc_tile_n(gbs);
  const int ntn = tc_col_tiles(c.V, tile_n);
  float* logits = out_logits ? out_logits : h->tc_logits;
  if (h->tc_map_w_ptr != w_t || h->tc_map_l_ptr != logits || h->tc_map_rows != gbs) {
    if (!encode_2d(&h->tc_map_w, w_t, false, static_cast<uint64_t>(c.V), static_cast<uint64_t>(c.H), 64, 64) ||
        !encode_2d(&h->tc_map_l, logits, true, static_cast<uint64_t>(c.V), static_cast<uint64_t>(gbs), 32, 32)) {
      h->tc_map_w_ptr = nullptr;
      set_last_error("cuTensorMapEncodeTiled rejected a tensor map of the tensor-core lm_head");
      return TAIL_ERR_CUDA;
    }
    h->tc_map_w_ptr = w_t;
    h->tc_map_l_ptr = logits;
    h->tc_map_rows = gbs;
  }
  cudaEvent_t* ev = (h->prof_on && h->prof_n < PROF_MAX) ? h->prof_ev + h->prof_n * PROF_EV : nullptr;
  if (ev) {
    ++h->prof_n;
    cudaEventRecord(ev[0], stream);
  }
  SplitArgs sa;
  sa.hidden = hidden;
  sa.dtype = c.hidden_dtype;
  sa.gamma = gamma;
  sa.B = gbs;
  sa.H = c.H;
  sa.Hu = c.hidden_actual;
  sa.eps = c.eps;
  sa.zero_pad = c.zero_interleaved_pad ? 1 : 0;
  sa.deferred = c.deferred_rms ? 1 : 0;
  sa.stacked = stacked;
  sa.act_img = h->tc_act;
  sa.row_scale = h->tc_rs;
  if (moe) {  // the split kernel forms each row from the residual and the slots itself
    sa.use_moe = 1;
    sa.moe = *moe;
  }
  cudaError_t e = launch_split(sa, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch (split)");
  if (ev) cudaEventRecord(ev[1], stream);

  TcArgs ta;
  ta.act_img = h->tc_act;
  if (h->tc_wpack != nullptr && h->tc_wpack_src == w_t) {
    ta.w_packed = h->tc_wpack;
    ta.w_groups = tc_weight_groups(c.V);
    ta.w_ahead = stacked ? TC_PACKED_AHEAD_STACKED : TC_PACKED_AHEAD_SEPARATE;
  }
  ta.row_scale = h->tc_rs;
  ta.logits = logits;
  ta.ld = c.V;
  ta.lists = h->tc_lists;
  ta.err = h->err;
  ta.B = gbs;
  ta.V = c.V;
  ta.ntn = ntn;
  ta.n_mb = n_mb;
  ta.kblocks = (c.H + TC_KB - 1) / TC_KB;
  ta.timeout_ns = h->wait_limit_ns;
  const int ntiles = ntn * n_mb;
  e = launch_tc(ta, h->tc_map_w, h->tc_map_l, stacked, ntiles < h->num_sms ? ntiles : h->num_sms,
                stream, true);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch (tensor-core lm_head)");
  if (ev) cudaEventRecord(ev[2], stream);

  MergeArgs ma;
  ma.lists = h->tc_lists;
  ma.logits = ta.logits;
  ma.ld = c.V;
  ma.topk_val = out_topk_vals ? out_topk_vals : h->topk_val;
  ma.topk_idx = out_topk_idx ? out_topk_idx : h->topk_idx;
  ma.topk_ld = c.k;
  ma.params = params;
  ma.ncols = ncols;
  ma.tokens = params ? out_tokens : nullptr;
  ma.B = gbs;
  ma.V = c.V;
  ma.K = c.k;
  ma.ntn = ntn;
  ma.tile_n = tile_n;
  ma.capc = h->merge_capc;
  ma.sortP = h->merge_sortP;
  ma.smem_bytes = h->merge_smem;
  ma.err = h->err;
  ma.timeout_ns = h->wait_limit_ns;
  e = launch_merge(ma, gbs, stream, true);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch (merge)");
  if (ev) cudaEventRecord(ev[3], stream);
  return TAIL_OK;
}

// Slot element bytes of a producer step.
static int moe_slot_bytes(const MoeIn& m) { return m.slot_dtype == 0 ? 4 : 2; }

// Whether every pass of a batch of gbs rows can run the producer step inside its first kernel:
// the split kernel on the tensor-core path; the lm_head kernel's activation warp (fused deferred
// form, at most MOE_FUSED_MAX_SLOTS slots, 16-byte aligned slots) on the mma.sync path.
static bool moe_fusable(const tail_t* h, int gbs, const MoeIn& m) {
  const tail_config& c = h->cfg;
  if (h->tc_min > 0 && gbs >= h->tc_min) return c.H <= SPLIT_MOE_MAX_H;
  if (h->rows_pass <= 0 || !c.deferred_rms || m.S > MOE_FUSED_MAX_SLOTS || !encode_tiled()) return false;
  if (m.S > 0 && !aligned(m.slots, 16)) return false;
  const int sizes[2] = {gbs < h->rows_pass ? gbs : h->rows_pass, gbs % h->rows_pass};
  for (int B : sizes) {
    if (B == 0) continue;
    const GemvPlan p = plan_gemv(B, c.H, c.V, c.k, h->nslab, h->max_smem, GEMV_KPB, GEMV_MAX_STAGES, m.S,
                                 moe_slot_bytes(m));
    if (!p.ok || !p.logits_in_smem || p.mt > FUSED_MAX_MT) return false;
  }
  return true;
}

// moe: run the producer step inside the first kernel of every pass (moe_fusable holds); hidden is
// then unused.
static int run_impl(tail_t* h, const void* hidden, const float* gamma, const uint16_t* w_t,
                    const float* params, int32_t ncols, int32_t gbs, int32_t* out_tokens, float* out_logits,
                    float* out_topk_vals, int32_t* out_topk_idx, cudaStream_t stream, const MoeIn* moe = nullptr) {
  const tail_config& c = h->cfg;
  if (h->small)  // moe is null here: moe_fusable does not hold on the small path
    return run_small(h, hidden, gamma, w_t, params, ncols, gbs, out_tokens, out_logits, out_topk_vals, out_topk_idx,
                     stream);
  if (h->tc_min > 0 && gbs >= h->tc_min)
    return run_tc(h, hidden, gamma, w_t, params, ncols, gbs, out_tokens, out_logits, out_topk_vals, out_topk_idx,
                  stream, moe);
  if (h->rows_pass <= 0) return TAIL_ERR_UNSUPPORTED;  // no mma.sync scratch (not reached: tc_min is 1)
  const int K = c.k;
  const int64_t npairs = c.V / 16;
  cudaError_t e = cudaSuccess;
  for (int r0 = 0; r0 < gbs && e == cudaSuccess; r0 += h->rows_pass) {
    const int B = gbs - r0 < h->rows_pass ? gbs - r0 : h->rows_pass;
    const GemvPlan plan = moe ? plan_gemv(B, c.H, c.V, K, h->nslab, h->max_smem, GEMV_KPB, GEMV_MAX_STAGES, moe->S,
                                          moe_slot_bytes(*moe))
                              : plan_gemv(B, c.H, c.V, K, h->nslab, h->max_smem);
    cudaEvent_t* ev = (h->prof_on && h->prof_n < PROF_MAX) ? h->prof_ev + h->prof_n * PROF_EV : nullptr;
    if (ev) {
      ++h->prof_n;
      cudaEventRecord(ev[0], stream);
    }

    RmsArgs ra;
    ra.hidden = hidden ? static_cast<const uint8_t*>(hidden) + static_cast<int64_t>(r0) * c.H * elem_bytes(c.hidden_dtype)
                       : nullptr;  // null with the producer step: the lm_head kernel forms the rows
    ra.dtype = c.hidden_dtype;
    ra.gamma = gamma;
    ra.B = B;
    ra.mt = plan.mt;
    ra.B_pad = plan.mt * MTILE_ROWS;
    ra.H = c.H;
    ra.Hu = c.hidden_actual;
    ra.eps = c.eps;
    ra.zero_pad = c.zero_interleaved_pad ? 1 : 0;
    ra.deferred = c.deferred_rms ? 1 : 0;
    ra.apack = h->apack;
    ra.row_scale = h->row_scale;
    // deferred RMSNorm with the slab logits in shared memory: the lm_head kernel forms the activations
    const bool fused = c.deferred_rms && plan.logits_in_smem && plan.mt <= FUSED_MAX_MT;
    if (moe && !fused) return TAIL_ERR_UNSUPPORTED;  // not reached: moe_fusable holds
    if (!fused) {
      e = launch_pdl(h, [&](bool pdl) { return launch_rms_pack(ra, stream, pdl); });
      if (e != cudaSuccess) break;
    }
    if (ev) cudaEventRecord(ev[1], stream);

    GemvArgs ga;
    ga.w = w_t;
    ga.apack = reinterpret_cast<const uint8_t*>(h->apack);
    ga.row_scale = h->row_scale;
    ga.fused = fused ? 1 : 0;
    ga.hidden = ra.hidden;
    ga.dtype = c.hidden_dtype;
    ga.gamma = gamma;
    ga.Hu = c.hidden_actual;
    ga.eps = c.eps;
    ga.zero_pad = ra.zero_pad;
    ga.logits_out = out_logits ? out_logits + static_cast<int64_t>(r0) * c.V : nullptr;
    ga.logits_out_ld = c.V;
    ga.logits_scratch = h->logit_scratch;
    ga.cand = h->cand;
    ga.err = h->err;
    ga.B = B;
    ga.H = c.H;
    ga.V = c.V;
    ga.K = K;
    ga.ksteps = c.H / KSTEP;
    ga.mt = plan.mt;
    ga.nslab = h->nslab;
    ga.npairs = npairs;
    ga.cb_pairs = plan.cb_pairs;
    ga.kpb = plan.kpb;
    ga.pitch = plan.pitch;
    ga.stage_bytes = plan.stage_bytes;
    ga.nstages = plan.nstages;
    ga.logits_in_smem = plan.logits_in_smem;
    ga.max_slab_cols = plan.max_slab_cols;
    ga.smem_bytes = plan.smem_bytes;
    ga.meta = h->meta;
    ga.row_sync = h->row_sync;
    ga.row_copy = h->row_sync + h->rows_pass;
    ga.topk_val = (out_topk_vals ? out_topk_vals : h->topk_val) + static_cast<int64_t>(r0) * K;
    ga.topk_idx = (out_topk_idx ? out_topk_idx : h->topk_idx) + static_cast<int64_t>(r0) * K;
    ga.topk_ld = K;
    ga.params = params ? params + static_cast<int64_t>(r0) * ncols : nullptr;
    ga.ncols = ncols;
    ga.tokens = params ? out_tokens + r0 : nullptr;
    ga.capc = plan.capc;
    ga.sortP = plan.sortP;
    ga.timeout_ns = h->wait_limit_ns;
    ga.drop_iter = h->drop_iter;
    ga.hid_slot_bytes = plan.hid_slot_bytes;
    if (moe) {  // this pass's rows of the residual, the slots, their weights and h
      ga.use_moe = 1;
      ga.moe = *moe;
      ga.moe.x = moe->x + static_cast<int64_t>(r0) * c.H;
      ga.moe.slots = static_cast<const uint8_t*>(moe->slots) +
                     static_cast<int64_t>(r0) * moe->S * c.H * moe_slot_bytes(*moe);
      ga.moe.w = moe->w + static_cast<int64_t>(r0) * moe->S;
      ga.moe.h_out = moe->h_out ? moe->h_out + static_cast<int64_t>(r0) * c.H : nullptr;
      if (!encode_moe_maps(ga, ga.moe, B, c.H)) {
        set_last_error("cuTensorMapEncodeTiled rejected a tensor map of the producer step");
        return TAIL_ERR_CUDA;
      }
    }
    e = launch_pdl(h, [&](bool pdl) { return launch_gemv(ga, stream, pdl); });
    if (e != cudaSuccess) break;
    if (ev) {
      cudaEventRecord(ev[2], stream);
      cudaEventRecord(ev[3], stream);  // the merge runs inside the lm_head launch
    }
  }
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return TAIL_OK;
}

static int validate_run(tail_t* h, const void* hidden, const float* gamma, const uint16_t* w_t,
                        const float* params, int32_t ncols, int32_t gbs, int32_t* out_tokens,
                        const float* out_logits, const float* tv, const int32_t* ti) {
  if (!h) return TAIL_ERR_INVALID_ARG;
  if (gbs < 0 || gbs > h->cfg.gbs_max) return TAIL_ERR_INVALID_ARG;
  if (gbs == 0) return TAIL_OK;
  if (!hidden || !gamma || !w_t) return TAIL_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(w_t, 16) || !aligned(gamma, 4)) return TAIL_ERR_INVALID_ARG;
  if (params) {
    if (ncols != 3 && ncols != 4) return TAIL_ERR_INVALID_ARG;
    if (!out_tokens || !aligned(params, 4) || !aligned(out_tokens, 4)) return TAIL_ERR_INVALID_ARG;
  }
  if (out_logits && !aligned(out_logits, 16)) return TAIL_ERR_INVALID_ARG;
  if ((tv && !aligned(tv, 4)) || (ti && !aligned(ti, 4))) return TAIL_ERR_INVALID_ARG;
  return TAIL_OK;
}

int tail_run_ex(tail_t* h, const void* hidden, const float* gamma, const uint16_t* w_t, const float* params,
                int32_t n_param_cols, int32_t gbs, int32_t* out_tokens, float* out_logits_opt,
                float* out_topk_vals_opt, int32_t* out_topk_idx_opt, void* stream) {
  int rc = validate_run(h, hidden, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt,
                        out_topk_vals_opt, out_topk_idx_opt);
  if (rc || gbs == 0) return rc;
  DeviceGuard guard(h->device);
  if (!guard.ok) return TAIL_ERR_CUDA;
  return run_impl(h, hidden, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt,
                  out_topk_vals_opt, out_topk_idx_opt, static_cast<cudaStream_t>(stream));
}

int tail_run_moe(tail_t* h, const uint16_t* residual, const void* slots, int32_t slot_dtype, int32_t nslots,
                 int32_t n_routed, const float* slot_w, const float* gamma, const uint16_t* w_t, const float* params,
                 int32_t n_param_cols, int32_t gbs, int32_t* out_tokens, float* out_logits_opt,
                 float* out_topk_vals_opt, int32_t* out_topk_idx_opt, uint16_t* out_hidden_opt, void* stream) {
  if (!h) return TAIL_ERR_INVALID_ARG;
  if (h->cfg.hidden_dtype != TAIL_BF16) return TAIL_ERR_UNSUPPORTED;  // the residual stream is bf16
  if (nslots < 0 || nslots > TAIL_MOE_MAX_SLOTS || (slot_dtype != TAIL_F32 && slot_dtype != TAIL_BF16))
    return TAIL_ERR_INVALID_ARG;
  if (n_routed < 0 || n_routed > nslots) return TAIL_ERR_INVALID_ARG;
  if (nslots > 0 && (!slots || !slot_w || !aligned(slots, 4) || !aligned(slot_w, 4))) return TAIL_ERR_INVALID_ARG;
  if (out_hidden_opt && !aligned(out_hidden_opt, 16)) return TAIL_ERR_INVALID_ARG;
  int rc = validate_run(h, residual, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt,
                        out_topk_vals_opt, out_topk_idx_opt);
  if (rc || gbs == 0) return rc;
  DeviceGuard guard(h->device);
  if (!guard.ok) return TAIL_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MoeIn m;
  m.x = residual;
  m.slots = slots;
  m.slot_dtype = slot_dtype == TAIL_F32 ? 0 : 2;
  m.w = slot_w;
  m.S = nslots;
  m.n_routed = n_routed;
  m.h_out = out_hidden_opt;
  if (moe_fusable(h, gbs, m))  // one launch fewer: the first kernel of the tail forms h itself
    return run_impl(h, nullptr, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt,
                    out_topk_vals_opt, out_topk_idx_opt, s, &m);
  // h lands in the caller's buffer, else in the handle's hidden staging (gbs_max x H bf16)
  m.h_out = out_hidden_opt ? out_hidden_opt : reinterpret_cast<uint16_t*>(h->st_hidden);
  cudaError_t e = launch_pdl(h, [&](bool pdl) { return launch_moe_combine(m, gbs, h->cfg.H, s, pdl); });
  if (e != cudaSuccess) return cuda_fail(e, "tail_run_moe: kernel launch");
  return run_impl(h, m.h_out, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt, out_topk_vals_opt,
                  out_topk_idx_opt, s);
}

int tail_tap_shape(const tail_t* h, int32_t gbs, int32_t* kind, int32_t* n_chunks, int32_t* cap,
                   int32_t* chunk_lo_host_opt) {
  if (!h || !kind || !n_chunks || !cap || gbs < 1 || gbs > h->cfg.gbs_max) return TAIL_ERR_INVALID_ARG;
  if (h->small) return TAIL_ERR_UNSUPPORTED;  // one top k over the whole row: no stage-1 chunks to tap
  const int V = h->cfg.V;
  if (h->tc_min > 0 && gbs >= h->tc_min) {
    const int tn = tc_tile_n(gbs);
    *kind = TAP_TILES;
    *n_chunks = tc_col_tiles(V, tn);
    *cap = TC_LIST;
    if (chunk_lo_host_opt) {
      for (int c = 0; c < *n_chunks; ++c) chunk_lo_host_opt[c] = c * tn;
      chunk_lo_host_opt[*n_chunks] = V;
    }
  } else {
    const int64_t npairs = V / 16;
    *kind = TAP_SLABS;
    *n_chunks = h->nslab;
    *cap = SLAB_CAND;
    if (chunk_lo_host_opt)
      for (int c = 0; c <= h->nslab; ++c) chunk_lo_host_opt[c] = static_cast<int32_t>(slab_pair_lo(npairs, h->nslab, c) * 16);
  }
  return TAIL_OK;
}

int tail_run_taps(tail_t* h, const void* hidden, const float* gamma, const uint16_t* w_t, const float* params,
                  int32_t n_param_cols, int32_t gbs, int32_t* out_tokens, float* out_logits_opt,
                  float* out_topk_vals_opt, int32_t* out_topk_idx_opt, float* tap_vals, int32_t* tap_idx,
                  int32_t* tap_count, float* tap_bound, void* stream) {
  if (!tap_vals || !tap_idx || !tap_count || !tap_bound) return TAIL_ERR_INVALID_ARG;
  if (!aligned(tap_vals, 4) || !aligned(tap_idx, 4) || !aligned(tap_count, 4) || !aligned(tap_bound, 4))
    return TAIL_ERR_INVALID_ARG;
  int rc = validate_run(h, hidden, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt,
                        out_topk_vals_opt, out_topk_idx_opt);
  if (rc || gbs == 0) return rc;
  const bool tc = h->tc_min > 0 && gbs >= h->tc_min;
  if (!tc && gbs > h->rows_pass) return TAIL_ERR_UNSUPPORTED;  // one mma.sync pass holds the taps
  DeviceGuard guard(h->device);
  if (!guard.ok) return TAIL_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = run_impl(h, hidden, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt, out_topk_vals_opt,
                out_topk_idx_opt, s);
  if (rc) return rc;
  TapArgs ta = {};
  int32_t kind = 0, nchunk = 0, cap = 0;
  tail_tap_shape(h, gbs, &kind, &nchunk, &cap, nullptr);
  ta.kind = kind;
  ta.meta = h->meta;
  ta.cand = h->cand;
  ta.lists = h->tc_lists;
  ta.B = gbs;
  ta.V = h->cfg.V;
  ta.nchunk = nchunk;
  ta.cap = cap;
  ta.tile_n = tc ? tc_tile_n(gbs) : 0;
  ta.vals = tap_vals;
  ta.idx = tap_idx;
  ta.count = tap_count;
  ta.bound = tap_bound;
  cudaError_t e = launch_tap_export(ta, s);
  if (e != cudaSuccess) return cuda_fail(e, "tail_run_taps: kernel launch");
  return TAIL_OK;
}

int tail_prepare_weight(tail_t* h, const uint16_t* w_t, void* stream) {
  if (!h) return TAIL_ERR_INVALID_ARG;
  if (w_t && !aligned(w_t, 16)) return TAIL_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return TAIL_ERR_CUDA;
  h->tc_wpack_src = nullptr;
  if (!w_t) {  // release the copy
    if (h->tc_wpack) {
      const cudaError_t e = cudaFree(h->tc_wpack);
      h->tc_wpack = nullptr;
      h->scratch_bytes -= h->tc_wpack_bytes;
      h->tc_wpack_bytes = 0;
      if (e != cudaSuccess) return cuda_fail(e, "tail_prepare_weight: cudaFree");
    }
    return TAIL_OK;
  }
  if (h->tc_min <= 0) return TAIL_OK;  // no tensor-core path: nothing reads a prepared copy
  if (!h->tc_wpack) {
    const int64_t bytes = tc_packed_weight_bytes(h->cfg.H, h->cfg.V);
    const cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&h->tc_wpack), static_cast<size_t>(bytes));
    if (e != cudaSuccess) {
      h->tc_wpack = nullptr;
      return cuda_fail(e, "tail_prepare_weight: allocation of the prepared weight");
    }
    h->tc_wpack_bytes = bytes;
    h->scratch_bytes += bytes;
  }
  const cudaError_t e = launch_weight_pack(w_t, h->cfg.H, h->cfg.V, h->tc_wpack, h->num_sms,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "tail_prepare_weight: kernel launch");
  h->tc_wpack_src = w_t;
  return TAIL_OK;
}

int tail_run(tail_t* h, const void* hidden, const float* gamma, const uint16_t* w_t, const float* params,
             int32_t n_param_cols, int32_t gbs, int32_t* out_tokens, float* out_logits_opt, void* stream) {
  return tail_run_ex(h, hidden, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt, nullptr,
                     nullptr, stream);
}

int tail_run_host(tail_t* h, const void* hidden_host, const float* gamma, const uint16_t* w_t,
                  const float* params_host, int32_t n_param_cols, int32_t gbs, int32_t* out_tokens_host,
                  float* out_logits_host_opt, void* stream) {
  if (!h) return TAIL_ERR_INVALID_ARG;
  if (gbs < 0 || gbs > h->cfg.gbs_max) return TAIL_ERR_INVALID_ARG;
  if (gbs == 0) return TAIL_OK;
  if (!hidden_host || (params_host && !out_tokens_host)) return TAIL_ERR_INVALID_ARG;
  if (params_host && n_param_cols != 3 && n_param_cols != 4) return TAIL_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return TAIL_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const tail_config& c = h->cfg;
  cudaError_t e = cudaSuccess;
  if (out_logits_host_opt && !h->st_logits) {
    e = cudaMalloc(reinterpret_cast<void**>(&h->st_logits), static_cast<size_t>(c.gbs_max) * c.V * 4);
    if (e != cudaSuccess) {
      h->st_logits = nullptr;
      cudaGetLastError();
      return TAIL_ERR_OOM;
    }
    h->scratch_bytes += static_cast<int64_t>(c.gbs_max) * c.V * 4;
  }
  // the tokens go straight to pinned, mapped host memory (no device-to-host copy), then to the caller
  int32_t* tok_dev = h->st_tokens;
  if (params_host && !h->st_tokens_mapped) {
    if (cudaHostAlloc(reinterpret_cast<void**>(&h->st_tokens_mapped), static_cast<size_t>(c.gbs_max) * 4,
                      cudaHostAllocMapped) != cudaSuccess) {
      h->st_tokens_mapped = nullptr;
      cudaGetLastError();  // fall back to the device staging and a copy
    }
  }
  if (params_host && h->st_tokens_mapped) {
    void* d = nullptr;
    if (cudaHostGetDevicePointer(&d, h->st_tokens_mapped, 0) == cudaSuccess) tok_dev = static_cast<int32_t*>(d);
    else cudaGetLastError();
  }
  // pinned parameters are read by the kernels where they are; others are copied first
  const float* par_dev = params_host ? h->st_params : nullptr;
  bool copy_params = params_host != nullptr;
  if (params_host) {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, params_host) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
        pa.devicePointer != nullptr && aligned(pa.devicePointer, 4)) {
      par_dev = static_cast<const float*>(pa.devicePointer);
      copy_params = false;
    }
    cudaGetLastError();
  }
  const size_t hbytes = static_cast<size_t>(gbs) * c.H * elem_bytes(c.hidden_dtype);
  e = cudaMemcpyAsync(h->st_hidden, hidden_host, hbytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && copy_params)
    e = cudaMemcpyAsync(h->st_params, params_host, static_cast<size_t>(gbs) * n_param_cols * 4,
                        cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return TAIL_ERR_CUDA;
  }
  int rc = tail_run_ex(h, h->st_hidden, gamma, w_t, par_dev, n_param_cols, gbs, tok_dev,
                       out_logits_host_opt ? h->st_logits : nullptr, nullptr, nullptr, stream);
  if (rc) return rc;
  if (params_host && tok_dev == h->st_tokens)
    e = cudaMemcpyAsync(out_tokens_host, h->st_tokens, static_cast<size_t>(gbs) * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && out_logits_host_opt)
    e = cudaMemcpyAsync(out_logits_host_opt, h->st_logits, static_cast<size_t>(gbs) * c.V * 4,
                        cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return TAIL_ERR_CUDA;
  }
  if (params_host && tok_dev != h->st_tokens)
    memcpy(out_tokens_host, h->st_tokens_mapped, static_cast<size_t>(gbs) * 4);
  return TAIL_OK;
}

int tail_check(tail_t* h) {
  if (!h) return TAIL_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return TAIL_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return TAIL_ERR_CUDA;
  }
  int flag = 0;
  if (cudaMemcpy(&flag, h->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TAIL_ERR_CUDA;
  if (flag != 0) {
    cudaMemset(h->err, 0, sizeof(int));
    // a wait that ran out leaves the per-row arrival words of the interrupted run behind
    if (h->rows_pass > 0) cudaMemset(h->row_sync, 0, static_cast<size_t>(2 * h->rows_pass) * sizeof(unsigned long long));
    if (h->small) cudaMemset(h->sm_sync, 0, static_cast<size_t>(h->cfg.gbs_max) * sizeof(unsigned long long));
    cudaDeviceSynchronize();
    return TAIL_ERR_DEVICE;
  }
  return TAIL_OK;
}

int tail_profile_enable(tail_t* h, int enable) {
  if (!h) return TAIL_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return TAIL_ERR_CUDA;
  if (enable && !h->prof_ev) {
    h->prof_ev = static_cast<cudaEvent_t*>(calloc(PROF_MAX * PROF_EV, sizeof(cudaEvent_t)));
    if (!h->prof_ev) return TAIL_ERR_OOM;
    for (int i = 0; i < PROF_MAX * PROF_EV; ++i) {
      if (cudaEventCreate(&h->prof_ev[i]) != cudaSuccess) {
        cudaGetLastError();
        return TAIL_ERR_CUDA;
      }
    }
  }
  h->prof_on = enable ? 1 : 0;
  if (enable) h->prof_n = 0;
  return TAIL_OK;
}

int tail_profile_read(tail_t* h, float* kernel_ms, int32_t* passes) {
  if (!h || !kernel_ms || !passes) return TAIL_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok) return TAIL_ERR_CUDA;
  for (int j = 0; j < PROF_EV - 1; ++j) kernel_ms[j] = 0.f;
  for (int i = 0; i < h->prof_n; ++i) {
    cudaEvent_t* ev = h->prof_ev + i * PROF_EV;
    if (cudaEventSynchronize(ev[PROF_EV - 1]) != cudaSuccess) {
      cudaGetLastError();
      return TAIL_ERR_CUDA;
    }
    for (int j = 0; j < PROF_EV - 1; ++j) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, ev[j], ev[j + 1]) != cudaSuccess) {
        cudaGetLastError();
        return TAIL_ERR_CUDA;
      }
      kernel_ms[j] += ms;
    }
  }
  *passes = h->prof_n;
  return TAIL_OK;
}

int tail_set_wait_limit(tail_t* h, uint64_t ns) {
  if (!h) return TAIL_ERR_INVALID_ARG;
  h->wait_limit_ns = ns;
  return TAIL_OK;
}

int tail_debug_drop_stage(tail_t* h, int32_t iteration) {
  if (!h || iteration < -1) return TAIL_ERR_INVALID_ARG;
  h->drop_iter = iteration;
  return TAIL_OK;
}

int tail_get_info(const tail_t* h, tail_info* out) {
  if (!h || !out) return TAIL_ERR_INVALID_ARG;
  out->num_sms = h->num_sms;
  out->nslab = h->nslab;
  out->merge_groups = 0;
  out->lmhead_path = h->pdl_ok ? 2 : 1;
  out->rows_per_pass = h->rows_pass;
  // one launch per pass when the lm_head kernel forms the activations itself, else RMSNorm + lm_head
  out->kernels_per_run = 2;
  if (h->rows_pass > 0 && h->cfg.deferred_rms) {
    const GemvPlan p = plan_gemv(h->rows_pass, h->cfg.H, h->cfg.V, h->cfg.k, h->nslab, h->max_smem);
    if (p.logits_in_smem && p.mt <= FUSED_MAX_MT) out->kernels_per_run = 1;
  }
  if (h->small) {
    out->lmhead_path = 3;
    out->rows_per_pass = h->cfg.gbs_max;
    out->kernels_per_run = 1;
  }
  out->scratch_bytes = h->scratch_bytes;
  out->tc_min_rows = h->tc_min;
  return TAIL_OK;
}

void tail_destroy(tail_t* h) {
  if (!h) return;
  {
    DeviceGuard guard(h->device);
    cudaDeviceSynchronize();
    free_all(h);
    if (h->prof_ev) {
      for (int i = 0; i < PROF_MAX * PROF_EV; ++i)
        if (h->prof_ev[i]) cudaEventDestroy(h->prof_ev[i]);
      free(h->prof_ev);
    }
  }
  delete h;
}

}  // extern "C"
