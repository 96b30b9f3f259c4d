// tail_run_noalloc: the tail without a handle and without any device
// allocation.  It launches the same mma.sync-path kernels as tail_run -- one
// launch a pass in the default deferred-RMSNorm form (the lm_head kernel forms
// the activations, then the global top-k and the sampler), two in the legacy
// form (rms_pack first) -- but their scratch lives in one file-scope device
// array of fixed size instead of handle-owned cudaMalloc memory.
//
// The array is part of this library's device image: it is created with the
// module, zero-filled, and its address is looked up once per device (with that
// device current) by the first call that runs there.  That first call also
// opts the lm_head kernels into their shared-memory size.  Every later call
// only computes a layout on the host, clears the error word and the per-row
// arrival words with one cudaMemsetAsync and launches kernels: no cudaMalloc,
// cudaFree or other allocating routine on any call.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>
#include <mutex>

#include "../../include/tail.h"
#include "abi_common.h"
#include "internal.h"

using namespace tail;

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(8) << 20;  // 8 MiB per device
constexpr int NOALLOC_MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

struct NoallocDevice {
  std::atomic<int> ready;   // 1 once setup on this device succeeded
  std::atomic<int> pdl_ok;  // 0 once a launch with programmatic serialization was refused
  uint8_t* base;            // device address of g_noalloc_scratch on this device
  int num_sms;
  int max_dyn;              // dynamic shared memory the lm_head kernels may use
};

NoallocDevice g_dev[NOALLOC_MAX_DEVICES];
std::mutex g_setup_mutex;

// One-time setup of device `dev` (the caller's current device).
int setup_device(int dev, NoallocDevice** out) {
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) {
    set_last_error("tail_run_noalloc: device ordinal beyond the 64 devices it keeps state for");
    return TAIL_ERR_UNSUPPORTED;
  }
  NoallocDevice& d = g_dev[dev];
  if (d.ready.load(std::memory_order_acquire)) {
    *out = &d;
    return TAIL_OK;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!d.ready.load(std::memory_order_relaxed)) {
    int major = 0, minor = 0, sms = 0, optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail(e, "tail_run_noalloc: cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) {
      set_last_error("tail_run_noalloc: the current device is not an sm_103 device");
      return TAIL_ERR_UNSUPPORTED;
    }
    void* base = nullptr;
    e = cudaGetSymbolAddress(&base, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "tail_run_noalloc: cudaGetSymbolAddress of the static scratch");
    if (!base || !aligned(base, 256)) {
      set_last_error("tail_run_noalloc: the static scratch has no usable device address");
      return TAIL_ERR_CUDA;
    }
    int max_dyn = 0;
    e = prepare_gemv(optin, &max_dyn);
    if (e != cudaSuccess) return cuda_fail(e, "tail_run_noalloc: cudaFuncSetAttribute (shared memory opt-in)");
    d.base = static_cast<uint8_t*>(base);
    d.num_sms = sms;
    d.max_dyn = max_dyn;
    d.pdl_ok.store(1, std::memory_order_relaxed);
    d.ready.store(1, std::memory_order_release);
  }
  *out = &d;
  return TAIL_OK;
}

// Launches with programmatic dependent launch while the device takes it.  A
// launch that fails with the attribute is retried once without it; only when
// that retry succeeds (the attribute was what the runtime refused) does the
// device stop using it.  Any other failure is returned as it is.
template <typename Launch>
cudaError_t launch_with_pdl_fallback(NoallocDevice* d, Launch launch) {
  if (!d->pdl_ok.load(std::memory_order_relaxed)) return launch(false);
  cudaError_t e = launch(true);
  if (e == cudaSuccess) return e;
  cudaGetLastError();  // a refused launch leaves a (non-sticky) error behind
  const cudaError_t e2 = launch(false);
  if (e2 == cudaSuccess) d->pdl_ok.store(0, std::memory_order_relaxed);
  return e2 == cudaSuccess ? e2 : e;
}

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte offsets of one pass's scratch inside the static array.
struct Layout {
  size_t err, rsync, apack, row_scale, meta, cand, lscr, tkv, tki, total;
};

// Scratch of a pass of B rows under `plan`; the first 256 bytes hold the error
// word (offset 8), the per-row arrival words follow; everything before `apack`
// starts each call at zero.  The logits staging is left out when the caller's
// logits serve the row owners' rescans (has_out) and the slab logits stay in
// shared memory.
Layout layout_for(const GemvPlan& plan, int B, int H, int V, int K, int nslab, bool has_out) {
  Layout L = {};
  size_t o = 0;
  L.err = 8;
  o = 256;
  L.rsync = o;  // arrivals [B], then copies [B]
  o += up256(static_cast<size_t>(B) * 16);
  L.apack = o;
  o += up256(static_cast<size_t>(H / KSTEP) * plan.mt * APACK_TILE_BYTES);
  L.row_scale = o;
  o += up256(static_cast<size_t>(plan.mt) * MTILE_ROWS * 4);
  L.meta = o;
  o += up256(static_cast<size_t>(B) * nslab * SLAB_META_WORDS * 4);
  L.cand = o;
  o += up256(static_cast<size_t>(B) * nslab * SLAB_CAND * 8);
  L.lscr = o;
  if (!has_out || !plan.logits_in_smem) o += up256(static_cast<size_t>(B) * V * 4);
  L.tkv = o;
  o += up256(static_cast<size_t>(B) * K * 4);
  L.tki = o;
  o += up256(static_cast<size_t>(B) * K * 4);
  L.total = o;
  return L;
}

}  // namespace

extern "C" int tail_run_noalloc(const tail_config* cfg, const void* hidden, const float* gamma,
                                const uint16_t* w_t, const float* params, int32_t n_param_cols, int32_t gbs,
                                int32_t* out_tokens, float* out_logits_opt, int32_t* out_status_opt,
                                void* stream) {
  int rc = validate_config(cfg);
  if (rc == TAIL_ERR_UNSUPPORTED)
    set_last_error("tail_run_noalloc: H and V must be multiples of 16 and H * V below 2^40");
  if (rc) return rc;
  if (gbs < 0 || gbs > cfg->gbs_max) return TAIL_ERR_INVALID_ARG;
  if (gbs == 0) return TAIL_OK;
  if (!hidden || !gamma || !w_t) return TAIL_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(w_t, 16) || !aligned(gamma, 4)) return TAIL_ERR_INVALID_ARG;
  if (params) {
    if (n_param_cols != 3 && n_param_cols != 4) return TAIL_ERR_INVALID_ARG;
    if (!out_tokens || !aligned(params, 4) || !aligned(out_tokens, 4)) return TAIL_ERR_INVALID_ARG;
  }
  if (out_logits_opt && !aligned(out_logits_opt, 16)) return TAIL_ERR_INVALID_ARG;
  if (out_status_opt && !aligned(out_status_opt, 4)) return TAIL_ERR_INVALID_ARG;

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "tail_run_noalloc: cudaGetDevice");
  NoallocDevice* d = nullptr;
  rc = setup_device(dev, &d);
  if (rc) return rc;

  const int H = cfg->H, V = cfg->V, K = cfg->k;
  const int Hu = cfg->hidden_actual <= 0 ? H : cfg->hidden_actual;
  const int64_t npairs = V / 16;
  const int nslab = slab_count(npairs, d->num_sms, MAX_SLABS);
  if ((npairs + nslab - 1) / nslab * 16 > 32 * SEL_NPL) {
    set_last_error("tail_run_noalloc: vocabulary slabs wider than the slab select holds");
    return TAIL_ERR_UNSUPPORTED;
  }

  // Rows per pass: the most (up to 64) whose plan is valid and whose scratch fits the static array.
  const bool has_out = out_logits_opt != nullptr;
  const int rmax = gbs < MAX_ROWS_PER_PASS ? gbs : MAX_ROWS_PER_PASS;
  int R = 0;
  size_t need1 = 0;
  for (int r = rmax; r >= 1; --r) {
    const GemvPlan p = plan_gemv(r, H, V, K, nslab, d->max_dyn);
    const size_t need = layout_for(p, r, H, V, K, nslab, has_out).total;
    if (r == 1) need1 = need;
    if (p.ok && need <= NOALLOC_SCRATCH_BYTES) {
      R = r;
      break;
    }
  }
  if (R == 0) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "tail_run_noalloc: one row needs %zu bytes of scratch (or has no shared-memory plan); "
             "the static scratch holds %zu bytes",
             need1, NOALLOC_SCRATCH_BYTES);
    set_last_error(msg);
    return TAIL_ERR_UNSUPPORTED;
  }
  const int rem = gbs % R;
  if (rem) {
    const GemvPlan p = plan_gemv(rem, H, V, K, nslab, d->max_dyn);
    if (!p.ok || layout_for(p, rem, H, V, K, nslab, has_out).total > NOALLOC_SCRATCH_BYTES) {
      set_last_error("tail_run_noalloc: the last pass of the batch has no plan that fits the static scratch");
      return TAIL_ERR_UNSUPPORTED;
    }
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = d->base;
  // The error word and the per-row arrival words must start at zero: a call
  // interrupted by a device error may leave them nonzero.
  const size_t zero_bytes = layout_for(plan_gemv(R, H, V, K, nslab, d->max_dyn), R, H, V, K, nslab, has_out).apack;
  e = cudaMemsetAsync(base, 0, zero_bytes, s);
  if (e != cudaSuccess) return cuda_fail(e, "tail_run_noalloc: cudaMemsetAsync");

  const int sz = elem_bytes(cfg->hidden_dtype);
  for (int r0 = 0; r0 < gbs; r0 += R) {
    const int B = gbs - r0 < R ? gbs - r0 : R;
    const GemvPlan plan = plan_gemv(B, H, V, K, nslab, d->max_dyn);
    const Layout L = layout_for(plan, B, H, V, K, nslab, has_out);

    RmsArgs ra;
    ra.hidden = static_cast<const uint8_t*>(hidden) + static_cast<int64_t>(r0) * H * sz;
    ra.dtype = cfg->hidden_dtype;
    ra.gamma = gamma;
    ra.B = B;
    ra.mt = plan.mt;
    ra.B_pad = plan.mt * MTILE_ROWS;
    ra.H = H;
    ra.Hu = Hu;
    ra.eps = cfg->eps;
    ra.zero_pad = cfg->zero_interleaved_pad ? 1 : 0;
    ra.deferred = cfg->deferred_rms ? 1 : 0;
    ra.apack = reinterpret_cast<uint32_t*>(base + L.apack);
    ra.row_scale = reinterpret_cast<float*>(base + L.row_scale);
    const bool fused = cfg->deferred_rms && plan.logits_in_smem && plan.mt <= FUSED_MAX_MT;
    if (!fused) {
      e = launch_with_pdl_fallback(d, [&](bool pdl) { return launch_rms_pack(ra, s, pdl); });
      if (e != cudaSuccess) return cuda_fail(e, "tail_run_noalloc: kernel launch");
    }

    GemvArgs ga;
    ga.w = w_t;
    ga.apack = base + L.apack;
    ga.row_scale = reinterpret_cast<const float*>(base + L.row_scale);
    ga.fused = fused ? 1 : 0;
    ga.hidden = ra.hidden;
    ga.dtype = cfg->hidden_dtype;
    ga.gamma = gamma;
    ga.Hu = Hu;
    ga.eps = cfg->eps;
    ga.zero_pad = ra.zero_pad;
    ga.logits_out = out_logits_opt ? out_logits_opt + static_cast<int64_t>(r0) * V : nullptr;
    ga.logits_out_ld = V;
    ga.logits_scratch = (has_out && plan.logits_in_smem) ? nullptr : reinterpret_cast<float*>(base + L.lscr);
    ga.meta = reinterpret_cast<uint32_t*>(base + L.meta);
    ga.cand = reinterpret_cast<uint64_t*>(base + L.cand);
    ga.row_sync = reinterpret_cast<unsigned long long*>(base + L.rsync);
    ga.row_copy = ga.row_sync + B;
    ga.topk_val = reinterpret_cast<float*>(base + L.tkv);
    ga.topk_idx = reinterpret_cast<int32_t*>(base + L.tki);
    ga.topk_ld = K;
    ga.params = params ? params + static_cast<int64_t>(r0) * n_param_cols : nullptr;
    ga.ncols = n_param_cols;
    ga.tokens = params ? out_tokens + r0 : nullptr;
    ga.err = reinterpret_cast<int*>(base + L.err);
    ga.B = B;
    ga.H = H;
    ga.V = V;
    ga.K = K;
    ga.ksteps = H / KSTEP;
    ga.mt = plan.mt;
    ga.nslab = nslab;
    ga.npairs = npairs;
    ga.cb_pairs = plan.cb_pairs;
    ga.kpb = plan.kpb;
    ga.pitch = plan.pitch;
    ga.stage_bytes = plan.stage_bytes;
    ga.nstages = plan.nstages;
    ga.logits_in_smem = plan.logits_in_smem;
    ga.max_slab_cols = plan.max_slab_cols;
    ga.smem_bytes = plan.smem_bytes;
    ga.capc = plan.capc;
    ga.sortP = plan.sortP;
    ga.timeout_ns = DEFAULT_TIMEOUT_NS;
    ga.drop_iter = -1;
    e = launch_with_pdl_fallback(d, [&](bool pdl) { return launch_gemv(ga, s, pdl); });
    if (e != cudaSuccess) return cuda_fail(e, "tail_run_noalloc: kernel launch");
  }
  if (out_status_opt) {
    e = cudaMemcpyAsync(out_status_opt, base + 8, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "tail_run_noalloc: cudaMemcpyAsync of the status word");
  }
  return TAIL_OK;
}
