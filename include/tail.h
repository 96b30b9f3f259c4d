/*
 * decode_sampling_tail_gb300: the GPT-OSS decode sampling tail on one GB300.
 *
 * One call runs the whole tail for a batch of gbs rows:
 *   final RMSNorm -> bf16 lm_head -> global top-k -> sampler -> one token per row.
 *
 * The operation is the one defined by "GPT-OSS Tail Chunked Megakernel Kernel
 * API Reference" (nkilib.experimental.gpt_oss_tail, function
 * gpt_oss_tail_chunked_megakernel): section "Background" names the four steps;
 * the parameter entries `hidden_states`, `gamma`, `lm_head_weight_t`, `eps`,
 * `hidden_actual`, `zero_interleaved_pad`, `k`, `emit_logits`,
 * `sampling_params` and `deferred_rms` define the inputs, options and outputs
 * mirrored below.  On one GPU the whole vocabulary is local (V_s = V).  The
 * page's vocabulary-parallel deployment (a slice per rank, one exchange, row
 * ownership) is served by tail_merge_shards below, with the exchange left to
 * the caller (the Python module decode_sampling_tail_gb300.vocab_parallel
 * does it with torch.distributed); the page's bf16 logits mirror and its
 * multi-hop meshes have no counterpart here.
 *
 * Conventions for every entry point:
 *   - Device pointers are caller-owned memory on the handle's device.  The
 *     library owns only its scratch, sized at create time from gbs_max.
 *   - Runs are asynchronous on the caller's stream (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).  No host synchronisation
 *     happens except in tail_run_host, tail_check and tail_destroy.
 *   - One run per handle at a time: concurrent runs on one handle share its
 *     scratch and race.
 *   - The weights are read from the start of a launch, before its dependency
 *     wait on the previous kernel of the stream (programmatic dependent
 *     launch): w_t on every path, gamma too on the small path.  A kernel that
 *     writes them must be ordered before the run by more than stream order
 *     (an event, or a synchronisation); the hidden rows, the parameters and
 *     the outputs follow stream order.
 *   - Every call returns TAIL_OK (0) or a negative tail_status.  Nothing
 *     aborts, traps or prints.
 */
#ifndef DECODE_SAMPLING_TAIL_GB300_TAIL_H
#define DECODE_SAMPLING_TAIL_GB300_TAIL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tail_s tail_t;

/* Element type of `hidden` (parameter `hidden_states`: fp32, fp16 or bf16). */
typedef enum { TAIL_F32 = 0, TAIL_F16 = 1, TAIL_BF16 = 2 } tail_dtype;

typedef enum {
  TAIL_OK = 0,
  TAIL_ERR_INVALID_ARG = -1,  /* null/misaligned pointer, bad size, gbs > gbs_max, bad n_param_cols */
  TAIL_ERR_UNSUPPORTED = -2,  /* shape, dtype or device the library cannot run: caller falls back */
  TAIL_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed */
  TAIL_ERR_OOM = -4,          /* scratch allocation failed at create */
  TAIL_ERR_DEVICE = -5        /* a kernel raised its error flag (a bounded wait ran out) */
} tail_status;

typedef struct {
  int32_t H;                    /* stored hidden width: row length of hidden, rows of w_t; H % 16 == 0 */
  int32_t hidden_actual;        /* H_u, the unpadded hidden; <= 0 means H; 1 <= H_u <= H */
  int32_t V;                    /* vocabulary: columns of w_t; V % 16 == 0 */
  int32_t k;                    /* candidates kept by the global top-k: 1 <= k <= min(V, 1024) */
  int32_t gbs_max;              /* largest gbs a run may pass: 1 .. 4096 */
  float eps;                    /* added to the mean of squares under the root; GPT-OSS: 1e-5 */
  int32_t hidden_dtype;         /* tail_dtype of hidden */
  int32_t zero_interleaved_pad; /* 1: pad lanes are zero in hidden, gamma and w_t wherever they sit,
                                      so all H lanes are summed; 0: lanes [H_u, H) are ignored */
  int32_t deferred_rms;         /* 1 (default): rstd scales the GEMM output per row;
                                   0: legacy form, (x * rstd) * gamma feeds the GEMM */
  int32_t path;                 /* tail_path: which lm_head serves which batch sizes (no page
                                   counterpart: both compute the same logits, within the
                                   logit tolerance).  Ignored by tail_run_noalloc. */
} tail_config;

/*
 * lm_head realisations.  The mma.sync kernel streams W once for up
 * to 8 rows and fuses the top-k and the sampler; it issues one bulk copy per
 * W row per CTA, so a narrow vocabulary leaves it bound by the copy engine's
 * request rate (a 256 x 4096 weight takes ~35 us a step).  The tensor-core
 * path (split, tcgen05 lm_head with per-tile candidate lists, merge +
 * sampler) serves any batch in one pass.  The small path is one launch of
 * CUDA-core arithmetic for problems bound by latency: each CTA forms the
 * activations (fp32, no bf16 rounding) and the fp32 logits of a vocabulary
 * slab with plain loads, and CTA b then keeps row b's exact top k over all V
 * logits and draws its token.
 */
typedef enum {
  TAIL_PATH_AUTO = 0,   /* tensor cores for every batch when V <= TAIL_TC_ALL_ROWS_MAX_V,
                           else as TAIL_PATH_GEMV */
  TAIL_PATH_GEMV = 1,   /* mma.sync kernel for gbs <= 8, tensor cores for gbs >= 9 */
  TAIL_PATH_TENSOR = 2, /* tensor cores for every batch (TAIL_ERR_UNSUPPORTED at create
                           when the merge cannot be planned for k and V) */
  TAIL_PATH_SMALL = 3   /* the one-launch small path for every batch: TAIL_ERR_UNSUPPORTED at
                           create unless gbs_max <= 8, H <= 8192, V <= 16384 and one CTA's
                           shared memory holds gbs_max x (H + 4096) fp32 values and a row's
                           V keys and indices.  No stage-1 taps (tail_tap_shape and
                           tail_run_taps return TAIL_ERR_UNSUPPORTED); tail_run_moe forms h
                           with a kernel of its own first. */
} tail_path;

#define TAIL_TC_ALL_ROWS_MAX_V 131072

/* Static facts about a handle, for benchmarks and tests. */
typedef struct {
  int32_t num_sms;          /* SMs of the device */
  int32_t nslab;            /* vocabulary slabs = CTAs of the lm_head kernel */
  int32_t merge_groups;     /* 0: the top-k merge runs inside the lm_head launch */
  int32_t lmhead_path;      /* 1: mma.sync lm_head + top-k + sampler launch;
                               2: the same, launched with programmatic serialization (it overlaps
                               the previous kernel on the stream until its dependency wait);
                               3: the one-launch small path (TAIL_PATH_SMALL) */
  int32_t rows_per_pass;    /* rows one mma.sync lm_head pass covers (the small path: gbs_max) */
  int32_t kernels_per_run;  /* kernel launches of one full pass on the mma.sync path: 1 when the
                               lm_head kernel forms the deferred-RMSNorm activations itself (up to
                               16 rows whose slab logits fit in shared memory), else 2 (RMSNorm
                               kernel + lm_head); 1 on the small path */
  int64_t scratch_bytes;    /* device scratch owned by the handle */
  int32_t tc_min_rows;      /* runs with gbs >= this take the tensor-core path (split, tcgen05
                               lm_head with per-tile candidate lists, merge + sampler: 3 kernels,
                               one pass): 1 or 9 by cfg.path; 0 when gbs_max is below it */
} tail_info;

/*
 * Create a handle on CUDA device `device`; validates the config and allocates
 * the scratch (activation pack, per-row scale, top-k candidates, logits
 * staging, error flag).  The caller's current device is restored on return.
 * Returns TAIL_ERR_INVALID_ARG for a bad config, TAIL_ERR_UNSUPPORTED when the
 * device is not sm_103, TAIL_ERR_OOM when scratch cannot be allocated.
 */
int tail_create(const tail_config* cfg, int device, tail_t** out);

/*
 * One decode step of the tail.
 *   hidden         [gbs, H] row-major, element type cfg.hidden_dtype, 16-byte aligned.
 *                  16-bit inputs are widened exactly to fp32 (`hidden_states`).
 *   gamma          [H] fp32 final RMSNorm weight (`gamma`).
 *   w_t            [H, V] bf16 bit patterns, C-contiguous, V fastest (`lm_head_weight_t`),
 *                  16-byte aligned.  Read once per step; never modified.
 *   params         [gbs, n_param_cols] fp32 rows [top_k, top_p, temperature(, u)]
 *                  (`sampling_params`), or NULL: no draw is made and
 *                  out_tokens is not written.  n_param_cols is 3 (u = 0.5) or 4.
 *   gbs            rows in this call, 0 <= gbs <= gbs_max (0 is a no-op).
 *   out_tokens     [gbs] int32 sampled vocabulary ids (may be NULL only if params is NULL).
 *   out_logits_opt [gbs, V] fp32 logits, or NULL (`emit_logits` off).
 * Inputs must not alias outputs.  Results are deterministic: repeated runs on
 * the same inputs give bitwise-equal outputs.  NaN inputs are outside the
 * method's domain (`skip_nan_fold`); +-inf logits are ordered normally.
 */
int tail_run(tail_t* h, const void* hidden, const float* gamma, const uint16_t* w_t,
             const float* params, int32_t n_param_cols, int32_t gbs, int32_t* out_tokens,
             float* out_logits_opt, void* stream);

/*
 * Weight preparation for the tensor-core path (`lm_head_weight_t` is read once
 * a step; its layout may be chosen once, when the model is loaded).  Makes a
 * handle-owned copy of w_t ([H, V] bf16, 16-byte aligned) in the layout of the
 * tensor-core lm_head's shared-memory weight stages: 8 KB blocks of 64 k-rows x
 * 64 columns with the 128-byte swizzle, k-block major, zero past H and V
 * (tail_info.scratch_bytes grows by ceil(H/64) * ceil(V/64) * 8 KB).  The copy
 * is written by a kernel on `stream`: runs on other streams must be ordered
 * after it by the caller, and runs still reading an earlier copy must have
 * finished before it is rewritten (a release with w_t = NULL synchronises).
 * From then on, runs of this handle that take the tensor-core path
 * (gbs >= tail_info.tc_min_rows) and pass the same w_t pointer read the copy:
 * one bulk copy per weight stage instead of one tensor-tile load per 64-column
 * box.  Results are bitwise those of the unprepared weight.  Runs with another
 * w_t pointer, and the mma.sync path, read w_t itself.  The copy is not
 * refreshed: after changing the contents of w_t, call this again (or stop
 * using the copy with w_t = NULL, which frees it).
 * Does nothing (and returns TAIL_OK) on a handle without a tensor-core path.
 * Returns TAIL_ERR_INVALID_ARG for a misaligned w_t, TAIL_ERR_OOM when the copy
 * cannot be allocated.
 */
int tail_prepare_weight(tail_t* h, const uint16_t* w_t, void* stream);

/*
 * tail_run plus the sorted global top-k (the merge's output, the stage that
 * feeds the sampler; the first stage's output is tail_run_taps'):
 *   out_topk_vals_opt [gbs, k] fp32 logits in (value desc, index asc) order, or NULL;
 *   out_topk_idx_opt  [gbs, k] int32 vocabulary ids in the same order, or NULL.
 */
int tail_run_ex(tail_t* h, const void* hidden, const float* gamma, const uint16_t* w_t,
                const float* params, int32_t n_param_cols, int32_t gbs, int32_t* out_tokens,
                float* out_logits_opt, float* out_topk_vals_opt, int32_t* out_topk_idx_opt,
                void* stream);

/*
 * Stage-1 taps (the page's `debug_taps`: the chunked top-k's first-stage
 * output, for defects that show on hardware only).  The vocabulary is cut
 * into chunks -- the mma.sync lm_head kernel's slabs, or the tensor-core
 * lm_head's column tiles -- and each (row, chunk) hands the merge a few
 * candidates (section "Background": the chunked top-k feeds one global top-k).
 *
 * tail_tap_shape: for a run of gbs rows on this handle, *kind = 1 (slabs) or
 * 2 (tiles), *n_chunks chunks a row, *cap candidate slots a chunk, and, when
 * chunk_lo_host_opt is non-NULL, the first vocabulary id of every chunk and V
 * after them ([n_chunks + 1] int32, host memory).
 *
 * tail_run_taps: tail_run_ex, then the taps of the same run (device memory):
 *   tap_vals  [gbs, n_chunks, cap] fp32: the chunk's candidates' logits (slots
 *             past the count hold -inf),
 *   tap_idx   [gbs, n_chunks, cap] int32: their vocabulary ids (-1 past the count),
 *   tap_count [gbs, n_chunks] int32: candidates handed over,
 *   tap_bound [gbs, n_chunks] fp32: every element of the chunk that is not a
 *             candidate has a logit <= bound.  Slabs: the candidates are every
 *             element >= bound when they fit the chunk's slots; when they do not,
 *             count = 0 and bound = +inf (the merge then rescans the slab if its
 *             hidden elements could reach the top k).  Tiles: the tile's top
 *             `cap` by (value desc, index asc); bound = the last of them, or -inf
 *             when they are all of the tile's columns.
 * Candidates are listed in no particular order for slabs, in (value desc, index
 * asc) order for tiles.  One extra kernel launch copies them out of the
 * handle's scratch after the run.  Returns TAIL_ERR_INVALID_ARG for a NULL tap
 * pointer (any of the four) or misaligned pointers.
 */
int tail_tap_shape(const tail_t* h, int32_t gbs, int32_t* kind, int32_t* n_chunks, int32_t* cap,
                   int32_t* chunk_lo_host_opt);
int tail_run_taps(tail_t* h, const void* hidden, const float* gamma, const uint16_t* w_t, const float* params,
                  int32_t n_param_cols, int32_t gbs, int32_t* out_tokens, float* out_logits_opt,
                  float* out_topk_vals_opt, int32_t* out_topk_idx_opt, float* tap_vals, int32_t* tap_idx,
                  int32_t* tap_count, float* tap_bound, void* stream);

/*
 * The tail fused with its producer: the MoE combine and residual add that form
 * the bf16 hidden state ("nemotron CUDA: RMSNorm rows run on the shared norms
 * and combine (#548, step 1)", TensorFold pull request #1353, section "What
 * moves", entry tf_nemo_add_moe_norm / tf_moe_add_rms_rows_bf16h, and its
 * author's fix reply: the fused residual keeps the routed chain and the shared
 * sum apart; "GPT-OSS Tail Chunked Megakernel Kernel API Reference", parameter
 * `hidden_states`: a 16-bit producer output feeds the norm directly).  For
 * every row b and hidden lane j:
 *   r  = 0;  r  = fp32 fma(slot_w[b][s], slots[b][s][j], r)  for s = 0 .. n_routed-1
 *   sh = 0;  sh = fp32 fma(slot_w[b][s], slots[b][s][j], sh) for s = n_routed .. nslots-1
 *   h[b][j] = bf16(residual[b][j] + bf16(r + sh))      (bf16: nearest, ties to even)
 * (Nemotron: 6 routed slots, then 2 shared slots of weight 1, whose chain is
 * the plain sum s0 + s1), then the tail of tail_run_ex on h.  Requires
 * cfg.hidden_dtype == TAIL_BF16.
 *   residual       [gbs, H] bf16 bit patterns, 16-byte aligned.
 *   slots          [gbs, nslots, H] expert outputs, fp32 (slot_dtype TAIL_F32) or bf16
 *                  bit patterns (TAIL_BF16), 4-byte aligned; may be NULL when nslots == 0.
 *   nslots         0 .. TAIL_MOE_MAX_SLOTS.
 *   n_routed       0 .. nslots: the leading slots that form the routed chain; the
 *                  others are shared (n_routed == nslots: no shared slot).
 *   slot_w         [gbs, nslots] fp32 weights, 4-byte aligned.
 *   out_hidden_opt [gbs, H] bf16 h, 16-byte aligned, or NULL.
 * The other arguments are those of tail_run_ex.  Launches: the tail's own
 * (h is formed inside its first kernel: on the tensor-core path by the
 * RMSNorm split for H <= 24576; on the mma.sync path by the lm_head kernel's
 * activation warp in the deferred form, for up to 8 slots whose pointer is
 * 16-byte aligned).  Otherwise one more kernel forms h first (into
 * out_hidden_opt, else the handle's scratch), chained with programmatic
 * dependent launch.  h is bitwise the same either way.  Returns
 * TAIL_ERR_UNSUPPORTED for a non-bf16 config, TAIL_ERR_INVALID_ARG for bad
 * pointers, alignment, sizes, slot counts or slot dtype.
 */
#define TAIL_MOE_MAX_SLOTS 256
int tail_run_moe(tail_t* h, const uint16_t* residual, const void* slots, int32_t slot_dtype, int32_t nslots,
                 int32_t n_routed, const float* slot_w, const float* gamma, const uint16_t* w_t,
                 const float* params, int32_t n_param_cols, int32_t gbs, int32_t* out_tokens,
                 float* out_logits_opt, float* out_topk_vals_opt, int32_t* out_topk_idx_opt,
                 uint16_t* out_hidden_opt, void* stream);

/*
 * End-to-end form for callers holding the per-step inputs in host memory:
 * copies hidden_host [gbs, H] into handle-owned device staging, runs the tail
 * on `stream`, brings the tokens (and the logits, when out_logits_host_opt is
 * non-NULL) back to host memory and synchronises the stream before returning.
 * params_host [gbs, n_param_cols] is copied to device staging too, unless it
 * is pinned (page-locked and mapped, as cudaHostAlloc memory is): the kernels
 * then read it in place.  The kernels write the tokens into a handle-owned
 * pinned, mapped buffer (made at the first call; a device buffer and a copy if
 * that allocation fails), copied to out_tokens_host after the synchronisation.
 * gamma and w_t stay device pointers (model weights are resident).  Pinned host
 * buffers make the copies asynchronous; pageable ones work too.
 */
int tail_run_host(tail_t* h, const void* hidden_host, const float* gamma, const uint16_t* w_t,
                  const float* params_host, int32_t n_param_cols, int32_t gbs,
                  int32_t* out_tokens_host, float* out_logits_host_opt, void* stream);

/*
 * Allocation-free form of tail_run, for callers that must not allocate device
 * memory: a serving runtime that hands nearly all of HBM to its own pools up
 * front and refuses any cudaMalloc behind its back, code that cannot keep a
 * handle alive between steps (an op or plugin called without lifetime hooks),
 * or a decode loop that cannot afford the device-wide synchronisation that
 * cudaMalloc and cudaFree may imply.  The page has no counterpart: it is a
 * calling convention of this library, not a step of the method.
 *
 * It runs the same kernels and gives the same results as tail_run with the
 * same config (bitwise equal when gbs <= 8 at GPT-OSS sizes; larger batches
 * run as several passes and agree within the logit tolerance).  Instead of
 * handle scratch it uses one static device array of 8 MiB per device, part of
 * this library's device image; no call allocates, frees or calls a routine
 * that allocates.
 *   cfg            the config tail_create would take (validated on every call);
 *                  gbs <= cfg->gbs_max.
 *   device         the caller's current CUDA device; `stream` must belong to it.
 *   hidden ... out_logits_opt, stream: as in tail_run.
 *   out_status_opt device int32, or NULL: receives (in stream order, after
 *                  the call's last kernel) 0, or the nonzero code of a
 *                  bounded device wait that ran out, in which case the
 *                  outputs are undefined.
 * Size limit: one pass of B rows needs, each part rounded up to 256 bytes,
 * 256 (error word) + 16 * B (per-row arrival and copy words)
 * + 32 * H * mt (activation pack; mt = 1,
 * 2, 4 or 8 for B up to 8, 16, 32, 64) + 32 * mt (row scales)
 * + 32 * B * nslab (per-slab publications) + 256 * B * nslab (published
 * candidates) + 8 * B * k (top-k staging) + 4 * B * V (logits staging,
 * left out when out_logits_opt is given and a slab's logits fit in shared
 * memory) bytes, nslab being the vocabulary slab count (min(SMs, V / 128),
 * at least 1).  Batches run in passes of as many rows (at most 64) as fit in
 * 8 MiB.  At H = 2880, V = 201088, k = 256 that is 9 rows per pass.  When
 * not even one row fits, the call returns
 * TAIL_ERR_UNSUPPORTED before launching anything, and tail_last_error()
 * states the bytes needed and the 8 MiB limit.
 * Zeroing: every call clears the error word and the per-row arrival words
 * with one cudaMemsetAsync on `stream`; the rest of the
 * scratch is fully written by the kernels before it is read.
 * First call on a device: sets up that device (looks up the static array's
 * address with cudaGetSymbolAddress, which loads the library's device image
 * if it is not loaded yet, and opts the lm_head kernels into their shared
 * memory size).  Make it once before any stream capture on that device.
 * The set-up is kept for the life of the process: after a reset of the
 * device's primary context (cudaDeviceReset, or the driver's own) the kept
 * address and attributes are stale, so this entry point must not be called
 * on that device again.
 * Overlapping calls race: all calls on one device share the one static
 * array, so two calls whose kernels may overlap (different streams, threads
 * or processes sharing a context, without ordering between them) corrupt
 * each other's results.  Serialise them on one stream.  Handles created with
 * tail_create own separate scratch and do not race with this call.
 */
int tail_run_noalloc(const tail_config* cfg, const void* hidden, const float* gamma, const uint16_t* w_t,
                     const float* params, int32_t n_param_cols, int32_t gbs, int32_t* out_tokens,
                     float* out_logits_opt, int32_t* out_status_opt, void* stream);

/*
 * Vocabulary-parallel tail: the merge step.  With the vocabulary split into
 * nshard contiguous slices (one per rank, as in the page's deployment; section
 * "Background": each rank's chunked top-k, then one top-k over the union), a
 * rank runs tail_run_ex on its own slice (a handle created with V = the slice
 * width, `w_t` its [H, V_s] columns, params NULL) to get its sorted top-k; the
 * ranks exchange those (k candidates per row each: values and slice-local
 * ids); this call then merges them on the current device and stream:
 *   cand_vals      [nshard][gbs][k_in] fp32, each shard's top-k values (device).
 *   cand_idx       [nshard][gbs][k_in] int32, their ids within the shard (device).
 *   shard_offsets  [nshard] int32 (host): the first global vocabulary id of each shard.
 *   k              the global top-k size, 1 <= k <= min(nshard * k_in, 1024);
 *                  exact when every shard passed its top k (k_in >= k).
 *   params, n_param_cols, out_tokens: as in tail_run (params NULL: no draw).
 *   out_topk_vals_opt / out_topk_idx_opt: [gbs][k] the merged top-k in
 *                  (value desc, global id asc) order, or NULL.
 * The result equals the unsharded tail's bitwise when the shards computed the
 * same fp32 logits (the lm_head's per-column arithmetic does not depend on how
 * the vocabulary is split).  nshard <= 64 and nshard * k_in <= 16384;
 * TAIL_ERR_UNSUPPORTED beyond.  No handle and no allocation.
 */
int tail_merge_shards(int32_t nshard, int32_t k_in, int32_t k, int32_t gbs, const float* cand_vals,
                      const int32_t* cand_idx, const int32_t* shard_offsets, const float* params,
                      int32_t n_param_cols, int32_t* out_tokens, float* out_topk_vals_opt,
                      int32_t* out_topk_idx_opt, void* stream);

/*
 * The calls below are the library's own plumbing (error reporting, timing, the
 * bound on device waits, a test hook, static facts, lifetime); no page defines
 * them.
 */

/*
 * Synchronises the handle's device work and reads the device error flag that
 * kernels raise when a bounded wait runs out.  Returns TAIL_ERR_DEVICE (and
 * clears the flag) if it was set, TAIL_ERR_CUDA on a sticky CUDA error, else
 * TAIL_OK.
 */
int tail_check(tail_t* h);

/*
 * Per-kernel device timing, for benchmarks.  While enabled, every run records
 * CUDA events on its stream before and after each of its kernel launches
 * (this gives up the programmatic overlap between the kernels, so enable it
 * only in a measuring loop of its own).  Enabling (again) starts a new
 * record of up to 256 lm_head passes.
 * tail_profile_read synchronises on the recorded events and returns, for the
 * passes recorded since enabling, the summed device milliseconds of each
 * kernel in kernel_ms[3] = {RMSNorm, lm_head, merge + sampler} and their count
 * in *passes.  On the mma.sync path the top-k and sampler run inside the
 * lm_head launch, so the third entry is 0.
 */
int tail_profile_enable(tail_t* h, int enable);
int tail_profile_read(tail_t* h, float* kernel_ms, int32_t* passes);

/*
 * Bounds every device-side wait of later runs to `ns` nanoseconds of GPU
 * global time (default 1e9).  A wait that runs out raises the device error
 * flag; the kernel stops issuing copies, waits (bounded) for the copies it
 * already issued, and returns; tail_check then reports TAIL_ERR_DEVICE.
 */
int tail_set_wait_limit(tail_t* h, uint64_t ns);

/*
 * Test hook for the bounded-wait path: while iteration >= 0, the lm_head
 * kernel of later runs never issues the copies of that ring iteration, so
 * the consumers' wait on it runs out after the wait limit (outputs of such a
 * run are undefined; nothing faults).  -1 turns the hook off.
 */
int tail_debug_drop_stage(tail_t* h, int32_t iteration);

/* Fills *out with the handle's static facts. */
int tail_get_info(const tail_t* h, tail_info* out);

/* Frees the handle and its scratch after synchronising its device.  NULL is a no-op. */
void tail_destroy(tail_t* h);

/* Static string for a status code. */
const char* tail_status_string(int status);

/* The CUDA call behind this thread's last TAIL_ERR_CUDA / TAIL_ERR_OOM, as text
   ("" when none); valid until the thread's next failing call. */
const char* tail_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_SAMPLING_TAIL_GB300_TAIL_H */
