/*
 * Plain, slow, fp64 CPU oracle of the GPT-OSS decode sampling tail.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Source of the method: "GPT-OSS Tail Chunked Megakernel Kernel API
 * Reference" (AWS Neuron NKI library, nkilib.experimental.gpt_oss_tail),
 * function gpt_oss_tail_chunked_megakernel.  Its "Background" section names
 * the four steps (final RMSNorm, lm_head, top-k, sampler); each function
 * below cites the parameter entry it follows.
 *
 * Every step is the plain definition, evaluated in double precision from the
 * exactly widened 16/32-bit inputs:
 *   widen      : bf16 / fp16 / fp32 bit patterns -> double (exact)
 *   rstd_b     = 1 / sqrt( (sum_h x_bh^2) / H_u + eps )
 *   logit_bv   = rstd_b * sum_h x_bh * gamma_h * W_hv
 *   top-k      = first k of all V columns sorted by (logit desc, index asc)
 *   sampler    = temperature, top-k, softmax, top-p, inverse-CDF draw
 * No blocking, fusion or reordering beyond what these definitions state.
 *
 * One producer step may precede the tail: the MoE combine and residual add
 * that forms the bf16 hidden state ("nemotron CUDA: RMSNorm rows run on the
 * shared norms and combine (#548, step 1)", TensorFold pull request #1353,
 * entry tf_nemo_add_moe_norm, with the routed chain and the shared sum kept
 * apart as its fix reply settles; oracle_moe_combine below).  Its precision
 * is fixed by that page (fp32 fmas and adds, bf16 roundings), so it is
 * evaluated in exactly those operations, not in double precision.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_F16 1
#define OR_BF16 2

int oracle_version(void) { return 1; }

/* ---------------------------------------------------------------------------
 * Widening.  Parameter `hidden_states`: fp32, fp16 or bf16 input; every fp16
 * and bf16 value is representable in fp32 (and every fp32 value in double),
 * so the conversion loses nothing and the oracle widens straight to double.
 * ------------------------------------------------------------------------- */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int f = bits & 0x3ff;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        mag = f ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

static double widen_one(const void *src, int dtype, int64_t i) {
    if (dtype == OR_F32) return (double)((const float *)src)[i];
    uint16_t b = ((const uint16_t *)src)[i];
    return dtype == OR_F16 ? oracle_f16_to_double(b) : oracle_bf16_to_double(b);
}

void oracle_widen(const void *src, int dtype, int64_t n, double *dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = widen_one(src, dtype, i);
}

/* ---------------------------------------------------------------------------
 * Final RMSNorm scale.  Parameters `eps`, `hidden_actual` and
 * `zero_interleaved_pad`.
 *   The mean of squares divides by H_u (the unpadded hidden), not by H.
 *   zero_pad = 1: the pad lanes are zero wherever they sit in [0, H), so the
 *                 sum runs over all H lanes.
 *   zero_pad = 0: lanes [H_u, H) are not part of the hidden state and are
 *                 ignored.
 *   eps is the fp32 value the caller passes, widened.
 * ------------------------------------------------------------------------- */
static int lane_active(int h, int Hu, int zero_pad) { return zero_pad ? 1 : (h < Hu); }

int oracle_rstd(const void *x, int dtype, int B, int H, int Hu, float eps, int zero_pad,
                double *rstd) {
    if (!x || !rstd || B < 0 || H <= 0 || Hu <= 0 || Hu > H) return -1;
    for (int b = 0; b < B; ++b) {
        double ss = 0.0;
        for (int h = 0; h < H; ++h) {
            if (!lane_active(h, Hu, zero_pad)) continue;
            double v = widen_one(x, dtype, (int64_t)b * H + h);
            ss += v * v;
        }
        rstd[b] = 1.0 / sqrt(ss / (double)Hu + (double)eps);
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * lm_head.  Parameters `lm_head_weight_t` ([H, V] bf16, already transposed,
 * C-contiguous) and `deferred_rms` (scaling each row before or after the
 * product gives the same value mathematically: the scale is one number per
 * row and the product is linear, so both realizations are this one formula):
 *   logit_bv = rstd_b * sum_h (x_bh * gamma_h) * W_hv
 * ------------------------------------------------------------------------- */
typedef struct {
    const double *a;   /* [B, H]: x * gamma, zero on ignored lanes */
    const double *rstd;
    const uint16_t *w; /* [H, V] bf16 */
    int B, H, V;
    int v0, v1;
    double *out;       /* [B, V] */
} logits_job;

static void *logits_worker(void *arg) {
    logits_job *j = (logits_job *)arg;
    const int n = j->v1 - j->v0;
    if (n <= 0) return NULL;
    double *acc = (double *)calloc((size_t)j->B * n, sizeof(double));
    double *wrow = (double *)malloc((size_t)n * sizeof(double));
    if (!acc || !wrow) {
        free(acc);
        free(wrow);
        return (void *)1;
    }
    for (int h = 0; h < j->H; ++h) {
        const uint16_t *src = j->w + (int64_t)h * j->V + j->v0;
        for (int v = 0; v < n; ++v) wrow[v] = oracle_bf16_to_double(src[v]);
        for (int b = 0; b < j->B; ++b) {
            const double ab = j->a[(int64_t)b * j->H + h];
            if (ab == 0.0) continue;
            double *dst = acc + (int64_t)b * n;
            for (int v = 0; v < n; ++v) dst[v] += ab * wrow[v];
        }
    }
    for (int b = 0; b < j->B; ++b)
        for (int v = 0; v < n; ++v)
            j->out[(int64_t)b * j->V + j->v0 + v] = j->rstd[b] * acc[(int64_t)b * n + v];
    free(acc);
    free(wrow);
    return NULL;
}

int oracle_logits(const void *x, int dtype, const float *gamma, const uint16_t *w_t, int B,
                  int H, int Hu, int V, float eps, int zero_pad, int nthreads,
                  double *logits) {
    if (!x || !gamma || !w_t || !logits || B < 0 || H <= 0 || V <= 0) return -1;
    if (B == 0) return 0;
    double *rstd = (double *)malloc((size_t)B * sizeof(double));
    double *a = (double *)malloc((size_t)B * H * sizeof(double));
    if (!rstd || !a) {
        free(rstd);
        free(a);
        return -2;
    }
    int rc = oracle_rstd(x, dtype, B, H, Hu, eps, zero_pad, rstd);
    if (rc) {
        free(rstd);
        free(a);
        return rc;
    }
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            a[(int64_t)b * H + h] = lane_active(h, Hu, zero_pad)
                                        ? widen_one(x, dtype, (int64_t)b * H + h) * (double)gamma[h]
                                        : 0.0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    /* Column blocks small enough that the accumulators stay in cache. */
    const int blk = 2048;
    const int nblk = (V + blk - 1) / blk;
    logits_job *jobs = (logits_job *)calloc((size_t)nblk, sizeof(logits_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        free(rstd);
        free(a);
        return -2;
    }
    for (int i = 0; i < nblk; ++i) {
        jobs[i].a = a;
        jobs[i].rstd = rstd;
        jobs[i].w = w_t;
        jobs[i].B = B;
        jobs[i].H = H;
        jobs[i].V = V;
        jobs[i].v0 = i * blk;
        jobs[i].v1 = (i + 1) * blk < V ? (i + 1) * blk : V;
        jobs[i].out = logits;
    }
    /* Waves of nthreads jobs each. */
    int failed = 0;
    for (int first = 0; first < nblk; first += nthreads) {
        int cnt = nblk - first < nthreads ? nblk - first : nthreads;
        for (int t = 0; t < cnt; ++t) pthread_create(&th[t], NULL, logits_worker, &jobs[first + t]);
        for (int t = 0; t < cnt; ++t) {
            void *r = NULL;
            pthread_join(th[t], &r);
            if (r) failed = 1;
        }
    }
    free(jobs);
    free(th);
    free(rstd);
    free(a);
    return failed ? -2 : 0;
}

/* ---------------------------------------------------------------------------
 * Global top-k.  "Background" (the kernel computes the global top-k over the
 * full vocabulary) and parameter `k`.  The order is (logit desc, index asc);
 * -0.0 and +0.0 compare equal, so they tie and fall back to the index.
 * NaN is outside the method's domain (parameter `skip_nan_fold`: the input is
 * the kernel's own finite GEMM output); +-inf order like any other value.
 * ------------------------------------------------------------------------- */
typedef struct {
    double v;
    int32_t i;
} vi_pair;

static int cmp_desc_then_index(const void *pa, const void *pb) {
    const vi_pair *a = (const vi_pair *)pa, *b = (const vi_pair *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

typedef struct {
    const double *logits;
    int V, k, r0, r1;
    double *vals;
    int32_t *idx;
    int fail;
} topk_job;

static void *topk_worker(void *arg) {
    topk_job *j = (topk_job *)arg;
    vi_pair *p = (vi_pair *)malloc((size_t)j->V * sizeof(vi_pair));
    if (!p) {
        j->fail = 1;
        return NULL;
    }
    for (int b = j->r0; b < j->r1; ++b) {
        const double *row = j->logits + (int64_t)b * j->V;
        for (int v = 0; v < j->V; ++v) {
            p[v].v = row[v];
            p[v].i = v;
        }
        qsort(p, (size_t)j->V, sizeof(vi_pair), cmp_desc_then_index);
        for (int t = 0; t < j->k; ++t) {
            j->vals[(int64_t)b * j->k + t] = p[t].v;
            j->idx[(int64_t)b * j->k + t] = p[t].i;
        }
    }
    free(p);
    return NULL;
}

int oracle_topk(const double *logits, int B, int V, int k, int nthreads, double *vals,
                int32_t *idx) {
    if (!logits || !vals || !idx || B < 0 || V <= 0 || k <= 0 || k > V) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B) nthreads = B > 0 ? B : 1;
    topk_job *jobs = (topk_job *)calloc((size_t)nthreads, sizeof(topk_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -2;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].logits = logits;
        jobs[t].V = V;
        jobs[t].k = k;
        jobs[t].r0 = (int)((int64_t)B * t / nthreads);
        jobs[t].r1 = (int)((int64_t)B * (t + 1) / nthreads);
        jobs[t].vals = vals;
        jobs[t].idx = idx;
        pthread_create(&th[t], NULL, topk_worker, &jobs[t]);
    }
    int fail = 0;
    for (int t = 0; t < nthreads; ++t) {
        pthread_join(th[t], NULL);
        fail |= jobs[t].fail;
    }
    free(jobs);
    free(th);
    return fail ? -2 : 0;
}

/* ---------------------------------------------------------------------------
 * Sampler.  Parameter `sampling_params`: per row [top_k, top_p, temperature]
 * and an optional 4th column u in [0, 1) that drives an inverse-CDF draw;
 * without it u is the fixed value 0.5.
 *
 * The page names the columns only.  The order of operations used here is the
 * standard nucleus-sampling one:
 *   1. kk = trunc(top_k) when 1 <= top_k < n + 1 (n: the candidates kept),
 *      else kk = n (the cut is disabled).
 *   2. temperature <= 0 (or NaN) or kk == 1: greedy, token = idx_0.
 *   3. s_i = (l_i - l_0) / T, e_i = exp(s_i), Z = sum_{i<kk} e_i, p_i = e_i/Z.
 *   4. top_p >= 1: m = kk; otherwise m = the smallest j+1 with
 *      sum_{i<=j} p_i >= top_p (so top_p <= 0 keeps one candidate).
 *   5. C_j = sum_{i<=j} e_i for j < m; the token is idx_j for the smallest j
 *      with u * C_{m-1} < C_j, and idx_{m-1} if there is none.
 * Outputs beyond the token (kk, m, the normalised CDF C_j / C_{m-1} and the
 * cumulative probabilities over kk) let a test judge how close a draw or a
 * top-p cut sits to a boundary.
 * ------------------------------------------------------------------------- */
int oracle_sample_row(const double *vals, const int32_t *idx, int n, const float *p4,
                      int ncols, int32_t *token, int32_t *kk_out, int32_t *m_out,
                      double *cdf_out, double *pcum_out) {
    if (!vals || !idx || !p4 || !token || n <= 0 || (ncols != 3 && ncols != 4)) return -1;
    const double top_k = (double)p4[0];
    const double top_p = (double)p4[1];
    const double temp = (double)p4[2];
    const double u = ncols == 4 ? (double)p4[3] : 0.5;

    /* top_k outside [1, n] (and NaN) disables the cut; compared as a double so
       that no out-of-range value is converted to an integer */
    long kk = (top_k >= 1.0 && top_k < (double)n + 1.0) ? (long)trunc(top_k) : (long)n;
    if (cdf_out)
        for (int i = 0; i < n; ++i) cdf_out[i] = 0.0;
    if (pcum_out)
        for (int i = 0; i < n; ++i) pcum_out[i] = 0.0;
    if (kk_out) *kk_out = (int32_t)kk;

    /* a temperature that is not positive (including NaN) means greedy */
    if (!(temp > 0.0) || kk == 1) {
        *token = idx[0];
        if (m_out) *m_out = 1;
        if (cdf_out) cdf_out[0] = 1.0;
        if (pcum_out) pcum_out[0] = 1.0;
        return 0;
    }
    double *e = (double *)malloc((size_t)kk * sizeof(double));
    if (!e) return -2;
    double Z = 0.0;
    for (long i = 0; i < kk; ++i) {
        e[i] = exp((vals[i] - vals[0]) / temp);
        Z += e[i];
    }
    long m = kk;
    double cum = 0.0;
    for (long j = 0; j < kk; ++j) {
        cum += e[j] / Z;
        if (pcum_out) pcum_out[j] = cum;
    }
    if (top_p < 1.0) {
        cum = 0.0;
        m = kk;
        for (long j = 0; j < kk; ++j) {
            cum += e[j] / Z;
            if (cum >= top_p) {
                m = j + 1;
                break;
            }
        }
    }
    double Cm = 0.0;
    for (long j = 0; j < m; ++j) Cm += e[j];
    const double target = u * Cm;
    long pick = -1;
    double C = 0.0;
    for (long j = 0; j < m; ++j) {
        C += e[j];
        if (cdf_out) cdf_out[j] = C / Cm;
        if (pick < 0 && target < C) pick = j;
    }
    if (pick < 0) pick = m - 1;
    *token = idx[pick];
    if (m_out) *m_out = (int32_t)m;
    free(e);
    return 0;
}

/* ---------------------------------------------------------------------------
 * The whole tail for B rows: logits, global top-k, sampler.  `params` may be
 * NULL (parameter `sampling_params`: without parameters there is no draw and
 * the call yields no token); then `tokens` is left untouched.
 * ------------------------------------------------------------------------- */
int oracle_tail(const void *x, int dtype, const float *gamma, const uint16_t *w_t, int B,
                int H, int Hu, int V, int k, float eps, int zero_pad, const float *params,
                int ncols, int nthreads, double *logits, double *topk_vals,
                int32_t *topk_idx, int32_t *tokens) {
    int rc = oracle_logits(x, dtype, gamma, w_t, B, H, Hu, V, eps, zero_pad, nthreads, logits);
    if (rc) return rc;
    rc = oracle_topk(logits, B, V, k, nthreads, topk_vals, topk_idx);
    if (rc) return rc;
    if (!params) return 0;
    for (int b = 0; b < B; ++b) {
        rc = oracle_sample_row(topk_vals + (int64_t)b * k, topk_idx + (int64_t)b * k, k,
                               params + (int64_t)b * ncols, ncols, tokens + b, NULL, NULL, NULL,
                               NULL);
        if (rc) return rc;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * MoE combine + residual add (the tail's producer).  Page: "nemotron CUDA:
 * RMSNorm rows run on the shared norms and combine (#548, step 1)" (TensorFold
 * pull request #1353): section "What moves", entry tf_nemo_add_moe_norm, and
 * the contract kinds moe_bf16_h / moe_f32_h, as settled by the author's fix
 * reply (commit 8e1115e05): the fused residual keeps the routed chain and the
 * shared sum apart.  For every hidden lane:
 *   r  = fp32 accumulator from 0, one fused multiply-add per ROUTED slot
 *        (slots 0 .. n_routed-1), in index order;
 *   sh = the same over the SHARED slots (n_routed .. S-1), a chain of its
 *        own; Nemotron's 2 shared slots carry weight 1, where each fma is the
 *        plain fp32 add s0 + s1;
 *   c  = r + sh (one fp32 add: r + (s0 + s1), not ((r + s0) + s1));
 *   h  = bf16(x + bf16(c)), the add in fp32 -- the hidden state that the
 *        final RMSNorm reads.
 *   x     [B, H]      bf16 residual
 *   slots [B, S, H]   expert outputs, fp32 (OR_F32) or bf16 (OR_BF16)
 *   w     [B, S]      fp32 slot weights
 *   h     [B, H]      bf16 output
 * With n_routed == S there is no shared slot and c = r (r + 0 = r: a chain
 * that starts at +0 never ends at -0).  The fp32 fma is C99's fmaf (one
 * rounding); bf16 rounding is to nearest, ties to even, NaN kept NaN.
 * ------------------------------------------------------------------------- */

static float bits_to_float(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* round an fp32 value to bf16 bits: nearest, ties to even */
uint16_t oracle_f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40u); /* NaN */
    const uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

int oracle_moe_combine(const uint16_t *x, const void *slots, int slot_dtype, int S, int n_routed, const float *w,
                       int B, int H, uint16_t *h) {
    if (B < 0 || H < 0 || S < 0 || n_routed < 0 || n_routed > S || (S > 0 && (!slots || !w)) ||
        (slot_dtype != OR_F32 && slot_dtype != OR_BF16))
        return -1;
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j < H; ++j) {
            float r = 0.0f, sh = 0.0f;
            for (int s = 0; s < S; ++s) {
                const int64_t e = ((int64_t)b * S + s) * H + j;
                const float y = slot_dtype == OR_F32 ? ((const float *)slots)[e]
                                                     : bits_to_float(((uint32_t)((const uint16_t *)slots)[e]) << 16);
                const float ws = w[(int64_t)b * S + s];
                if (s < n_routed)
                    r = fmaf(ws, y, r);
                else
                    sh = fmaf(ws, y, sh);
            }
            const float acc = r + sh;
            const float d = bits_to_float(((uint32_t)oracle_f32_to_bf16_rne(acc)) << 16);
            const float xv = bits_to_float(((uint32_t)x[(int64_t)b * H + j]) << 16);
            const float sum = xv + d;
            h[(int64_t)b * H + j] = oracle_f32_to_bf16_rne(sum);
        }
    }
    return 0;
}
