/*
 * Oracle for the chunked gated-delta-rule prefill path — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, sequential fp64 CPU implementation of what the GPU path computes.
 * Only the test suite, the smoke check and the bench's CPU-baseline leg use it; the
 * product path never links, loads or calls it. It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Sources (pages of the metrale engine documentation):
 *  - "split_prefill.rs" (trait LayerSplitPrefill): prefill_phase1_conv1d_one (conv over one
 *    request's tokens, advancing its conv state), prefill_phase1_l2_batched (L2 norm over
 *    the stacked q|k), prefill_gdn_full / prefill_gdn_full_batched /
 *    prefill_gdn_full_batched_fla_varlen (the GDN recurrence per stream, batched, varlen).
 *  - "glm5next_kda/prefill.rs" (Glm5NextKdaLayer::prefill_with_pad_fill): the conv_prefill
 *    launch (conv + SiLU, optional bias slot passed as NULL), the l2 launch (per head over the
 *    q|k channels, eps = cfg.l2_eps), the chunk_scan launch (scale = 1/sqrt(head_dim)).
 *  - The recurrence itself is the gated delta rule (Gated DeltaNet, Yang, Kautz &
 *    Hatamizadeh 2024; per-channel gate as in Kimi Delta Attention, 2025):
 *        S_t = S_{t-1} diag(alpha_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *        o_t = scale * S_t q_t,   alpha_t = exp(g_t).
 *    It is evaluated token by token, exactly as written; no chunking.
 *
 * State layout: H = S^T, row-major [Hv][dk][dv] per stream (H[c][d] = S[d][c]).
 *
 * Parity pins live in tests/ (brute-force products of transition matrices, closed forms,
 * numpy.convolve, invariants). Every function here is pinned there.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Causal depthwise conv1d + SiLU over one stream ("glm5next_kda/prefill.rs", conv_prefill
 * launch; "split_prefill.rs", prefill_phase1_conv1d_one).
 *   xh = [state (K-1 rows, oldest first) ; x (t rows)]
 *   y[tau][c] = bias[c] + sum_{j<K} w[c][j] * xh[tau + j][c]   (tap K-1 = current token)
 *   out[tau][c] = y / (1 + exp(-y))                              (SiLU)
 *   new_state = xh[t .. t+K-2]
 * x rows are x_stride apart, out rows out_stride apart. new_state may alias state. */
void or_conv1d_silu(const double *state, const double *x, const double *w, const double *bias,
                    double *out, double *new_state, int t, int C, int K, long x_stride,
                    long out_stride)
{
    int nh = K - 1 + t;
    double *xh = (double *)malloc(sizeof(double) * (size_t)(nh > 0 ? nh : 1) * (size_t)C);
    for (int r = 0; r < K - 1; ++r)
        for (int c = 0; c < C; ++c) xh[(size_t)r * C + c] = state[(size_t)r * C + c];
    for (int r = 0; r < t; ++r)
        for (int c = 0; c < C; ++c) xh[(size_t)(K - 1 + r) * C + c] = x[(size_t)r * x_stride + c];
    for (int tau = 0; tau < t; ++tau) {
        for (int c = 0; c < C; ++c) {
            double y = bias ? bias[c] : 0.0;
            for (int j = 0; j < K; ++j) y += w[(size_t)c * K + j] * xh[(size_t)(tau + j) * C + c];
            out[(size_t)tau * out_stride + c] = y / (1.0 + exp(-y));
        }
    }
    for (int r = 0; r < K - 1; ++r)
        for (int c = 0; c < C; ++c) new_state[(size_t)r * C + c] = xh[(size_t)(t + r) * C + c];
    free(xh);
}

/* Per-(token, head) L2 norm, in place ("glm5next_kda/prefill.rs", l2 launch; grid over
 * q|k heads x tokens, one head_dim vector each):  x <- x / sqrt(sum x^2 + eps). */
void or_l2norm_heads(double *x, int t, int n_heads, int hd, long row_stride, double eps)
{
    for (int tau = 0; tau < t; ++tau) {
        for (int h = 0; h < n_heads; ++h) {
            double *p = x + (size_t)tau * row_stride + (size_t)h * hd;
            double ss = 0.0;
            for (int c = 0; c < hd; ++c) ss += p[c] * p[c];
            double inv = 1.0 / sqrt(ss + eps);
            for (int c = 0; c < hd; ++c) p[c] *= inv;
        }
    }
}

/* Gated RMSNorm of the recurrence output, per (token, v-head) row of dv values
 * ("split_prefill.rs", LayerSplitPrefill::prefill_phase3: gated RMSNorm of the GDN output with
 * Z). The pages name the step only; read plainly:
 *   y[c] = o[c] / sqrt(mean_c o^2 + eps) * w[c] * SiLU(z[c]),   SiLU(z) = z / (1 + e^-z),
 * with one weight per channel (dv values) shared by all heads. o, z, y: n_rows x dv. */
void or_gated_rmsnorm(const double *o, const double *z, const double *w, double *y, long n_rows,
                      int dv, double eps)
{
    for (long r = 0; r < n_rows; ++r) {
        const double *orow = o + (size_t)r * dv, *zrow = z + (size_t)r * dv;
        double *yrow = y + (size_t)r * dv;
        double ss = 0.0;
        for (int c = 0; c < dv; ++c) ss += orow[c] * orow[c];
        const double inv = 1.0 / sqrt(ss / dv + eps);
        for (int c = 0; c < dv; ++c) {
            const double gate = zrow[c] / (1.0 + exp(-zrow[c]));
            yrow[c] = orow[c] * inv * w[c] * gate;
        }
    }
}

/* One (stream, v-head) unit of the gated delta rule, token by token.
 *   H  : [dk][dv] state of this v-head (in/out)
 *   q,k: rows of dk values for the unit's k-head, row strides q_stride, k_stride
 *   v  : rows of dv values, row stride v_stride
 *   g  : per token, 1 value (GDN) or dk values (KDA), row stride g_stride
 *   beta: per token, row stride b_stride
 *   o  : rows of dv values, row stride o_stride                                          */
static void unit_recurrence(double *H, const double *q, const double *k, const double *v,
                            const double *g, const double *beta, double *o, int t, int dk,
                            int dv, long q_stride, long k_stride, long v_stride, long g_stride,
                            long b_stride, long o_stride, int per_channel, double scale)
{
    double *r = (double *)malloc(sizeof(double) * (size_t)dv);
    for (int tau = 0; tau < t; ++tau) {
        const double *qt = q + (size_t)tau * q_stride;
        const double *kt = k + (size_t)tau * k_stride;
        const double *vt = v + (size_t)tau * v_stride;
        const double *gt = g + (size_t)tau * g_stride;
        double bt = beta[(size_t)tau * b_stride];
        /* S <- S diag(alpha): column c of S is row c of H */
        for (int c = 0; c < dk; ++c) {
            double a = exp(per_channel ? gt[c] : gt[0]);
            for (int d = 0; d < dv; ++d) H[(size_t)c * dv + d] *= a;
        }
        /* r = S k */
        for (int d = 0; d < dv; ++d) r[d] = 0.0;
        for (int c = 0; c < dk; ++c)
            for (int d = 0; d < dv; ++d) r[d] += H[(size_t)c * dv + d] * kt[c];
        /* S <- S + beta (v - r) k^T */
        for (int d = 0; d < dv; ++d) r[d] = bt * (vt[d] - r[d]);
        for (int c = 0; c < dk; ++c)
            for (int d = 0; d < dv; ++d) H[(size_t)c * dv + d] += kt[c] * r[d];
        /* o = scale S q */
        double *ot = o + (size_t)tau * o_stride;
        for (int d = 0; d < dv; ++d) ot[d] = 0.0;
        for (int c = 0; c < dk; ++c)
            for (int d = 0; d < dv; ++d) ot[d] += H[(size_t)c * dv + d] * qt[c];
        for (int d = 0; d < dv; ++d) ot[d] *= scale;
    }
    free(r);
}

typedef struct {
    double **h_ptrs;
    const double *q, *k, *v, *g, *beta;
    double *out;
    const int32_t *cu;
    int B, Hk, Hv, dk, dv, per_channel;
    long q_stride, k_stride, v_stride;
    double scale;
    volatile long next;
} job_t;

static void run_unit(job_t *J, long u)
{
    int s = (int)(u / J->Hv), j = (int)(u % J->Hv);
    int kh = (int)((long)j * J->Hk / J->Hv); /* v-head j reads q/k head floor(j*Hk/Hv) */
    long t0 = J->cu[s], t = J->cu[s + 1] - J->cu[s];
    if (t <= 0) return;
    long gw = J->per_channel ? (long)J->dk : 1;
    unit_recurrence(J->h_ptrs[s] + (size_t)j * J->dk * J->dv,
                    J->q + (size_t)t0 * J->q_stride + (size_t)kh * J->dk,
                    J->k + (size_t)t0 * J->k_stride + (size_t)kh * J->dk,
                    J->v + (size_t)t0 * J->v_stride + (size_t)j * J->dv,
                    J->g + (size_t)t0 * J->Hv * gw + (size_t)j * gw,
                    J->beta + (size_t)t0 * J->Hv + j,
                    J->out + (size_t)t0 * J->Hv * J->dv + (size_t)j * J->dv,
                    (int)t, J->dk, J->dv, J->q_stride, J->k_stride, J->v_stride,
                    (long)J->Hv * gw, J->Hv,
                    (long)J->Hv * J->dv, J->per_channel, J->scale);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    long n = (long)J->B * J->Hv;
    for (;;) {
        long u = __sync_fetch_and_add(&J->next, 1);
        if (u >= n) break;
        run_unit(J, u);
    }
    return NULL;
}

/* Gated delta rule over B streams packed back to back (cu_seqlens[B+1] token offsets),
 * one state pointer per stream ("split_prefill.rs", prefill_gdn_full_batched /
 * prefill_gdn_full_batched_fla_varlen; batched = equal lengths).
 *   q: [T][Hk][dk] at row stride q_stride; k likewise (k_stride); v: [T][Hv][dv] (v_stride)
 *   g: [T][Hv] (GDN) or [T][Hv][dk] (KDA, per_channel=1); beta: [T][Hv]
 *   out: [T][Hv][dv] contiguous; h_ptrs[s]: [Hv][dk][dv], updated in place.
 * Units (stream, v-head) are independent and run on n_threads host threads; each unit's
 * arithmetic is sequential, so results do not depend on n_threads. */
void or_gated_delta_varlen(double **h_ptrs, const double *q, const double *k, const double *v,
                           const double *g, const double *beta, double *out,
                           const int32_t *cu_seqlens, int B, int Hk, int Hv, int dk, int dv,
                           long q_stride, long k_stride, long v_stride, int per_channel,
                           double scale, int n_threads)
{
    job_t J;
    J.h_ptrs = h_ptrs; J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.out = out;
    J.cu = cu_seqlens; J.B = B; J.Hk = Hk; J.Hv = Hv; J.dk = dk; J.dv = dv;
    J.per_channel = per_channel; J.q_stride = q_stride; J.k_stride = k_stride;
    J.v_stride = v_stride; J.scale = scale; J.next = 0;
    if (n_threads <= 1) {
        worker(&J);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, worker, &J);
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
    free(th);
}
