/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the gated delta rule forward scan.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this file; the CUDA library never links
 * or calls it, and it shares no code with the CUDA kernels.
 *
 * It computes, token by token and in double precision, exactly what the
 * pages define; no chunking, blocking or re-association is done here.
 *
 *   State S (K x V, rows = key features, columns = value features), per
 *   (sequence, head), for t = 0 .. len-1 in order:
 *     1. decay        S <- diag(exp(gk_t)) S      (scalar gate: exp(g_t) S)
 *     2. prediction   p = S^T k_t                  (a V-vector)
 *     3. delta        d = beta_t (v_t - p)
 *     4. write        S <- S + k_t d^T
 *     5. output       o_t = S^T q_t                (inclusive: after the write)
 *   The final state is S after the last token.
 *
 *   Passages followed: SANA `fused_gdn.py` page, `_fused_gdn_kernel`
 *   ("Pass 1 -- State Accumulation": decay first, then V_pred = K state_prev,
 *   dv = (V - V_pred) beta, state += K^T dv; "Pass 2 -- Output (reads
 *   state_curr, inclusive)"); SANA `fused_cam_gdn.py` page,
 *   `_cam_scan_kernel` (same order, init/final state contract: the loaded
 *   state is the state at the end of a prefix and the first decay of this
 *   call applies to it).
 *
 *   Reverse (anti-causal) scan, SANA `fused_cam_gdn.py` page,
 *   `_torch_cam_scan_reference` / `_flip_and_shift`: q is flipped, k, v,
 *   beta are flipped and shifted right by one (pad 0), the decay is flipped
 *   and shifted (pad: decay 1), the output is flipped back. Written here
 *   without any flips: walking p = len-1 .. 0, the state first absorbs token
 *   p+1 (its decay, then its write; nothing for p = len-1) and then emits
 *   o_p = R^T q_p. Hence o_{len-1} = 0 and no token contributes to its own
 *   output.
 *
 *   Denominator scan (SANA `fused_gdn.py` page, `_fused_gdn_kernel`,
 *   z_hat / dz / den): the same recurrence with V = 1 and v = 1; the caller
 *   passes a ones vector.
 *
 * Prep (SANA `fused_gdn.py` page, `_precompute_inv_rms` and
 * `_fused_qk_inv_rms_kernel`; `_fused_gdn_kernel` ReLU and k_scale):
 *   L2:  y = x / sqrt(sum_d x_d^2 + eps) per (token, head)
 *   RMS: inv = 1 / sqrt(sum_{h,d} x^2 / (H*D) + eps) per token over all
 *        channels, y = x * inv, then optional ReLU, then y *= scale.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int n_seq, H, K, V, reverse;
    const int64_t *row0, *len;
    const double *q, *k, *v, *g, *gk, *beta, *h0;
    double *out, *h_final;
    long next;            /* work counter, (seq, head) pairs */
    int status;
} scan_job;

/* Absorb one token (row r, head h) into S: decay, delta, write. */
static void absorb(const scan_job *J, double *S, double *p, int64_t r, int h) {
    const int K = J->K, V = J->V, H = J->H;
    const double *kt = J->k + (r * H + h) * (int64_t)K;
    const double *vt = J->v + (r * H + h) * (int64_t)V;
    const double bt = J->beta[r * H + h];
    for (int a = 0; a < K; ++a) {
        double d = J->gk ? exp(J->gk[(r * H + h) * (int64_t)K + a])
                         : exp(J->g[r * H + h]);
        for (int b = 0; b < V; ++b) S[a * V + b] *= d;
    }
    for (int b = 0; b < V; ++b) {
        double acc = 0.0;
        for (int a = 0; a < K; ++a) acc += S[a * V + b] * kt[a];
        p[b] = bt * (vt[b] - acc);
    }
    for (int a = 0; a < K; ++a)
        for (int b = 0; b < V; ++b) S[a * V + b] += kt[a] * p[b];
}

/* o = S^T q for token row r, head h. */
static void emit(const scan_job *J, const double *S, int64_t r, int h) {
    const int K = J->K, V = J->V, H = J->H;
    const double *qt = J->q + (r * H + h) * (int64_t)K;
    double *ot = J->out + (r * H + h) * (int64_t)V;
    for (int b = 0; b < V; ++b) {
        double acc = 0.0;
        for (int a = 0; a < K; ++a) acc += S[a * V + b] * qt[a];
        ot[b] = acc;
    }
}

static void scan_one(const scan_job *J, int s, int h, double *S, double *p) {
    const int K = J->K, V = J->V, H = J->H;
    const int64_t r0 = J->row0[s], n = J->len[s];
    if (J->h0)
        memcpy(S, J->h0 + ((int64_t)s * H + h) * K * V, sizeof(double) * K * V);
    else
        memset(S, 0, sizeof(double) * K * V);
    if (!J->reverse) {
        for (int64_t t = 0; t < n; ++t) {
            absorb(J, S, p, r0 + t, h);
            emit(J, S, r0 + t, h);
        }
    } else {
        for (int64_t t = n - 1; t >= 0; --t) {
            if (t + 1 < n) absorb(J, S, p, r0 + t + 1, h);
            emit(J, S, r0 + t, h);
        }
    }
    if (J->h_final)
        memcpy(J->h_final + ((int64_t)s * H + h) * K * V, S, sizeof(double) * K * V);
}

static void *scan_worker(void *arg) {
    scan_job *J = (scan_job *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)J->K * J->V);
    double *p = (double *)malloc(sizeof(double) * (size_t)J->V);
    if (!S || !p) {
        __atomic_store_n(&J->status, 1, __ATOMIC_RELAXED);
        free(S);
        free(p);
        return NULL;
    }
    const long total = (long)J->n_seq * J->H;
    for (;;) {
        long w = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (w >= total) break;
        scan_one(J, (int)(w / J->H), (int)(w % J->H), S, p);
    }
    free(S);
    free(p);
    return NULL;
}

/*
 * Run the scan for n_seq sequences x H heads.
 *   Sequence s occupies rows row0[s] .. row0[s]+len[s]-1 of the packed
 *   arrays q, k (rows, H, K), v, out (rows, H, V), beta, g (rows, H),
 *   gk (rows, H, K). Exactly one of g / gk is non-NULL.
 *   h0 (n_seq, H, K, V) may be NULL (zero state); h_final may be NULL.
 * Returns 0 on success, nonzero on bad arguments or allocation failure.
 */
int oracle_gdn_scan(int n_seq, const int64_t *row0, const int64_t *len, int H,
                    int K, int V, const double *q, const double *k,
                    const double *v, const double *g, const double *gk,
                    const double *beta, const double *h0, int reverse,
                    double *out, double *h_final, int n_threads) {
    if (n_seq < 0 || H <= 0 || K <= 0 || V <= 0) return 2;
    if ((g == NULL) == (gk == NULL)) return 3;
    scan_job J = {n_seq, H, K, V, reverse, row0, len, q, k, v, g, gk, beta,
                  h0, out, h_final, 0, 0};
    long total = (long)n_seq * H;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > total) n_threads = (int)(total > 0 ? total : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * n_threads);
    if (!th) return 1;
    int started = 0;
    for (int i = 1; i < n_threads; ++i)
        if (pthread_create(&th[started], NULL, scan_worker, &J) == 0) ++started;
    scan_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    return J.status;
}

/*
 * Frame-causal scan (SANA `fused_gdn.py` page, `_fused_gdn_kernel` with S
 * tokens per frame; SANA `fused_cam_gdn.py` page, `_cam_scan_kernel`): per
 * (sequence, head), frames of `frame` tokens, one log-decay per frame:
 *   forward, frame f = 0 .. F-1:
 *     S <- exp(gf_f) S;  S_pre = S
 *     for every token t of frame f:  d = beta_t (v_t - S_pre^T k_t);
 *                                    S <- S + k_t d^T
 *     (every token predicts from the same pre-frame state S_pre)
 *     then o_t = S^T q_t for every token of frame f (the post-frame state)
 *   reverse, step i = 0 .. F-1: the output frame is F-1-i; for i > 0 the
 *     state first absorbs frame F-i (its decay, then its tokens as above);
 *     step 0 absorbs nothing. So frame f reads frames f+1 .. F-1.
 * gf is (n_seq, F, H); h0 / h_final as for oracle_gdn_scan.
 */
typedef struct {
    int n_seq, H, K, V, frame, reverse;
    const int64_t *row0, *len;
    const double *q, *k, *v, *gf, *beta, *h0;
    double *out, *h_final;
    long next;
    int status;
} frame_job;

static void frame_absorb(const frame_job *J, double *S, double *Spre, double *p, int s, int f, int h) {
    const int K = J->K, V = J->V, H = J->H;
    const int F = (int)(J->len[s] / J->frame);
    const double d = exp(J->gf[((int64_t)s * F + f) * H + h]);
    for (int a = 0; a < K * V; ++a) S[a] *= d;
    memcpy(Spre, S, sizeof(double) * K * V);
    for (int t = 0; t < J->frame; ++t) {
        const int64_t r = J->row0[s] + (int64_t)f * J->frame + t;
        const double *kt = J->k + (r * H + h) * (int64_t)K;
        const double *vt = J->v + (r * H + h) * (int64_t)V;
        const double bt = J->beta[r * H + h];
        for (int b = 0; b < V; ++b) {
            double acc = 0.0;
            for (int a = 0; a < K; ++a) acc += Spre[a * V + b] * kt[a];
            p[b] = bt * (vt[b] - acc);
        }
        for (int a = 0; a < K; ++a)
            for (int b = 0; b < V; ++b) S[a * V + b] += kt[a] * p[b];
    }
}

static void frame_emit(const frame_job *J, const double *S, int s, int f, int h) {
    const int K = J->K, V = J->V, H = J->H;
    for (int t = 0; t < J->frame; ++t) {
        const int64_t r = J->row0[s] + (int64_t)f * J->frame + t;
        const double *qt = J->q + (r * H + h) * (int64_t)K;
        double *ot = J->out + (r * H + h) * (int64_t)V;
        for (int b = 0; b < V; ++b) {
            double acc = 0.0;
            for (int a = 0; a < K; ++a) acc += S[a * V + b] * qt[a];
            ot[b] = acc;
        }
    }
}

static void *frame_worker(void *arg) {
    frame_job *J = (frame_job *)arg;
    const int K = J->K, V = J->V, H = J->H;
    double *S = (double *)malloc(sizeof(double) * (size_t)K * V);
    double *Spre = (double *)malloc(sizeof(double) * (size_t)K * V);
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    if (!S || !Spre || !p) {
        __atomic_store_n(&J->status, 1, __ATOMIC_RELAXED);
        free(S);
        free(Spre);
        free(p);
        return NULL;
    }
    const long total = (long)J->n_seq * H;
    for (;;) {
        long w = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (w >= total) break;
        const int s = (int)(w / H), h = (int)(w % H);
        const int F = (int)(J->len[s] / J->frame);
        if (J->h0)
            memcpy(S, J->h0 + ((int64_t)s * H + h) * K * V, sizeof(double) * K * V);
        else
            memset(S, 0, sizeof(double) * K * V);
        for (int i = 0; i < F; ++i) {
            if (!J->reverse) {
                frame_absorb(J, S, Spre, p, s, i, h);
                frame_emit(J, S, s, i, h);
            } else {
                if (i > 0) frame_absorb(J, S, Spre, p, s, F - i, h);
                frame_emit(J, S, s, F - 1 - i, h);
            }
        }
        if (J->h_final) memcpy(J->h_final + ((int64_t)s * H + h) * K * V, S, sizeof(double) * K * V);
    }
    free(S);
    free(Spre);
    free(p);
    return NULL;
}

int oracle_gdn_frame_scan(int n_seq, const int64_t *row0, const int64_t *len, int H, int K, int V,
                          const double *q, const double *k, const double *v, const double *gf,
                          const double *beta, const double *h0, int frame, int reverse,
                          double *out, double *h_final, int n_threads) {
    if (n_seq < 0 || H <= 0 || K <= 0 || V <= 0 || frame <= 0) return 2;
    for (int s = 0; s < n_seq; ++s)
        if (len[s] % frame != 0) return 2;
    frame_job J = {n_seq, H, K, V, frame, reverse, row0, len, q, k, v, gf, beta, h0, out, h_final, 0, 0};
    long total = (long)n_seq * H;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > total) n_threads = (int)(total > 0 ? total : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * n_threads);
    if (!th) return 1;
    int started = 0;
    for (int i = 1; i < n_threads; ++i)
        if (pthread_create(&th[started], NULL, frame_worker, &J) == 0) ++started;
    frame_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    return J.status;
}

/*
 * L2 prep: x and y are (rows, D); y_r = x_r / sqrt(|x_r|^2 + eps).
 */
void oracle_l2norm(const double *x, int64_t rows, int D, double eps, double *y) {
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * D;
        double ss = 0.0;
        for (int d = 0; d < D; ++d) ss += xr[d] * xr[d];
        double inv = 1.0 / sqrt(ss + eps);
        for (int d = 0; d < D; ++d) y[r * D + d] = xr[d] * inv;
    }
}

/*
 * Full-channel RMS prep: x and y are (rows, C) with C = H*D channels of one
 * token; inv_rms (rows) may be NULL. y = relu?(x * inv) * scale.
 */
void oracle_rmsnorm(const double *x, int64_t rows, int C, double eps, int relu,
                    double scale, double *y, double *inv_rms) {
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * C;
        double ss = 0.0;
        for (int c = 0; c < C; ++c) ss += xr[c] * xr[c];
        double inv = 1.0 / sqrt(ss / C + eps);
        if (inv_rms) inv_rms[r] = inv;
        for (int c = 0; c < C; ++c) {
            double t = xr[c] * inv;
            if (relu && t < 0.0) t = 0.0;
            y[r * C + c] = t * scale;
        }
    }
}
