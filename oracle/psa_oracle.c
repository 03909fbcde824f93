/*
 * psa_oracle.c -- plain, slow, fp64 CPU oracle for the YOLO26 Position-Sensitive
 * Attention (PSA) path.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the CPU-baseline leg
 * of bench.py call it; the library's product path never does.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it follows (vision-rs book, page "Custom Kernels"):
 *   - section "Flash Attention 2": attention over [BATCH*N_HEADS, N_CTX, HEAD_DIM]
 *     tensors with an online softmax, forward / dQ / dK-dV as separate kernels.
 *     The online softmax reaches exactly (up to rounding order) the plain result
 *     O = softmax(scale * Q K^T) V, so the oracle forms the N x N scores of one
 *     query row explicitly and applies that plain definition.
 *   - section "Position-Sensitive Attention (PSA)": PsaPackQkv, PsaExtractV,
 *     PsaMergeAttn and the V_lo / V_hi split with attention run once per half.
 *
 * Readings where the page is silent (listed with reasons in the design notes):
 *   spatial index n = h*W + w; head-batch index bh = b*num_heads + head;
 *   QKV channel of plane s (0=Q,1=K,2=V_lo,3=V_hi) element d of head hd is
 *   hd*4*KD + s*KD + d; merged channel of half t element d is hd*2*KD + t*KD + d;
 *   extracted V channel j (< 2*KD) is QKV channel hd*4*KD + 2*KD + j;
 *   no mask, no causality; LSE is the natural log of the softmax denominator
 *   including the running max; the backward is the analytic gradient of the same
 *   definition (dV = P^T dO, dP = dO V^T, D = rowsum(P o dP), dS = P o (dP - D),
 *   dQ = scale dS K, dK = scale dS^T Q).
 *
 * Layout routines move raw elements of any byte width (es), so they are exact
 * for bf16, fp32 or fp64 storage alike.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Layouts (page "Custom Kernels", section "Position-Sensitive Attention")    */
/* ------------------------------------------------------------------------- */

/* PsaPackQkv: qkv [B, nh*4*KD, H*W] -> packed [4, B*nh, H*W, KD]. */
void oracle_pack_qkv(const void *qkv, void *packed, int B, int nh, int KD, int N, int es)
{
    const char *src = (const char *)qkv;
    char *dst = (char *)packed;
    const long C = (long)nh * 4 * KD;
    const long BH = (long)B * nh;
    for (long b = 0; b < B; ++b)
        for (long hd = 0; hd < nh; ++hd)
            for (long s = 0; s < 4; ++s)
                for (long d = 0; d < KD; ++d)
                    for (long n = 0; n < N; ++n) {
                        long from = (b * C + hd * 4 * KD + s * KD + d) * N + n;
                        long to = ((s * BH + b * nh + hd) * N + n) * KD + d;
                        memcpy(dst + to * es, src + from * es, (size_t)es);
                    }
}

/* Inverse permutation of PsaPackQkv (the adjoint used by the backward). */
void oracle_unpack_qkv(const void *packed, void *qkv, int B, int nh, int KD, int N, int es)
{
    const char *src = (const char *)packed;
    char *dst = (char *)qkv;
    const long C = (long)nh * 4 * KD;
    const long BH = (long)B * nh;
    for (long b = 0; b < B; ++b)
        for (long hd = 0; hd < nh; ++hd)
            for (long s = 0; s < 4; ++s)
                for (long d = 0; d < KD; ++d)
                    for (long n = 0; n < N; ++n) {
                        long to = (b * C + hd * 4 * KD + s * KD + d) * N + n;
                        long from = ((s * BH + b * nh + hd) * N + n) * KD + d;
                        memcpy(dst + to * es, src + from * es, (size_t)es);
                    }
}

/* PsaExtractV: the V section [V_lo | V_hi] of every head, in NCHW [B, nh*2*KD, H*W]. */
void oracle_extract_v(const void *qkv, void *v, int B, int nh, int KD, int N, int es)
{
    const char *src = (const char *)qkv;
    char *dst = (char *)v;
    const long C = (long)nh * 4 * KD;
    const long c = (long)nh * 2 * KD;
    for (long b = 0; b < B; ++b)
        for (long hd = 0; hd < nh; ++hd)
            for (long j = 0; j < 2 * KD; ++j)
                for (long n = 0; n < N; ++n) {
                    long from = (b * C + hd * 4 * KD + 2 * KD + j) * N + n;
                    long to = (b * c + hd * 2 * KD + j) * N + n;
                    memcpy(dst + to * es, src + from * es, (size_t)es);
                }
}

/* PsaMergeAttn: o_lo, o_hi [B*nh, H*W, KD] -> out NCHW [B, nh*2*KD, H*W]. */
void oracle_merge_attn(const void *o_lo, const void *o_hi, void *out, int B, int nh, int KD,
                       int N, int es)
{
    const char *half[2] = {(const char *)o_lo, (const char *)o_hi};
    char *dst = (char *)out;
    const long c = (long)nh * 2 * KD;
    for (long b = 0; b < B; ++b)
        for (long hd = 0; hd < nh; ++hd)
            for (long t = 0; t < 2; ++t)
                for (long d = 0; d < KD; ++d)
                    for (long n = 0; n < N; ++n) {
                        long from = ((b * nh + hd) * N + n) * KD + d;
                        long to = (b * c + hd * 2 * KD + t * KD + d) * N + n;
                        memcpy(dst + to * es, half[t] + from * es, (size_t)es);
                    }
}

/* Inverse of PsaMergeAttn (the adjoint used by the backward). */
void oracle_unmerge_attn(const void *out, void *o_lo, void *o_hi, int B, int nh, int KD, int N,
                         int es)
{
    const char *src = (const char *)out;
    char *half[2] = {(char *)o_lo, (char *)o_hi};
    const long c = (long)nh * 2 * KD;
    for (long b = 0; b < B; ++b)
        for (long hd = 0; hd < nh; ++hd)
            for (long t = 0; t < 2; ++t)
                for (long d = 0; d < KD; ++d)
                    for (long n = 0; n < N; ++n) {
                        long to = ((b * nh + hd) * N + n) * KD + d;
                        long from = (b * c + hd * 2 * KD + t * KD + d) * N + n;
                        memcpy(half[t] + to * es, src + from * es, (size_t)es);
                    }
}

/* ------------------------------------------------------------------------- */
/* Softmax attention of one query row (section "Flash Attention 2": the       */
/* plain result the online softmax reaches).                                  */
/* ------------------------------------------------------------------------- */

/* Row i of one head: p[j] = softmax_j(scale * q_i . k_j); returns LSE_i. */
static double softmax_row(const double *q, const double *k, int N, int dqk, double scale, long i,
                          double *p)
{
    double m = -INFINITY;
    for (long j = 0; j < N; ++j) {
        double s = 0.0;
        for (long c = 0; c < dqk; ++c)
            s += q[i * dqk + c] * k[j * dqk + c];
        p[j] = scale * s;
        if (p[j] > m)
            m = p[j];
    }
    double l = 0.0;
    for (long j = 0; j < N; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    for (long j = 0; j < N; ++j)
        p[j] /= l;
    return m + log(l);
}

/* Forward of one head: o [N, dv], lse [N]. */
static void attn_fwd_head(const double *q, const double *k, const double *v, double *o,
                          double *lse, int N, int dqk, int dv, double scale, double *p)
{
    for (long i = 0; i < N; ++i) {
        double L = softmax_row(q, k, N, dqk, scale, i, p);
        if (lse)
            lse[i] = L;
        for (long c = 0; c < dv; ++c) {
            double acc = 0.0;
            for (long j = 0; j < N; ++j)
                acc += p[j] * v[j * dv + c];
            o[i * dv + c] = acc;
        }
    }
}

/*
 * Backward of one head, one query row at a time (the N x N matrices are never
 * needed whole): with P the softmax of row i,
 *   dV_j += P_ij dO_i,  dP_ij = dO_i . V_j,  D_i = sum_j P_ij dP_ij,
 *   dS_ij = P_ij (dP_ij - D_i),  dQ_i = scale sum_j dS_ij K_j,  dK_j += scale dS_ij Q_i.
 * dq/dk/dv are overwritten.
 */
static void attn_bwd_head(const double *q, const double *k, const double *v, const double *dout,
                          double *dq, double *dk, double *dvv, int N, int dqk, int dv,
                          double scale, double *p, double *dp)
{
    memset(dk, 0, sizeof(double) * (size_t)N * dqk);
    memset(dvv, 0, sizeof(double) * (size_t)N * dv);
    for (long i = 0; i < N; ++i) {
        softmax_row(q, k, N, dqk, scale, i, p);
        double D = 0.0;
        for (long j = 0; j < N; ++j) {
            double s = 0.0;
            for (long c = 0; c < dv; ++c)
                s += dout[i * dv + c] * v[j * dv + c];
            dp[j] = s;
            D += p[j] * s;
        }
        for (long c = 0; c < dqk; ++c)
            dq[i * dqk + c] = 0.0;
        for (long j = 0; j < N; ++j) {
            double ds = p[j] * (dp[j] - D);
            for (long c = 0; c < dv; ++c)
                dvv[j * dv + c] += p[j] * dout[i * dv + c];
            for (long c = 0; c < dqk; ++c) {
                dq[i * dqk + c] += scale * ds * k[j * dqk + c];
                dk[j * dqk + c] += scale * ds * q[i * dqk + c];
            }
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Threading over independent heads (bh units share nothing).                 */
/* ------------------------------------------------------------------------- */

typedef struct {
    const double *q, *k, *v, *dout;
    double *o, *lse, *dq, *dk, *dv;
    int BH, N, dqk, dvd;
    double scale;
    int backward;
    int tid, nthreads;
} job_t;

static void *attn_worker(void *arg)
{
    job_t *j = (job_t *)arg;
    double *p = (double *)malloc(sizeof(double) * (size_t)j->N * 2);
    double *dp = p + j->N;
    for (long bh = j->tid; bh < j->BH; bh += j->nthreads) {
        const long Nq = (long)j->N * j->dqk, Nv = (long)j->N * j->dvd;
        if (!j->backward) {
            attn_fwd_head(j->q + bh * Nq, j->k + bh * Nq, j->v + bh * Nv, j->o + bh * Nv,
                          j->lse ? j->lse + bh * j->N : NULL, j->N, j->dqk, j->dvd, j->scale, p);
        } else {
            attn_bwd_head(j->q + bh * Nq, j->k + bh * Nq, j->v + bh * Nv, j->dout + bh * Nv,
                          j->dq + bh * Nq, j->dk + bh * Nq, j->dv + bh * Nv, j->N, j->dqk,
                          j->dvd, j->scale, p, dp);
        }
    }
    free(p);
    return NULL;
}

static void run_heads(job_t proto, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > proto.BH)
        nthreads = proto.BH;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].tid = t;
        jobs[t].nthreads = nthreads;
        pthread_create(&th[t], NULL, attn_worker, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        pthread_join(th[t], NULL);
    free(jobs);
    free(th);
}

/* Attention forward over [BH, N, d]: o [BH, N, dv], lse [BH, N] (lse may be NULL). */
void oracle_attn_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
                     int BH, int N, int dqk, int dv, double scale, int nthreads)
{
    job_t j = {q, k, v, NULL, o, lse, NULL, NULL, NULL, BH, N, dqk, dv, scale, 0, 0, 1};
    run_heads(j, nthreads);
}

/* Attention backward over [BH, N, d]: gradients of sum(dout o O) w.r.t. q, k, v. */
void oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                     double *dq, double *dk, double *dv, int BH, int N, int dqk, int dvd,
                     double scale, int nthreads)
{
    job_t j = {q, k, v, dout, NULL, NULL, dq, dk, dv, BH, N, dqk, dvd, scale, 1, 0, 1};
    run_heads(j, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Sampled rows of one head, for checks at sizes where the whole head is too  */
/* slow: pointers address one head ([N, d] each).                             */
/* ------------------------------------------------------------------------- */

/* Forward output rows rows[0..nr) -> o [nr, dv], lse [nr]. */
void oracle_attn_fwd_rows(const double *q, const double *k, const double *v, int N, int dqk,
                          int dv, double scale, const long *rows, int nr, double *o, double *lse)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)N);
    for (int r = 0; r < nr; ++r) {
        long i = rows[r];
        lse[r] = softmax_row(q, k, N, dqk, scale, i, p);
        for (long c = 0; c < dv; ++c) {
            double acc = 0.0;
            for (long j = 0; j < N; ++j)
                acc += p[j] * v[j * dv + c];
            o[(long)r * dv + c] = acc;
        }
    }
    free(p);
}

/* dQ rows rows[0..nr) -> dq [nr, dqk] (needs only row i of P and dP). */
void oracle_attn_bwd_dq_rows(const double *q, const double *k, const double *v,
                             const double *dout, int N, int dqk, int dv, double scale,
                             const long *rows, int nr, double *dq)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)N * 2);
    double *dp = p + N;
    for (int r = 0; r < nr; ++r) {
        long i = rows[r];
        softmax_row(q, k, N, dqk, scale, i, p);
        double D = 0.0;
        for (long j = 0; j < N; ++j) {
            double s = 0.0;
            for (long c = 0; c < dv; ++c)
                s += dout[i * dv + c] * v[j * dv + c];
            dp[j] = s;
            D += p[j] * s;
        }
        for (long c = 0; c < dqk; ++c) {
            double acc = 0.0;
            for (long j = 0; j < N; ++j)
                acc += p[j] * (dp[j] - D) * k[j * dqk + c];
            dq[(long)r * dqk + c] = scale * acc;
        }
    }
    free(p);
}

typedef struct {
    const double *q, *k, *v, *dout;
    int N, dqk, dv;
    double scale;
    const long *keys;
    int nk;
    double *dk, *dvv; /* partial sums of this thread: [nk, dqk], [nk, dv] */
    int tid, nthreads;
} kjob_t;

static void *dkdv_rows_worker(void *arg)
{
    kjob_t *j = (kjob_t *)arg;
    const int N = j->N, dqk = j->dqk, dv = j->dv;
    double *p = (double *)malloc(sizeof(double) * (size_t)N);
    memset(j->dk, 0, sizeof(double) * (size_t)j->nk * dqk);
    memset(j->dvv, 0, sizeof(double) * (size_t)j->nk * dv);
    for (long i = j->tid; i < N; i += j->nthreads) {
        softmax_row(j->q, j->k, N, dqk, j->scale, i, p);
        double D = 0.0;
        for (long jj = 0; jj < N; ++jj) {
            double s = 0.0;
            for (long c = 0; c < dv; ++c)
                s += j->dout[i * dv + c] * j->v[jj * dv + c];
            D += p[jj] * s;
        }
        for (int r = 0; r < j->nk; ++r) {
            long key = j->keys[r];
            double s = 0.0;
            for (long c = 0; c < dv; ++c)
                s += j->dout[i * dv + c] * j->v[key * dv + c];
            double ds = p[key] * (s - D);
            for (long c = 0; c < dv; ++c)
                j->dvv[(long)r * dv + c] += p[key] * j->dout[i * dv + c];
            for (long c = 0; c < dqk; ++c)
                j->dk[(long)r * dqk + c] += j->scale * ds * j->q[i * dqk + c];
        }
    }
    free(p);
    return NULL;
}

/* dK and dV rows for keys[0..nk) -> dk [nk, dqk], dv [nk, dv]; every query row
 * contributes, so the work is O(N^2 d); it is split over nthreads and the
 * partial sums are added in thread order. */
void oracle_attn_bwd_dkdv_rows(const double *q, const double *k, const double *v,
                               const double *dout, int N, int dqk, int dv, double scale,
                               const long *keys, int nk, double *dk, double *dvv, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    kjob_t *jobs = (kjob_t *)malloc(sizeof(kjob_t) * (size_t)nthreads);
    double *part = (double *)malloc(sizeof(double) * (size_t)nthreads * nk * (dqk + dv));
    for (int t = 0; t < nthreads; ++t) {
        kjob_t j = {q, k, v, dout, N, dqk, dv, scale, keys, nk,
                    part + (size_t)t * nk * (dqk + dv), part + (size_t)t * nk * (dqk + dv) + (size_t)nk * dqk,
                    t, nthreads};
        jobs[t] = j;
        pthread_create(&th[t], NULL, dkdv_rows_worker, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        pthread_join(th[t], NULL);
    memset(dk, 0, sizeof(double) * (size_t)nk * dqk);
    memset(dvv, 0, sizeof(double) * (size_t)nk * dv);
    for (int t = 0; t < nthreads; ++t) {
        for (long e = 0; e < (long)nk * dqk; ++e)
            dk[e] += jobs[t].dk[e];
        for (long e = 0; e < (long)nk * dv; ++e)
            dvv[e] += jobs[t].dvv[e];
    }
    free(part);
    free(jobs);
    free(th);
}

/* ------------------------------------------------------------------------- */
/* The PSA chain as the page composes it: PsaPackQkv, attention once per V    */
/* half (HEAD_DIM = KD), PsaMergeAttn, PsaExtractV for the residual.          */
/* ------------------------------------------------------------------------- */

/* qkv NCHW [B, nh*4KD, N] fp64 -> out [B, nh*2KD, N], lse [B*nh, N], vres [B, nh*2KD, N]
 * (lse / vres may be NULL). */
void oracle_psa_fwd(const double *qkv, double *out, double *lse, double *vres, int B, int nh,
                    int KD, int N, double scale, int nthreads)
{
    const long BH = (long)B * nh, plane = BH * N * KD;
    double *packed = (double *)malloc(sizeof(double) * (size_t)(4 * plane));
    double *o_lo = (double *)malloc(sizeof(double) * (size_t)(2 * plane));
    double *o_hi = o_lo + plane;
    double *lse_hi = (double *)malloc(sizeof(double) * (size_t)(BH * N));
    oracle_pack_qkv(qkv, packed, B, nh, KD, N, (int)sizeof(double));
    const double *Q = packed, *K = packed + plane, *Vlo = packed + 2 * plane,
                 *Vhi = packed + 3 * plane;
    oracle_attn_fwd(Q, K, Vlo, o_lo, lse, (int)BH, N, KD, KD, scale, nthreads);
    oracle_attn_fwd(Q, K, Vhi, o_hi, lse_hi, (int)BH, N, KD, KD, scale, nthreads);
    oracle_merge_attn(o_lo, o_hi, out, B, nh, KD, N, (int)sizeof(double));
    if (vres)
        oracle_extract_v(qkv, vres, B, nh, KD, N, (int)sizeof(double));
    free(lse_hi);
    free(o_lo);
    free(packed);
}

/* Backward of the chain above: dqkv = d(sum(dout o out) + sum(dvres o vres)) / dqkv,
 * obtained by running each step's adjoint in reverse order (dvres may be NULL). */
/* The QKV 1x1 convolution whose NCHW output PsaPackQkv repacks (page "Custom
 * Kernels", section "Position-Sensitive Attention (PSA)": PsaPackQkv takes a QKV
 * conv's NCHW output): qkv[b, o, n] = bias[o] + sum_c w[o, c] x[b, c, n], with
 * x [B, cin, N], w [cout, cin] and bias [cout] (NULL: no bias).  The plain
 * definition, one output element at a time. */
void oracle_qkv_conv(const double *x, const double *w, const double *bias, double *qkv, int B,
                     int cin, int cout, int N)
{
    for (long b = 0; b < B; ++b)
        for (long o = 0; o < cout; ++o)
            for (long n = 0; n < N; ++n) {
                double acc = bias ? bias[o] : 0.0;
                for (long c = 0; c < cin; ++c)
                    acc += w[o * cin + c] * x[(b * cin + c) * N + n];
                qkv[(b * cout + o) * N + n] = acc;
            }
}

/* The attention output with its residual path added: out_res = out + vres, where
 * out is the merged attention output and vres the PsaExtractV output of
 * oracle_psa_fwd (page "Custom Kernels", section "Position-Sensitive Attention
 * (PSA)": PsaExtractV pulls the V section out in NCHW for the residual path; the
 * reading taken is that this path adds it, element by element, to the merged
 * attention output of the same shape).  lse may be NULL. */
void oracle_psa_fwd_residual(const double *qkv, double *out_res, double *lse, int B, int nh,
                             int KD, int N, double scale, int nthreads)
{
    const long n = (long)B * nh * 2 * KD * N;
    double *v = (double *)malloc(sizeof(double) * (size_t)n);
    double *lse_buf = lse ? lse : (double *)malloc(sizeof(double) * (size_t)((long)B * nh * N));
    oracle_psa_fwd(qkv, out_res, lse_buf, v, B, nh, KD, N, scale, nthreads);
    for (long i = 0; i < n; ++i)
        out_res[i] = out_res[i] + v[i];
    if (!lse)
        free(lse_buf);
    free(v);
}

void oracle_psa_bwd(const double *qkv, const double *dout, const double *dvres, double *dqkv,
                    int B, int nh, int KD, int N, double scale, int nthreads)
{
    const long BH = (long)B * nh, plane = BH * N * KD;
    const long C = (long)nh * 4 * KD, c = (long)nh * 2 * KD;
    double *packed = (double *)malloc(sizeof(double) * (size_t)(4 * plane));
    double *dpacked = (double *)malloc(sizeof(double) * (size_t)(4 * plane));
    double *do_lo = (double *)malloc(sizeof(double) * (size_t)(2 * plane));
    double *do_hi = do_lo + plane;
    double *dq2 = (double *)malloc(sizeof(double) * (size_t)(2 * plane));
    double *dk2 = dq2 + plane;
    oracle_pack_qkv(qkv, packed, B, nh, KD, N, (int)sizeof(double));
    oracle_unmerge_attn(dout, do_lo, do_hi, B, nh, KD, N, (int)sizeof(double));
    const double *Q = packed, *K = packed + plane, *Vlo = packed + 2 * plane,
                 *Vhi = packed + 3 * plane;
    double *dQ = dpacked, *dK = dpacked + plane, *dVlo = dpacked + 2 * plane,
           *dVhi = dpacked + 3 * plane;
    oracle_attn_bwd(Q, K, Vlo, do_lo, dQ, dK, dVlo, (int)BH, N, KD, KD, scale, nthreads);
    oracle_attn_bwd(Q, K, Vhi, do_hi, dq2, dk2, dVhi, (int)BH, N, KD, KD, scale, nthreads);
    for (long e = 0; e < plane; ++e) {
        dQ[e] += dq2[e];
        dK[e] += dk2[e];
    }
    oracle_unpack_qkv(dpacked, dqkv, B, nh, KD, N, (int)sizeof(double));
    if (dvres) {
        for (long b = 0; b < B; ++b)
            for (long hd = 0; hd < nh; ++hd)
                for (long j = 0; j < 2 * KD; ++j)
                    for (long n = 0; n < N; ++n)
                        dqkv[(b * C + hd * 4 * KD + 2 * KD + j) * N + n] +=
                            dvres[(b * c + hd * 2 * KD + j) * N + n];
    }
    free(dq2);
    free(do_lo);
    free(dpacked);
    free(packed);
}
