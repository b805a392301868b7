/*
 * fp64 CPU oracle for the FlashAttention-2 forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition that the CUDA path is checked against.  Only the tests, the
 * package smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes is plain scaled-dot-product attention written as the
 * three-pass softmax of the pages, not the tiled method:
 *   "Flash Attention 全解析(上)", section 1.2 (标准 Attention 的三趟式计算流程):
 *     pass 1  S = Q K^T (scaled), row max m
 *     pass 2  l = rowsum exp(S - m)
 *     pass 3  O = (exp(S - m) / l) V
 *   "FlashAttention 怎么做?online softmax 怎么更新?", section "shape" and the
 *   FlashAttention-2 follow-up question: one logsumexp per row, L = m + log l.
 * The tiled method reaches exactly this result up to rounding order (the same
 * page, "online softmax" paragraph: the block-wise l equals the one-shot sum).
 *
 * Readings taken where the pages are silent:
 *   - inputs are bf16 or fp16 bit patterns (fp16: the input dtype of the
 *     "Triton内核实战" wrapper); each is widened exactly to double, so the
 *     oracle sees the same rounded values the GPU sees;
 *   - scale is the caller's float, widened (not recomputed as 1/sqrt(d));
 *   - causal masking is top-left aligned: row i keeps keys j <= i (and j < Nk).
 *     Masked keys are excluded from all three passes, so no row is ever empty
 *     while Nk >= 1;
 *   - logsumexp is the natural logarithm of the sum over kept keys of
 *     exp(scaled score).
 *
 * Layout: Q [B,H,Nq,d], K and V [B,H,Nk,d], all contiguous (BHSD).  Outputs
 * are double: O [rows, d] and LSE [rows].
 *
 * oracle_attention_backward (below) gives the gradients of the same
 * definition with respect to Q, K and V.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact widening of a bf16 bit pattern: bf16 is the upper half of a binary32. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Exact widening of an IEEE 754 binary16 bit pattern: 1 sign bit, 5 exponent
 * bits (bias 15), 10 fraction bits; exponent 0 encodes zero and subnormals
 * (fraction * 2^-24), exponent 31 encodes infinities and NaNs. */
static double fp16_bits_to_double(uint16_t bits)
{
    const int sign = (bits >> 15) & 1;
    const int exponent = (bits >> 10) & 0x1f;
    const int fraction = bits & 0x3ff;
    double v;
    if (exponent == 0)
        v = ldexp((double)fraction, -24);
    else if (exponent == 31)
        v = fraction ? NAN : INFINITY;
    else
        v = ldexp((double)(fraction | 0x400), exponent - 25);
    return sign ? -v : v;
}

/* Input element types. */
enum { ORACLE_BF16 = 0, ORACLE_FP16 = 1 };

static double widen(uint16_t bits, int dtype)
{
    return dtype == ORACLE_FP16 ? fp16_bits_to_double(bits) : bf16_bits_to_double(bits);
}

typedef struct {
    const uint16_t *Q, *K, *V;
    int64_t H, Nq, Nk, d;
    int causal;
    int dtype;
    double scale;
    const int64_t *rows;    /* flattened (b*H + h)*Nq + i; NULL = all rows */
    int64_t nrows;
    double *O, *LSE;        /* indexed by position in the row list */
    int64_t next;           /* shared work counter (atomic) */
    int error;
} oracle_job;

/* One output row, three passes over the kept keys. */
static void attend_one_row(const oracle_job *J, int64_t flat, double *s,
                           double *o, double *lse)
{
    const int64_t d = J->d;
    const int64_t bh = flat / J->Nq;
    const int64_t i = flat % J->Nq;
    const uint16_t *q = J->Q + flat * d;
    const uint16_t *kb = J->K + bh * J->Nk * d;
    const uint16_t *vb = J->V + bh * J->Nk * d;

    /* kept key set J_i: all keys, or j <= i under the causal mask */
    int64_t n = J->Nk;
    if (J->causal && i + 1 < n)
        n = i + 1;

    /* pass 1: scaled scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c)
            acc += widen(q[c], J->dtype) * widen(kb[j * d + c], J->dtype);
        s[j] = J->scale * acc;
        if (s[j] > m)
            m = s[j];
    }

    /* pass 2: normaliser */
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j)
        l += exp(s[j] - m);

    /* pass 3: normalised weights times V */
    for (int64_t c = 0; c < d; ++c)
        o[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double w = exp(s[j] - m) / l;
        for (int64_t c = 0; c < d; ++c)
            o[c] += w * widen(vb[j * d + c], J->dtype);
    }
    *lse = m + log(l);
}

#define ORACLE_CHUNK 8

static void *oracle_worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    double *s = (double *)malloc((size_t)(J->Nk > 0 ? J->Nk : 1) * sizeof(double));
    if (!s) {
        __atomic_store_n(&J->error, 1, __ATOMIC_RELAXED);
        return NULL;
    }
    for (;;) {
        int64_t start = __atomic_fetch_add(&J->next, ORACLE_CHUNK, __ATOMIC_RELAXED);
        if (start >= J->nrows)
            break;
        int64_t end = start + ORACLE_CHUNK < J->nrows ? start + ORACLE_CHUNK : J->nrows;
        for (int64_t r = start; r < end; ++r) {
            int64_t flat = J->rows ? J->rows[r] : r;
            attend_one_row(J, flat, s, J->O + r * J->d, J->LSE + r);
        }
    }
    free(s);
    return NULL;
}

/*
 * Attention for a list of output rows.
 *   rows   flattened row ids (b*H + h)*Nq + i, or NULL for every row in order;
 *   nrows  number of rows to compute (must be B*H*Nq when rows is NULL);
 *   O      nrows*d doubles, LSE nrows doubles, written in row-list order;
 *   nthreads  worker threads (<= 0: one).
 * Returns 0 on success, 1 on a bad argument (including a row id out of
 * range or Nk < 1), 2 if a worker could not allocate its score buffer.
 */
int oracle_attention_rows_typed(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                                int causal, float scale, int dtype, const int64_t *rows,
                                int64_t nrows, double *O, double *LSE, int nthreads)
{
    if (!Q || !K || !V || !O || !LSE || B < 0 || H < 0 || Nq < 0 || Nk < 1 || d < 1 || nrows < 0)
        return 1;
    if (dtype != ORACLE_BF16 && dtype != ORACLE_FP16)
        return 1;
    const int64_t total = B * H * Nq;
    if (!rows && nrows != total)
        return 1;
    if (rows)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= total)
                return 1;
    if (nrows == 0)
        return 0;

    oracle_job J;
    J.Q = Q; J.K = K; J.V = V;
    J.H = H; J.Nq = Nq; J.Nk = Nk; J.d = d;
    J.causal = causal ? 1 : 0;
    J.dtype = dtype;
    J.scale = (double)scale;
    J.rows = rows; J.nrows = nrows;
    J.O = O; J.LSE = LSE;
    J.next = 0; J.error = 0;

    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 1024)
        nthreads = 1024;
    pthread_t tid[1024];
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[started], NULL, oracle_worker, &J) != 0)
            break;
        ++started;
    }
    oracle_worker(&J);
    for (int t = 0; t < started; ++t)
        pthread_join(tid[t], NULL);
    return J.error ? 2 : 0;
}

/* bf16 inputs (the original entry point). */
int oracle_attention_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                          int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                          int causal, float scale, const int64_t *rows, int64_t nrows,
                          double *O, double *LSE, int nthreads)
{
    return oracle_attention_rows_typed(Q, K, V, B, H, Nq, Nk, d, causal, scale, ORACLE_BF16,
                                       rows, nrows, O, LSE, nthreads);
}

/* Widened value of one 16-bit pattern (exposed for the widening pins). */
double oracle_widen(uint16_t bits, int dtype)
{
    return widen(bits, dtype);
}

/*
 * Gradients of the attention above (the backward pass).  The pages name a
 * backward pass that recomputes the scores from the saved logsumexp
 * ("FlashAttention 怎么做?", FlashAttention-2 question; "Triton内核实战",
 * closing section) but print no formulas, so this is the chain rule of the
 * definition, written out for an upstream gradient dO:
 *   s_ij  = scale q_i . k_j            (j in J_i)
 *   p_ij  = exp(s_ij - LSE_i)          (the softmax weights)
 *   dV_j  = sum over rows i with j in J_i of p_ij dO_i
 *   dp_ij = dO_i . v_j
 *   D_i   = sum_{j in J_i} p_ij dp_ij  (softmax Jacobian: the row term)
 *   ds_ij = p_ij (dp_ij - D_i)
 *   dQ_i  = scale sum_{j in J_i} ds_ij k_j
 *   dK_j  = scale sum over rows i with j in J_i of ds_ij q_i
 * Alongside each output element it returns a magnitude from which rounding
 * bounds for a low-precision implementation follow:
 *   M_dV_jc = sum_i p_ij |dO_ic|
 *   M_dQ_ic = scale sum_j (|ds_ij| + p_ij A_i) |k_jc|
 *   M_dK_jc = scale sum_i (|ds_ij| + p_ij A_i) |q_ic|
 * with A_i = sum_j p_ij sum_c |dO_ic| |v_jc|.  Rounding p (for dV) or ds
 * (for dQ, dK) to a b-bit significand moves an element by at most 2^-b times
 * the |p| or |ds| part; computing D_i from an output o_i whose weights were
 * rounded that way moves D_i by at most 2^-b A_i, hence ds_ij by p_ij 2^-b
 * A_i, which the p_ij A_i part covers.
 */
typedef struct {
    const uint16_t *Q, *K, *V, *dO;
    int64_t Nq, Nk, d;
    int causal, dtype;
    double scale;
    int64_t bh;                 /* head being processed */
    double *LSE, *Dr, *Ar;      /* per query row of the head (phase 1 output) */
    double *dQ, *dK, *dV, *MdQ, *MdK, *MdV;   /* this head's slices */
    int64_t next, count;
    int phase, error;
} oracle_bwd_job;

static int64_t kept_keys(const oracle_bwd_job *J, int64_t i)
{
    return (J->causal && i + 1 < J->Nk) ? i + 1 : J->Nk;
}

/* Phase 1, query row i: LSE_i, D_i and dQ_i. */
static void bwd_query_row(oracle_bwd_job *J, int64_t i, double *s, double *dp, double *da)
{
    const int64_t d = J->d;
    const uint16_t *q = J->Q + (J->bh * J->Nq + i) * d;
    const uint16_t *g = J->dO + (J->bh * J->Nq + i) * d;
    const uint16_t *kb = J->K + J->bh * J->Nk * d;
    const uint16_t *vb = J->V + J->bh * J->Nk * d;
    const int64_t n = kept_keys(J, i);
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0, gv = 0.0, ga = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            acc += widen(q[c], J->dtype) * widen(kb[j * d + c], J->dtype);
            gv += widen(g[c], J->dtype) * widen(vb[j * d + c], J->dtype);
            ga += fabs(widen(g[c], J->dtype)) * fabs(widen(vb[j * d + c], J->dtype));
        }
        s[j] = J->scale * acc;
        dp[j] = gv;
        da[j] = ga;
        if (s[j] > m)
            m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j)
        l += exp(s[j] - m);
    const double lse = m + log(l);
    double D = 0.0, A = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        D += exp(s[j] - lse) * dp[j];
        A += exp(s[j] - lse) * da[j];
    }
    J->LSE[i] = lse;
    J->Dr[i] = D;
    J->Ar[i] = A;
    double *dq = J->dQ + i * d, *mq = J->MdQ ? J->MdQ + i * d : NULL;
    for (int64_t c = 0; c < d; ++c) {
        dq[c] = 0.0;
        if (mq)
            mq[c] = 0.0;
    }
    for (int64_t j = 0; j < n; ++j) {
        const double ds = exp(s[j] - lse) * (dp[j] - D);
        const double w = fabs(ds) + exp(s[j] - lse) * A;
        for (int64_t c = 0; c < d; ++c) {
            const double kc = widen(kb[j * d + c], J->dtype);
            dq[c] += J->scale * ds * kc;
            if (mq)
                mq[c] += J->scale * w * fabs(kc);
        }
    }
}

/* Phase 2, key row j: dK_j and dV_j over the rows that keep key j. */
static void bwd_key_row(oracle_bwd_job *J, int64_t j)
{
    const int64_t d = J->d;
    const uint16_t *k = J->K + (J->bh * J->Nk + j) * d;
    const uint16_t *v = J->V + (J->bh * J->Nk + j) * d;
    const uint16_t *qb = J->Q + J->bh * J->Nq * d;
    const uint16_t *gb = J->dO + J->bh * J->Nq * d;
    double *dk = J->dK + j * d, *dv = J->dV + j * d;
    double *mk = J->MdK ? J->MdK + j * d : NULL, *mv = J->MdV ? J->MdV + j * d : NULL;
    for (int64_t c = 0; c < d; ++c) {
        dk[c] = dv[c] = 0.0;
        if (mk)
            mk[c] = mv[c] = 0.0;
    }
    for (int64_t i = 0; i < J->Nq; ++i) {
        if (j >= kept_keys(J, i))
            continue;
        double acc = 0.0, gv = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            acc += widen(qb[i * d + c], J->dtype) * widen(k[c], J->dtype);
            gv += widen(gb[i * d + c], J->dtype) * widen(v[c], J->dtype);
        }
        const double p = exp(J->scale * acc - J->LSE[i]);
        const double ds = p * (gv - J->Dr[i]);
        const double w = fabs(ds) + p * J->Ar[i];
        for (int64_t c = 0; c < d; ++c) {
            const double qc = widen(qb[i * d + c], J->dtype);
            const double gc = widen(gb[i * d + c], J->dtype);
            dv[c] += p * gc;
            dk[c] += J->scale * ds * qc;
            if (mk) {
                mv[c] += p * fabs(gc);
                mk[c] += J->scale * w * fabs(qc);
            }
        }
    }
}

static void *oracle_bwd_worker(void *arg)
{
    oracle_bwd_job *J = (oracle_bwd_job *)arg;
    const int64_t len = (J->Nk > J->Nq ? J->Nk : J->Nq) + 1;
    double *s = (double *)malloc((size_t)len * sizeof(double));
    double *dp = (double *)malloc((size_t)len * sizeof(double));
    double *da = (double *)malloc((size_t)len * sizeof(double));
    if (!s || !dp || !da) {
        __atomic_store_n(&J->error, 1, __ATOMIC_RELAXED);
        free(s);
        free(dp);
        free(da);
        return NULL;
    }
    for (;;) {
        int64_t r = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (r >= J->count)
            break;
        if (J->phase == 1)
            bwd_query_row(J, r, s, dp, da);
        else
            bwd_key_row(J, r);
    }
    free(s);
    free(dp);
    free(da);
    return NULL;
}

static int run_bwd_phase(oracle_bwd_job *J, int phase, int64_t count, int nthreads)
{
    J->phase = phase;
    J->count = count;
    J->next = 0;
    pthread_t tid[1024];
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[started], NULL, oracle_bwd_worker, J) != 0)
            break;
        ++started;
    }
    oracle_bwd_worker(J);
    for (int t = 0; t < started; ++t)
        pthread_join(tid[t], NULL);
    return J->error;
}

/*
 * Gradients for selected heads.
 *   Q [B,H,Nq,d], K and V [B,H,Nk,d], dO [B,H,Nq,d]: 16-bit patterns of `dtype`;
 *   heads   flattened head ids b*H + h (NULL: every head in order), nheads of them;
 *   dQ      nheads*Nq*d doubles, dK and dV nheads*Nk*d doubles (head-list order);
 *   MdQ, MdK, MdV  the matching absolute-term sums, or all three NULL.
 * Returns 0 on success, 1 on a bad argument, 2 if memory ran out.
 */
int oracle_attention_backward(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                              const uint16_t *dO, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                              int64_t d, int causal, float scale, int dtype, const int64_t *heads,
                              int64_t nheads, double *dQ, double *dK, double *dV, double *MdQ,
                              double *MdK, double *MdV, int nthreads)
{
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV || B < 0 || H < 0 || Nq < 0 || Nk < 1 ||
        d < 1 || nheads < 0)
        return 1;
    if (dtype != ORACLE_BF16 && dtype != ORACLE_FP16)
        return 1;
    if (!((MdQ && MdK && MdV) || (!MdQ && !MdK && !MdV)))
        return 1;
    if (!heads && nheads != B * H)
        return 1;
    if (heads)
        for (int64_t t = 0; t < nheads; ++t)
            if (heads[t] < 0 || heads[t] >= B * H)
                return 1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 1024)
        nthreads = 1024;
    double *lse = (double *)malloc((size_t)(Nq > 0 ? Nq : 1) * sizeof(double));
    double *dr = (double *)malloc((size_t)(Nq > 0 ? Nq : 1) * sizeof(double));
    double *ar = (double *)malloc((size_t)(Nq > 0 ? Nq : 1) * sizeof(double));
    if (!lse || !dr || !ar) {
        free(lse);
        free(dr);
        free(ar);
        return 2;
    }
    oracle_bwd_job J;
    J.Q = Q; J.K = K; J.V = V; J.dO = dO;
    J.Nq = Nq; J.Nk = Nk; J.d = d;
    J.causal = causal ? 1 : 0;
    J.dtype = dtype;
    J.scale = (double)scale;
    J.LSE = lse; J.Dr = dr; J.Ar = ar;
    J.error = 0;
    int rc = 0;
    for (int64_t t = 0; t < nheads && rc == 0; ++t) {
        J.bh = heads ? heads[t] : t;
        J.dQ = dQ + t * Nq * d;
        J.dK = dK + t * Nk * d;
        J.dV = dV + t * Nk * d;
        J.MdQ = MdQ ? MdQ + t * Nq * d : NULL;
        J.MdK = MdK ? MdK + t * Nk * d : NULL;
        J.MdV = MdV ? MdV + t * Nk * d : NULL;
        if (run_bwd_phase(&J, 1, Nq, nthreads) || run_bwd_phase(&J, 2, Nk, nthreads))
            rc = 2;
    }
    free(lse);
    free(dr);
    free(ar);
    return rc;
}

/* Every row of every (b, h): O [B,H,Nq,d], LSE [B,H,Nq]. */
int oracle_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                     int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                     int causal, float scale, double *O, double *LSE, int nthreads)
{
    return oracle_attention_rows(Q, K, V, B, H, Nq, Nk, d, causal, scale,
                                 NULL, B * H * Nq, O, LSE, nthreads);
}
