/*
 * oracle.c -- plain fp64 CPU reference for multi-head scaled dot-product
 * attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes (the definition, written out, no blocking or fusion):
 *
 *   Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k) + M) V
 *     -- "How Transformers Work" (worksonmygpu.com), section "Scaled
 *        dot-product attention", steps 1-4; "The Transformer"
 *        (hoshank.vercel.app), section "The Mathematics", first equation.
 *   M is an additive mask: 0 where key j is visible from query i, -inf where
 *   it is blocked, so that a blocked key gets weight exactly 0
 *     -- "The Transformer" (rayaq.ca), section "Masks: who may look at whom".
 *   Causal: key j is blocked for query i when j > i (the strict upper
 *   triangle, as in the printed 4x4 mask of that section).
 *   Key padding: key j is blocked for every query of batch item b when
 *   j >= key_lengths[b] (one row of the mask per batch item, same section).
 *   Bottom-right causal (decoding against a cache): the Lq queries are the
 *   last Lq positions of the len_b tokens whose keys and values are held
 *   (len_b = key_lengths[b] with key padding, else Lk), so query i sits at
 *   position len_b - Lq + i and key j is blocked when j > len_b - Lq + i --
 *   the decoder's restriction to earlier positions applied while generating
 *   left to right ("How Transformers Work" (worksonmygpu.com), "What changed
 *   since 2017"; "The Transformer" (hoshank.vercel.app), "The Breakthrough";
 *   "The Transformer" (rayaq.ca), "The decoder stack").  With Lq == len_b it
 *   is the causal mask above.
 *   Additive float mask: an optional [Lq, Lk] array A (per batch item and
 *   head through strides, 0 to broadcast) added to the scaled scores like
 *   the causal mask's 0/-inf entries are -- the optional mask of the
 *   reference SDPA the same page describes ("Attention, by hand").
 *
 *   MultiHead(x_q, x_kv) = Concat(head_1, ..., head_h) W^O,
 *   head_i = Attention(x_q W^Q_i, x_kv W^K_i, x_kv W^V_i)
 *     -- "The Transformer" (hoshank.vercel.app), "The Mathematics", the
 *        multi-head equation; "32 Transformer" (ml-canon-en), section
 *        "PyTorch Implementation": the projections are x @ W with W stored
 *        [d_model, d_model], head i is column block [i*d_k, (i+1)*d_k) of the
 *        projection, and the heads are concatenated in head order before
 *        the product with W^O.
 *
 * Readings where the pages leave a step open:
 *   - scale == 0 selects the default 1/sqrt(d_k); any other value is used
 *     as given (the pages only ever use 1/sqrt(d_k)).
 *   - the row maximum is subtracted before exp; softmax is invariant under
 *     that shift, so the result is the definition's.
 *   - a query row with no visible key has no defined softmax (0/0); the
 *     oracle writes NaN there and returns a nonzero status.
 *   - no bias terms (the pages' formula and snippet have none).
 *
 * All arithmetic is IEEE double.  Inputs are double arrays (the exact values
 * the GPU reads, upcast from bf16 or fp32 by the caller).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MASK_CAUSAL 1
#define ORACLE_MASK_KEY_PADDING 2
#define ORACLE_MASK_CAUSAL_BOTTOM_RIGHT 4

/* Additive mask entry M[i][j] for query i of Lq, key j (0 or -inf). */
static double mask_entry(int i, int j, int mask_kind, int len_b, int Lq)
{
    if ((mask_kind & ORACLE_MASK_CAUSAL) && j > i)
        return -INFINITY;
    if ((mask_kind & ORACLE_MASK_CAUSAL_BOTTOM_RIGHT) && j > len_b - Lq + i)
        return -INFINITY;
    if ((mask_kind & ORACLE_MASK_KEY_PADDING) && j >= len_b)
        return -INFINITY;
    return 0.0;
}

/*
 * One query row of attention.
 *   q      : d values
 *   K, V   : Lk rows, row j at K + j*ldk / V + j*ldv, d values each
 *   w      : out, Lk attention weights (softmax of the masked scores)
 *   o      : out, d values, o[c] = sum_j w[j] * V[j][c]
 * Returns 0, or 1 when the row has no visible key (w and o become NaN).
 */
static int attend_row(const double *q, const double *K, ptrdiff_t ldk,
                      const double *V, ptrdiff_t ldv, int Lk, int d,
                      double scale, int i, int Lq, int mask_kind, int len_b,
                      const double *add_row, double *w, double *o)
{
    /* scores s_j = scale * <q, k_j> + M_ij (+ A_ij, an additive float mask
     * row given by the caller, when add_row is not NULL) */
    for (int j = 0; j < Lk; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += q[c] * K[(ptrdiff_t)j * ldk + c];
        w[j] = scale * dot + mask_entry(i, j, mask_kind, len_b, Lq);
        if (add_row)
            w[j] += add_row[j];
    }
    /* row maximum */
    double m = -INFINITY;
    for (int j = 0; j < Lk; ++j)
        if (w[j] > m)
            m = w[j];
    if (m == -INFINITY) {
        for (int j = 0; j < Lk; ++j)
            w[j] = NAN;
        for (int c = 0; c < d; ++c)
            o[c] = NAN;
        return 1;
    }
    /* softmax: exp(s_j - m) / sum_k exp(s_k - m); exp(-inf) is exactly 0 */
    double Z = 0.0;
    for (int j = 0; j < Lk; ++j) {
        w[j] = exp(w[j] - m);
        Z += w[j];
    }
    for (int j = 0; j < Lk; ++j)
        w[j] = w[j] / Z;
    /* weighted sum of value rows */
    for (int c = 0; c < d; ++c)
        o[c] = 0.0;
    for (int j = 0; j < Lk; ++j)
        for (int c = 0; c < d; ++c)
            o[c] += w[j] * V[(ptrdiff_t)j * ldv + c];
    return 0;
}

static double resolve_scale(double scale, int d)
{
    return scale == 0.0 ? 1.0 / sqrt((double)d) : scale;
}

static int len_of(const int32_t *key_lengths, int mask_kind, int b, int Lk)
{
    return (mask_kind & ORACLE_MASK_KEY_PADDING) ? key_lengths[b] : Lk;
}

/*
 * Scaled dot-product attention over [B, H, L, d] tensors.
 *   Q [B,H,Lq,d], K [B,H,Lk,d], V [B,H,Lk,d]  ->  O [B,H,Lq,d]
 *   W (optional, may be NULL) receives the weights [B,H,Lq,Lk].
 * Returns the number of rows that had no visible key.
 */
int oracle_sdpa(const double *Q, const double *K, const double *V, double *O,
                double *W, int B, int H, int Lq, int Lk, int d, double scale,
                int mask_kind, const int32_t *key_lengths, const double *add_mask,
                int64_t add_stride_b, int64_t add_stride_h, int nthreads)
{
    const double sc = resolve_scale(scale, d);
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#endif
    (void)nthreads;
#pragma omp parallel for schedule(dynamic) reduction(+ : bad)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        const int b = (int)(bh / H);
        const int len_b = len_of(key_lengths, mask_kind, b, Lk);
        const double *Qh = Q + (size_t)bh * Lq * d;
        const double *Kh = K + (size_t)bh * Lk * d;
        const double *Vh = V + (size_t)bh * Lk * d;
        double *wrow = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        const int hh = (int)(bh % H);
        for (int i = 0; i < Lq; ++i) {
            const double *arow = add_mask ? add_mask + (int64_t)b * add_stride_b +
                                                (int64_t)hh * add_stride_h + (int64_t)i * Lk
                                          : NULL;
            bad += attend_row(Qh + (size_t)i * d, Kh, d, Vh, d, Lk, d, sc, i, Lq,
                              mask_kind, len_b, arow, wrow, O + ((size_t)bh * Lq + i) * d);
            if (W)
                memcpy(W + ((size_t)bh * Lq + i) * Lk, wrow, sizeof(double) * (size_t)Lk);
        }
        free(wrow);
    }
    return bad;
}

/*
 * The same attention, for a list of query rows only (for workloads whose
 * full output is too costly on the CPU).  rows[r] = (b*H + h)*Lq + i.
 * O_rows receives nrows x d values, row r for rows[r].
 */
int oracle_sdpa_rows(const double *Q, const double *K, const double *V,
                     double *O_rows, const int64_t *rows, int nrows, int B,
                     int H, int Lq, int Lk, int d, double scale, int mask_kind,
                     const int32_t *key_lengths, const double *add_mask,
                     int64_t add_stride_b, int64_t add_stride_h, int nthreads)
{
    const double sc = resolve_scale(scale, d);
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#endif
    (void)nthreads;
    (void)B;
#pragma omp parallel for schedule(dynamic) reduction(+ : bad)
    for (int r = 0; r < nrows; ++r) {
        const int64_t bh = rows[r] / Lq;
        const int i = (int)(rows[r] % Lq);
        const int b = (int)(bh / H);
        const int len_b = len_of(key_lengths, mask_kind, b, Lk);
        const int hh = (int)(bh % H);
        const double *arow = add_mask ? add_mask + (int64_t)b * add_stride_b +
                                            (int64_t)hh * add_stride_h + (int64_t)i * Lk
                                      : NULL;
        double *wrow = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        bad += attend_row(Q + (size_t)rows[r] * d, K + (size_t)bh * Lk * d, d,
                          V + (size_t)bh * Lk * d, d, Lk, d, sc, i, Lq, mask_kind,
                          len_b, arow, wrow, O_rows + (size_t)r * d);
        free(wrow);
    }
    return bad;
}

/* Y[M, N] = X[M, Kd] @ W[Kd, N], all row-major, plain triple loop. */
static void matmul(const double *X, const double *Wt, double *Y, long M, int Kd, int N)
{
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < Kd; ++k)
                acc += X[(size_t)m * Kd + k] * Wt[(size_t)k * N + n];
            Y[(size_t)m * N + n] = acc;
        }
    }
}

/*
 * Multi-head attention layer forward (no biases).
 *   x_q [B,Lq,D], x_kv [B,Lk,D], Wq/Wk/Wv/Wo [D,D] (y = x @ W)
 *   out [B,Lq,D]
 * Head i uses columns [i*d, (i+1)*d) of the projections, d = D/h, and the
 * default scale 1/sqrt(d).  Returns -1 when D % h != 0, else the number of
 * query rows with no visible key.
 */
int oracle_mha(const double *x_q, const double *x_kv, const double *Wq,
               const double *Wk, const double *Wv, const double *Wo,
               double *out, int B, int Lq, int Lk, int D, int h,
               int mask_kind, const int32_t *key_lengths, int nthreads)
{
    if (h <= 0 || D % h != 0)
        return -1;
    const int d = D / h;
    const double sc = 1.0 / sqrt((double)d);
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#endif
    (void)nthreads;
    double *Qp = (double *)malloc(sizeof(double) * (size_t)B * Lq * D + 8);
    double *Kp = (double *)malloc(sizeof(double) * (size_t)B * Lk * D + 8);
    double *Vp = (double *)malloc(sizeof(double) * (size_t)B * Lk * D + 8);
    double *ctx = (double *)malloc(sizeof(double) * (size_t)B * Lq * D + 8);
    /* projections: Q = x_q Wq, K = x_kv Wk, V = x_kv Wv */
    matmul(x_q, Wq, Qp, (long)B * Lq, D, D);
    matmul(x_kv, Wk, Kp, (long)B * Lk, D, D);
    matmul(x_kv, Wv, Vp, (long)B * Lk, D, D);
    /* per head: attention on column block [hh*d, (hh+1)*d); the head's
     * output lands in the same column block of ctx (the concatenation) */
    int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(+ : bad)
    for (long bh = 0; bh < (long)B * h; ++bh) {
        const int b = (int)(bh / h);
        const int hh = (int)(bh % h);
        const int len_b = len_of(key_lengths, mask_kind, b, Lk);
        double *wrow = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        for (int i = 0; i < Lq; ++i) {
            const double *q = Qp + ((size_t)b * Lq + i) * D + (size_t)hh * d;
            const double *Kh = Kp + (size_t)b * Lk * D + (size_t)hh * d;
            const double *Vh = Vp + (size_t)b * Lk * D + (size_t)hh * d;
            double *o = ctx + ((size_t)b * Lq + i) * D + (size_t)hh * d;
            bad += attend_row(q, Kh, D, Vh, D, Lk, d, sc, i, Lq, mask_kind, len_b, NULL, wrow, o);
        }
        free(wrow);
    }
    /* out = Concat(heads) Wo */
    matmul(ctx, Wo, out, (long)B * Lq, D, D);
    free(Qp);
    free(Kp);
    free(Vp);
    free(ctx);
    return bad;
}

/* Y[M, N] = X[M, Kd] @ W[Kd, N] + bias[N] (bias may be NULL). */
static void matmul_bias(const double *X, const double *Wt, const double *bias, double *Y,
                        long M, int Kd, int N)
{
    matmul(X, Wt, Y, M, Kd, N);
    if (!bias)
        return;
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n)
            Y[(size_t)m * N + n] += bias[n];
}

/*
 * LayerNorm of every row of R = A + B ([M, D] each), in place into Y:
 *   Y[m, :] = (R[m, :] - mean) / sqrt(var + eps) * gamma + beta,
 * mean and var (population variance, divisor D) over the row's D values.
 *   -- "The Transformer" (rayaq.ca), "Residuals and LayerNorm": each
 *      position's values are rescaled to mean 0 and variance 1, then a
 *      learned scale and shift are applied; the residual is added first
 *      (post-norm, output = LayerNorm(x + Sublayer(x)), hoshank.vercel.app,
 *      "The Mathematics").
 */
static void add_layernorm(const double *A, const double *B, const double *gamma,
                          const double *beta, double eps, double *Y, long M, int D)
{
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m) {
        double mean = 0.0;
        for (int c = 0; c < D; ++c)
            mean += A[(size_t)m * D + c] + B[(size_t)m * D + c];
        mean /= D;
        double var = 0.0;
        for (int c = 0; c < D; ++c) {
            const double r = A[(size_t)m * D + c] + B[(size_t)m * D + c] - mean;
            var += r * r;
        }
        var /= D;
        const double inv = 1.0 / sqrt(var + eps);
        for (int c = 0; c < D; ++c) {
            const double r = A[(size_t)m * D + c] + B[(size_t)m * D + c] - mean;
            Y[(size_t)m * D + c] = r * inv * gamma[c] + beta[c];
        }
    }
}

/*
 * One post-norm Transformer encoder layer, forward, no dropout:
 *   a   = MultiHead(x, x, x) with biases: Q = x Wq + bq, K = x Wk + bk,
 *         V = x Wv + bv, heads as in oracle_mha, a = Concat(heads) Wo + bo
 *   x1  = LayerNorm1(x + a)
 *   f   = max(0, x1 W1 + b1) W2 + b2          (position-wise FFN)
 *   out = LayerNorm2(x1 + f)
 *   -- hoshank.vercel.app, "The Mathematics" (FFN and sublayer equations);
 *      rayaq.ca, "The feed-forward block", "Residuals and LayerNorm", "The
 *      encoder stack" and the EncoderLayer of "Implementation".
 * Shapes: x, out [B, L, D]; Wq..Wo [D, D]; b* [D]; W1 [D, F]; b1 [F];
 * W2 [F, D]; b2 [D]; ln gamma/beta [D].  Returns -1 when D % h != 0, else
 * the number of query rows with no visible key.
 */
int oracle_encoder_layer(const double *x, const double *Wq, const double *Wk,
                         const double *Wv, const double *Wo, const double *bq,
                         const double *bk, const double *bv, const double *bo,
                         const double *g1, const double *be1, const double *W1,
                         const double *b1, const double *W2, const double *b2,
                         const double *g2, const double *be2, double eps,
                         double *out, int B, int L, int D, int h, int F,
                         int mask_kind, const int32_t *key_lengths, int nthreads)
{
    if (h <= 0 || D % h != 0)
        return -1;
    const int d = D / h;
    const double sc = 1.0 / sqrt((double)d);
    const long M = (long)B * L;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#endif
    (void)nthreads;
    double *Qp = (double *)malloc(sizeof(double) * (size_t)M * D + 8);
    double *Kp = (double *)malloc(sizeof(double) * (size_t)M * D + 8);
    double *Vp = (double *)malloc(sizeof(double) * (size_t)M * D + 8);
    double *ctx = (double *)malloc(sizeof(double) * (size_t)M * D + 8);
    double *a = (double *)malloc(sizeof(double) * (size_t)M * D + 8);
    double *x1 = (double *)malloc(sizeof(double) * (size_t)M * D + 8);
    double *hid = (double *)malloc(sizeof(double) * (size_t)M * F + 8);
    double *f = (double *)malloc(sizeof(double) * (size_t)M * D + 8);
    matmul_bias(x, Wq, bq, Qp, M, D, D);
    matmul_bias(x, Wk, bk, Kp, M, D, D);
    matmul_bias(x, Wv, bv, Vp, M, D, D);
    int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(+ : bad)
    for (long bh = 0; bh < (long)B * h; ++bh) {
        const int b = (int)(bh / h);
        const int hh = (int)(bh % h);
        const int len_b = len_of(key_lengths, mask_kind, b, L);
        double *wrow = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        for (int i = 0; i < L; ++i) {
            const double *q = Qp + ((size_t)b * L + i) * D + (size_t)hh * d;
            const double *Kh = Kp + (size_t)b * L * D + (size_t)hh * d;
            const double *Vh = Vp + (size_t)b * L * D + (size_t)hh * d;
            double *o = ctx + ((size_t)b * L + i) * D + (size_t)hh * d;
            bad += attend_row(q, Kh, D, Vh, D, L, d, sc, i, L, mask_kind, len_b, NULL, wrow, o);
        }
        free(wrow);
    }
    matmul_bias(ctx, Wo, bo, a, M, D, D);
    add_layernorm(x, a, g1, be1, eps, x1, M, D);
    matmul_bias(x1, W1, b1, hid, M, D, F);
#pragma omp parallel for schedule(static)
    for (long i = 0; i < M * F; ++i)
        hid[i] = hid[i] > 0.0 ? hid[i] : 0.0;
    matmul_bias(hid, W2, b2, f, M, F, D);
    add_layernorm(x1, f, g2, be2, eps, out, M, D);
    free(Qp);
    free(Kp);
    free(Vp);
    free(ctx);
    free(a);
    free(x1);
    free(hid);
    free(f);
    return bad;
}

/* Number of parameters of the encoder layer above (weights, biases and the
 * two LayerNorms' scale and shift), for d_model D and FFN width F. */
long oracle_encoder_layer_num_params(int D, int F)
{
    return 4L * D * D + 4L * D          /* Wq, Wk, Wv, Wo and their biases */
           + (long)D * F + F            /* W1, b1 */
           + (long)F * D + D            /* W2, b2 */
           + 2L * (D + D);              /* two LayerNorms: gamma, beta */
}

/*
 * Gradient of scaled dot-product attention (the backward pass of training).
 * Given dO = dL/dO for O = softmax(S) V with S = scale * Q K^T + M, the
 * chain rule through the row softmax gives, per (b, h) and query row i:
 *   P_ij  = softmax_j(S_ij)                  (the forward weights)
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = <dO_i, V_j>
 *   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)  (softmax Jacobian)
 *   dQ_i  = scale * sum_j dS_ij K_j
 *   dK_j  = scale * sum_i dS_ij Q_i
 * Training backpropagates through the attention formula of "How
 * Transformers Work" (worksonmygpu.com), "Scaled dot-product attention";
 * "32 Transformer" (ml-canon-en), "Why we divide by sqrt(dk)", discusses
 * the gradient of this softmax (vanishing at inactive positions of a
 * saturated row).  Masked keys have P = 0, so they receive no gradient.  A
 * query row with no visible key has no defined softmax: its dQ row is NaN
 * and it contributes nothing to dK and dV.  Returns the number of such
 * rows.
 */
int oracle_sdpa_backward(const double *Q, const double *K, const double *V, const double *dO,
                         double *dQ, double *dK, double *dV, int B, int H, int Lq, int Lk, int d,
                         double scale, int mask_kind, const int32_t *key_lengths, int nthreads)
{
    const double sc = resolve_scale(scale, d);
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#endif
    (void)nthreads;
#pragma omp parallel for schedule(dynamic) reduction(+ : bad)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        const int b = (int)(bh / H);
        const int len_b = len_of(key_lengths, mask_kind, b, Lk);
        const double *Qh = Q + (size_t)bh * Lq * d;
        const double *Kh = K + (size_t)bh * Lk * d;
        const double *Vh = V + (size_t)bh * Lk * d;
        const double *dOh = dO + (size_t)bh * Lq * d;
        double *dQh = dQ + (size_t)bh * Lq * d;
        double *dKh = dK + (size_t)bh * Lk * d;
        double *dVh = dV + (size_t)bh * Lk * d;
        for (size_t e = 0; e < (size_t)Lk * d; ++e) {
            dKh[e] = 0.0;
            dVh[e] = 0.0;
        }
        const size_t n = (size_t)(Lk > 0 ? Lk : 1);
        double *w = (double *)malloc(sizeof(double) * n);
        double *dP = (double *)malloc(sizeof(double) * n);
        double *o = (double *)malloc(sizeof(double) * (size_t)(d > 0 ? d : 1));
        for (int i = 0; i < Lq; ++i) {
            const double *q = Qh + (size_t)i * d;
            const double *g = dOh + (size_t)i * d;
            double *dq = dQh + (size_t)i * d;
            if (attend_row(q, Kh, d, Vh, d, Lk, d, sc, i, Lq, mask_kind, len_b, NULL, w, o)) {
                for (int c = 0; c < d; ++c)
                    dq[c] = NAN;
                ++bad;
                continue;
            }
            /* dP_ij = <dO_i, V_j> and its P-weighted row mean */
            double mean = 0.0;
            for (int j = 0; j < Lk; ++j) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c)
                    acc += g[c] * Vh[(size_t)j * d + c];
                dP[j] = acc;
                mean += w[j] * acc;
            }
            for (int c = 0; c < d; ++c)
                dq[c] = 0.0;
            for (int j = 0; j < Lk; ++j) {
                const double ds = w[j] * (dP[j] - mean);
                for (int c = 0; c < d; ++c) {
                    dq[c] += sc * ds * Kh[(size_t)j * d + c];
                    dKh[(size_t)j * d + c] += sc * ds * q[c];
                    dVh[(size_t)j * d + c] += w[j] * g[c];
                }
            }
        }
        free(w);
        free(dP);
        free(o);
    }
    return bad;
}

/*
 * Sinusoidal positional encoding, [n_pos, D] row-major:
 *   PE(pos, 2i)   = sin(pos / 10000^(2i / D))
 *   PE(pos, 2i+1) = cos(pos / 10000^(2i / D))
 * for positions first_pos .. first_pos + n_pos - 1 -- "How Transformers
 * Work" (worksonmygpu.com), "Positional encoding"; "The Transformer"
 * (hoshank.vercel.app), "The Mathematics", the last pair of equations (pos
 * counts from 0; i indexes the dimension pair).  An odd D leaves the last
 * column a sine.
 */
void oracle_sinusoidal_pe(double *pe, int first_pos, int n_pos, int D)
{
    for (int r = 0; r < n_pos; ++r) {
        const double pos = (double)(first_pos + r);
        for (int c = 0; c < D; ++c) {
            const int i = c / 2;
            const double angle = pos / pow(10000.0, (2.0 * i) / (double)D);
            pe[(size_t)r * D + c] = (c % 2 == 0) ? sin(angle) : cos(angle);
        }
    }
}

/*
 * Input of the first layer: x[b, l, :] = table[ids[b, l], :] * scale
 * + PE(pos_offset + l, :), the token embedding scaled by sqrt(d_model) plus
 * the positional encoding ("The Transformer" (rayaq.ca), "Embeddings and
 * positions" and the encode() step of "Implementation"; "The Transformer"
 * (hoshank.vercel.app): the encodings are added to the input embeddings).
 * scale == 0 selects sqrt(D).  Returns the number of ids outside
 * [0, vocab); their rows are NaN.
 */
int oracle_embed_pe(const int32_t *ids, const double *table, int vocab, double *x, int B,
                    int L, int D, int pos_offset, double scale)
{
    const double sc = scale == 0.0 ? sqrt((double)D) : scale;
    double *pe = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)D);
    oracle_sinusoidal_pe(pe, pos_offset, L, D);
    int bad = 0;
    for (int b = 0; b < B; ++b)
        for (int l = 0; l < L; ++l) {
            const int32_t id = ids[(size_t)b * L + l];
            double *row = x + ((size_t)b * L + l) * D;
            if (id < 0 || id >= vocab) {
                for (int c = 0; c < D; ++c)
                    row[c] = NAN;
                ++bad;
                continue;
            }
            for (int c = 0; c < D; ++c)
                row[c] = table[(size_t)id * D + c] * sc + pe[(size_t)l * D + c];
        }
    free(pe);
    return bad;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
