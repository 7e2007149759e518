/*
 * mha_oracle.c -- plain fp64 CPU oracle for scaled dot-product attention and
 * multi-head attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the test suite, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code with the CUDA library.
 *
 * What it computes is the textbook definition, written out with no blocking,
 * fusion or reordering:
 *
 *   Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V
 *     ("Attention Is All You Need" (azimuth.plus), "The idea: every word
 *      queries every word"; cuijiawei.cn "The core idea: scaled dot-product
 *      attention"; aiany.app Step 6, matrix form S = QK^T/sqrt(d_k),
 *      A = softmax(S), Z = AV).
 *   The softmax subtracts the row maximum before exponentiating (azimuth.plus,
 *   "The same idea in code", stable softmax) -- an exact identity.
 *   Masking sets a score to -infinity before the softmax, so its weight is
 *   exactly zero (aiany.app Step 10; notebook chapter "Masked Attention in the
 *   Decoder", e_tj = -inf for j > t; cuijiawei.cn masked_fill(mask == 0, -inf)).
 *   Here a masked key is simply left out of the max, the sum and the weighted
 *   average, which is the same thing.
 *
 *   MultiHead = Concat(head_1..head_h) W^O, head_i = Attention(X_q W_i^Q,
 *   X_kv W_i^K, X_kv W_i^V)  (muhitai.com "Multi-Head Attention Formula";
 *   notebook chapter "Multi-Head Self-Attention" and "The Decoder's
 *   Cross-Attention": Q = s W^Q, K = z W^K, V = z W^V).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - the scale is a parameter (1/sqrt(d_k) by default at the caller);
 *   - causal visibility is top-left aligned: key j is visible to query i iff
 *     j <= i (the pages only define T_q == T_k);
 *   - key padding masks keys j >= key_lens[b]; padded query rows are computed
 *     normally;
 *   - a row with no visible key outputs zeros (the pages' formula gives NaN);
 *     parity for that case is unpinned;
 *   - projections have no bias; head i owns columns [i*d, (i+1)*d) of the
 *     projection matrices and the concatenation is in head order.
 *
 * Layouts (all row-major, contiguous):
 *   q (B,H,Tq,dk)  k (B,H,Tk,dk)  v (B,H,Tk,dv)  o (B,H,Tq,dv)
 *   weights (B,H,Tq,Tk) optional
 *   x_q (B,Tq,D)  x_kv (B,Tk,D)  Wq,Wk (D,H*dk)  Wv (D,H*dv)  Wo (H*dv,D)
 *   out (B,Tq,D)
 *
 * Mask kinds: 0 none, 1 causal, 2 key padding, 3 causal + key padding.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define MASK_CAUSAL_BIT 1
#define MASK_PADDING_BIT 2

/* Is key j visible to query i of batch b? */
static int key_visible(int mask_kind, const int32_t *key_lens, int b, int i, int j)
{
    if ((mask_kind & MASK_CAUSAL_BIT) && j > i)
        return 0;
    if ((mask_kind & MASK_PADDING_BIT) && key_lens && j >= key_lens[b])
        return 0;
    return 1;
}

/* q_i . k_j over the dk key features. */
static double qk_dot(const double *qi, const double *kb, int j, int dk)
{
    double dot = 0.0;
    for (int c = 0; c < dk; ++c)
        dot += qi[c] * kb[(size_t)j * dk + c];
    return dot;
}

/* One output row of scaled dot-product attention.
 * qi: dk values; kb: Tk x dk; vb: Tk x dv; oi: dv values out;
 * wi: Tk weights out (may be NULL); s: Tk doubles of scratch. */
static void sdpa_row(const double *qi, const double *kb, const double *vb, double *oi,
                     double *wi, double *s, int Tk, int dk, int dv, double scale,
                     int mask_kind, const int32_t *key_lens, int b, int i)
{
    int any = 0;
    double m = -INFINITY;
    for (int j = 0; j < Tk; ++j) {
        if (!key_visible(mask_kind, key_lens, b, i, j))
            continue;
        const double dot = qk_dot(qi, kb, j, dk);
        s[j] = scale * dot;
        if (!any || s[j] > m)
            m = s[j];
        any = 1;
    }
    for (int c = 0; c < dv; ++c)
        oi[c] = 0.0;
    if (wi)
        for (int j = 0; j < Tk; ++j)
            wi[j] = 0.0;
    if (!any)
        return; /* no visible key: zero row */

    double denom = 0.0;
    for (int j = 0; j < Tk; ++j) {
        if (!key_visible(mask_kind, key_lens, b, i, j))
            continue;
        s[j] = exp(s[j] - m);
        denom += s[j];
    }
    for (int j = 0; j < Tk; ++j) {
        if (!key_visible(mask_kind, key_lens, b, i, j))
            continue;
        double w = s[j] / denom;
        if (wi)
            wi[j] = w;
        for (int c = 0; c < dv; ++c)
            oi[c] += w * vb[(size_t)j * dv + c];
    }
}

/* Scaled dot-product attention over all rows.  Returns 0, or -1 on a bad
 * argument / allocation failure. */
int oracle_sdpa(const double *q, const double *k, const double *v, double *o,
                double *weights, int B, int H, int Tq, int Tk, int dk, int dv,
                double scale, int mask_kind, const int32_t *key_lens)
{
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || dk <= 0 || dv <= 0)
        return -1;
    long rows = (long)B * H * Tq;
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long r = 0; r < rows; ++r) {
                int i = (int)(r % Tq);
                long bh = r / Tq;
                int b = (int)(bh / H);
                const double *kb = k + (size_t)bh * Tk * dk;
                const double *vb = v + (size_t)bh * Tk * dv;
                sdpa_row(q + (size_t)r * dk, kb, vb, o + (size_t)r * dv,
                         weights ? weights + (size_t)r * Tk : NULL, s, Tk, dk, dv, scale,
                         mask_kind, key_lens, b, i);
            }
            free(s);
        }
    }
    return failed ? -1 : 0;
}

/* Scaled dot-product attention for a list of rows only: rows[n] is the flat
 * index (b*H + h)*Tq + i; o receives n_rows x dv values in list order. */
int oracle_sdpa_rows(const double *q, const double *k, const double *v, double *o,
                     const int64_t *rows, long n_rows, int B, int H, int Tq, int Tk,
                     int dk, int dv, double scale, int mask_kind, const int32_t *key_lens)
{
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || dk <= 0 || dv <= 0)
        return -1;
    long total = (long)B * H * Tq;
    for (long n = 0; n < n_rows; ++n)
        if (rows[n] < 0 || rows[n] >= total)
            return -1;
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long n = 0; n < n_rows; ++n) {
                long r = rows[n];
                int i = (int)(r % Tq);
                long bh = r / Tq;
                int b = (int)(bh / H);
                sdpa_row(q + (size_t)r * dk, k + (size_t)bh * Tk * dk, v + (size_t)bh * Tk * dv,
                         o + (size_t)n * dv, NULL, s, Tk, dk, dv, scale, mask_kind, key_lens,
                         b, i);
            }
            free(s);
        }
    }
    return failed ? -1 : 0;
}

/* y (M x N) = x (M x K) @ W (K x N), plain triple loop. */
static void matmul(const double *x, const double *W, double *y, long M, int K, int N)
{
#pragma omp parallel for schedule(static)
    for (long r = 0; r < M; ++r) {
        double *yr = y + (size_t)r * N;
        for (int n = 0; n < N; ++n)
            yr[n] = 0.0;
        for (int kk = 0; kk < K; ++kk) {
            double a = x[(size_t)r * K + kk];
            const double *wr = W + (size_t)kk * N;
            for (int n = 0; n < N; ++n)
                yr[n] += a * wr[n];
        }
    }
}

/* Split (B, T, H*d) head-major columns into (B, H, T, d). */
static void split_heads(const double *src, double *dst, int B, int T, int H, int d)
{
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t)
            for (int hh = 0; hh < H; ++hh)
                memcpy(dst + (((size_t)b * H + hh) * T + t) * d,
                       src + ((size_t)b * T + t) * H * d + (size_t)hh * d, sizeof(double) * d);
}

/* Multi-head attention.  If query_rows is non-NULL, only those (b*Tq + i)
 * output rows are produced, in list order, into out (n_query_rows x D);
 * otherwise out is (B, Tq, D).  Returns 0 or -1. */
int oracle_mha(const double *x_q, const double *x_kv, const double *Wq, const double *Wk,
               const double *Wv, const double *Wo, double *out, int B, int H, int Tq, int Tk,
               int D, int dk, int dv, double scale, int mask_kind, const int32_t *key_lens,
               const int64_t *query_rows, long n_query_rows)
{
    if (B < 0 || H <= 0 || Tq < 0 || Tk < 0 || D <= 0 || dk <= 0 || dv <= 0)
        return -1;
    long Mq = (long)B * Tq, Mk = (long)B * Tk;
    size_t nq = (size_t)Mq * H * dk, nk = (size_t)Mk * H * dk, nv = (size_t)Mk * H * dv;
    double *qp = malloc(sizeof(double) * (nq ? nq : 1));
    double *kp = malloc(sizeof(double) * (nk ? nk : 1));
    double *vp = malloc(sizeof(double) * (nv ? nv : 1));
    double *qh = malloc(sizeof(double) * (nq ? nq : 1));
    double *kh = malloc(sizeof(double) * (nk ? nk : 1));
    double *vh = malloc(sizeof(double) * (nv ? nv : 1));
    size_t no = (size_t)Mq * H * dv;
    double *oh = malloc(sizeof(double) * (no ? no : 1));
    double *cat = malloc(sizeof(double) * (no ? no : 1));
    int rc = 0;
    if (!qp || !kp || !vp || !qh || !kh || !vh || !oh || !cat) {
        rc = -1;
        goto done;
    }
    /* Projections Q = X_q W^Q, K = X_kv W^K, V = X_kv W^V. */
    matmul(x_q, Wq, qp, Mq, D, H * dk);
    matmul(x_kv, Wk, kp, Mk, D, H * dk);
    matmul(x_kv, Wv, vp, Mk, D, H * dv);
    split_heads(qp, qh, B, Tq, H, dk);
    split_heads(kp, kh, B, Tk, H, dk);
    split_heads(vp, vh, B, Tk, H, dv);

    if (!query_rows) {
        rc = oracle_sdpa(qh, kh, vh, oh, NULL, B, H, Tq, Tk, dk, dv, scale, mask_kind, key_lens);
        if (rc)
            goto done;
        /* Concat(head_1..head_h): (B,H,Tq,dv) -> (B,Tq,H*dv), head order. */
        for (int b = 0; b < B; ++b)
            for (int hh = 0; hh < H; ++hh)
                for (int t = 0; t < Tq; ++t)
                    memcpy(cat + ((size_t)b * Tq + t) * H * dv + (size_t)hh * dv,
                           oh + (((size_t)b * H + hh) * Tq + t) * dv, sizeof(double) * dv);
        matmul(cat, Wo, out, Mq, H * dv, D);
    } else {
        for (long n = 0; n < n_query_rows; ++n)
            if (query_rows[n] < 0 || query_rows[n] >= Mq) {
                rc = -1;
                goto done;
            }
        long nr = n_query_rows * H;
        int64_t *rows = malloc(sizeof(int64_t) * (nr ? nr : 1));
        double *orows = malloc(sizeof(double) * (size_t)(nr ? nr : 1) * dv);
        if (!rows || !orows) {
            free(rows);
            free(orows);
            rc = -1;
            goto done;
        }
        for (long n = 0; n < n_query_rows; ++n) {
            long b = query_rows[n] / Tq, t = query_rows[n] % Tq;
            for (int hh = 0; hh < H; ++hh)
                rows[n * H + hh] = (b * H + hh) * Tq + t;
        }
        rc = oracle_sdpa_rows(qh, kh, vh, orows, rows, nr, B, H, Tq, Tk, dk, dv, scale,
                              mask_kind, key_lens);
        /* orows is already (n, H*dv) in head order: the concatenation. */
        if (!rc)
            matmul(orows, Wo, out, n_query_rows, H * dv, D);
        free(rows);
        free(orows);
    }
done:
    free(qp);
    free(kp);
    free(vp);
    free(qh);
    free(kh);
    free(vh);
    free(oh);
    free(cat);
    return rc;
}

/*
 * Log-sum-exp of each query row's visible scores,
 *   lse_i = log sum_{j visible} exp(scale * q_i . k_j),
 * the normaliser of the softmax (its denominator in log form; the weights
 * are exp(s_j - lse_i)).  Computed as m + log(sum exp(s_j - m)) with m the row
 * maximum, an exact identity.  -inf for a row with no visible key.
 * q (B,H,Tq,dk), k (B,H,Tk,dk), lse (B,H,Tq).
 */
int oracle_sdpa_lse(const double *q, const double *k, double *lse, int B, int H, int Tq, int Tk,
                    int dk, double scale, int mask_kind, const int32_t *key_lens)
{
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || dk <= 0)
        return -1;
    long rows = (long)B * H * Tq;
#pragma omp parallel for schedule(dynamic, 16)
    for (long r = 0; r < rows; ++r) {
        const int i = (int)(r % Tq);
        const long bh = r / Tq;
        const int b = (int)(bh / H);
        const double *qi = q + (size_t)r * dk;
        const double *kb = k + (size_t)bh * Tk * dk;
        double m = -INFINITY;
        for (int j = 0; j < Tk; ++j) {
            if (!key_visible(mask_kind, key_lens, b, i, j))
                continue;
            const double dot = qk_dot(qi, kb, j, dk);
            if (scale * dot > m)
                m = scale * dot;
        }
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int j = 0; j < Tk; ++j) {
            if (!key_visible(mask_kind, key_lens, b, i, j))
                continue;
            const double dot = qk_dot(qi, kb, j, dk);
            sum += exp(scale * dot - m);
        }
        lse[r] = m + log(sum);
    }
    return 0;
}

/*
 * Gradients of scaled dot-product attention, written out from the forward
 * definition by the chain rule (the pages give the forward only; this is its
 * derivative, no further reading needed).  Per (b, h), with S = scale Q K^T
 * (masked entries -inf), P = softmax(S) row-wise, O = P V and an incoming
 * gradient dO:
 *   dV = P^T dO,
 *   dP = dO V^T,
 *   dS_ij = P_ij (dP_ij - sum_l P_il dP_il)      (softmax Jacobian per row),
 *   dQ = scale dS K,   dK = scale dS^T Q.
 * Masked entries have P = 0 and so dS = 0; a row with no visible key has
 * P = 0 everywhere.  q, do (B,H,Tq,d); k, v (B,H,Tk,d); dq (B,H,Tq,d),
 * dk, dv (B,H,Tk,d).  The weights are recomputed here from q and k.
 */
static int sdpa_backward_from(const double *q, const double *k, const double *v, const double *dout,
                              double *dq, double *dk, double *dv, int B, int H, int Tq, int Tk,
                              int d, double scale, int mask_kind, const int32_t *key_lens, int i0)
{
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0 || d <= 0 || i0 < 0 || i0 > Tq)
        return -1;
    const long BH = (long)B * H;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh) {
        const int b = (int)(bh / H);
        const double *qb = q + (size_t)bh * Tq * d, *kb = k + (size_t)bh * Tk * d;
        const double *vb = v + (size_t)bh * Tk * d, *gb = dout + (size_t)bh * Tq * d;
        double *dqb = dq + (size_t)bh * Tq * d, *dkb = dk + (size_t)bh * Tk * d;
        double *dvb = dv + (size_t)bh * Tk * d;
        double *p = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
        if (!p || !dp) {
#pragma omp atomic write
            failed = 1;
            free(p);
            free(dp);
            continue;
        }
        for (size_t x = 0; x < (size_t)Tq * d; ++x)
            dqb[x] = 0.0;
        for (size_t x = 0; x < (size_t)Tk * d; ++x)
            dkb[x] = dvb[x] = 0.0;
        for (int i = i0; i < Tq; ++i) {
            const double *qi = qb + (size_t)i * d, *gi = gb + (size_t)i * d;
            /* P_i (the forward's weights) */
            double m = -INFINITY;
            for (int j = 0; j < Tk; ++j) {
                p[j] = key_visible(mask_kind, key_lens, b, i, j) ? scale * qk_dot(qi, kb, j, d)
                                                                 : -INFINITY;
                if (p[j] > m)
                    m = p[j];
            }
            if (m == -INFINITY)
                continue; /* no visible key: P_i = 0, no gradient flows */
            double den = 0.0;
            for (int j = 0; j < Tk; ++j) {
                p[j] = p[j] == -INFINITY ? 0.0 : exp(p[j] - m);
                den += p[j];
            }
            /* dP_ij = dO_i . V_j and the row sum of P dP */
            double pdp = 0.0;
            for (int j = 0; j < Tk; ++j) {
                p[j] /= den;
                double g = 0.0;
                for (int c = 0; c < d; ++c)
                    g += gi[c] * vb[(size_t)j * d + c];
                dp[j] = g;
                pdp += p[j] * g;
            }
            for (int j = 0; j < Tk; ++j) {
                if (p[j] == 0.0)
                    continue;
                const double ds = p[j] * (dp[j] - pdp);
                for (int c = 0; c < d; ++c) {
                    dvb[(size_t)j * d + c] += p[j] * gi[c];
                    dqb[(size_t)i * d + c] += scale * ds * kb[(size_t)j * d + c];
                    dkb[(size_t)j * d + c] += scale * ds * qi[c];
                }
            }
        }
        free(p);
        free(dp);
    }
    return failed ? -1 : 0;
}

int oracle_sdpa_backward(const double *q, const double *k, const double *v, const double *dout,
                         double *dq, double *dk, double *dv, int B, int H, int Tq, int Tk, int d,
                         double scale, int mask_kind, const int32_t *key_lens)
{
    return sdpa_backward_from(q, k, v, dout, dq, dk, dv, B, H, Tq, Tk, d, scale, mask_kind, key_lens,
                              0);
}

/*
 * The same sums taken over the query rows i >= i0 only (rows before i0 add
 * nothing; their dq rows are left 0).  dq rows i >= i0 are then the full
 * gradient, and under the causal mask (key j visible to row i iff j <= i)
 * so are dk and dv rows j >= i0, which no earlier row sees: the tail of the
 * gradient of a long sequence, at the cost of its last Tq - i0 rows.
 */
int oracle_sdpa_backward_tail(const double *q, const double *k, const double *v,
                              const double *dout, double *dq, double *dk, double *dv, int B, int H,
                              int Tq, int Tk, int d, double scale, int mask_kind,
                              const int32_t *key_lens, int i0)
{
    return sdpa_backward_from(q, k, v, dout, dq, dk, dv, B, H, Tq, Tk, d, scale, mask_kind, key_lens,
                              i0);
}

/*
 * Residual connection and layer normalisation around a sublayer, per row:
 *   v = x + s  (the sublayer's input added back to its output),
 *   y = (v - mu) / sigma * gamma + beta,
 * mu and sigma the mean and standard deviation of v over the D features
 * ("Attention Is All You Need" (aiany.app) Step 9, LayerNorm(x + Sublayer(x));
 * notebook chapter "Layer Normalization and Residual Connections",
 * LayerNorm(x) = (x - mu)/sigma (.) gamma + beta).  Reading where the pages
 * are silent: sigma = sqrt(mean((v - mu)^2) + eps) -- the population standard
 * deviation with a small eps the caller chooses (eps = 0 is the formula as
 * printed).  x, s, y (rows, D); gamma, beta (D).
 */
int oracle_add_layernorm(const double *x, const double *s, const double *gamma,
                         const double *beta, double eps, double *y, long rows, int D)
{
    if (rows < 0 || D <= 0 || eps < 0.0) return 1;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        const double *xr = x + r * D, *sr = s + r * D;
        double *yr = y + r * D;
        double mu = 0.0;
        for (int c = 0; c < D; ++c) mu += xr[c] + sr[c];
        mu /= D;
        double var = 0.0;
        for (int c = 0; c < D; ++c) {
            const double d = xr[c] + sr[c] - mu;
            var += d * d;
        }
        var /= D;
        const double sigma = sqrt(var + eps);
        for (int c = 0; c < D; ++c) yr[c] = (xr[c] + sr[c] - mu) / sigma * gamma[c] + beta[c];
    }
    return 0;
}

/*
 * Sinusoidal positional encoding of positions pos0 .. pos0+T-1 over D
 * features ("Attention is All You Need" notebook chapter and aiany.app Step 8):
 *   PE(pos, 2i)   = sin(pos / 10000^(2i/D)),
 *   PE(pos, 2i+1) = cos(pos / 10000^(2i/D)).
 * pe (T, D).
 */
int oracle_positional_encoding(double *pe, int T, int D, int pos0)
{
    if (T < 0 || D <= 0)
        return -1;
    for (int t = 0; t < T; ++t)
        for (int c = 0; c < D; ++c) {
            const int i2 = c - (c % 2); /* 2i */
            const double angle = (double)(pos0 + t) / pow(10000.0, (double)i2 / D);
            pe[(size_t)t * D + c] = (c % 2 == 0) ? sin(angle) : cos(angle);
        }
    return 0;
}

/*
 * Position-wise feed-forward network, applied to every row independently
 * (aiany.app Step 9; notebook chapter "Feed-Forward Network"):
 *   FFN(x) = max(0, x W1 + b1) W2 + b2.
 * x (M, D), W1 (D, F), b1 (F), W2 (F, D), b2 (D), y (M, D).
 */
int oracle_ffn(const double *x, const double *W1, const double *b1, const double *W2,
               const double *b2, double *y, long M, int D, int F)
{
    if (M < 0 || D <= 0 || F <= 0)
        return -1;
    double *hid = (double *)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1) * F);
    if (!hid)
        return -1;
    matmul(x, W1, hid, M, D, F);
#pragma omp parallel for schedule(static)
    for (long r = 0; r < M; ++r)
        for (int f = 0; f < F; ++f) {
            const double a = hid[(size_t)r * F + f] + b1[f];
            hid[(size_t)r * F + f] = a > 0.0 ? a : 0.0;
        }
    matmul(hid, W2, y, M, F, D);
#pragma omp parallel for schedule(static)
    for (long r = 0; r < M; ++r)
        for (int c = 0; c < D; ++c)
            y[(size_t)r * D + c] += b2[c];
    free(hid);
    return 0;
}

/* Number of host threads OpenMP will use (for reporting). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads the next calls use (the benchmark times the oracle on one thread
 * as well as on all cores); n < 1 is ignored.  No arithmetic depends on it. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
