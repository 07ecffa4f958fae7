/*
 * oracle.c -- plain, slow, fp64 CPU reference for causal grouped-query
 * attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes (the plain definitions, no tiling, no online softmax):
 *
 *   "NanoEuler: Hand-writing GPT-2 in Pure C/CUDA", section "Tiled
 *   FlashAttention": the tiled kernel with its online softmax is a faster
 *   route to exact softmax attention, so the reference here is softmax
 *   attention written out row by row:
 *       S_ij  = scale * sum_k Q_ik K_jk
 *       P_ij  = exp(S_ij - m_i) / sum_j' exp(S_ij' - m_i),  m_i = max_j S_ij
 *       O_i   = sum_j P_ij V_j
 *       LSE_i = m_i + ln sum_j exp(S_ij - m_i)          (natural log)
 *   same post, "Architecture Deep Dive": a GPT-2 style decoder-only model,
 *   so the mask is causal: row i sees keys j <= i (diagonal included).
 *   same post, "Build and Run", the config file (num_heads 12,
 *   num_kv_heads 4): grouped-query attention; query head h reads KV head
 *   h / (H / Hkv) (contiguous groups; the post does not say which order).
 *   same post, "Hand-written Backpropagation": the backward is written by
 *   hand; here it is the textbook softmax-attention gradient for an
 *   upstream dO:
 *       dP_ij = sum_k dO_ik V_jk
 *       D_i   = sum_k dO_ik O_ik     (= sum_j P_ij dP_ij, both are returned)
 *       dS_ij = P_ij (dP_ij - D_i)
 *       dQ_i  = scale * sum_j dS_ij K_j
 *       dK_j  = scale * sum_{h in group} sum_i dS_ij Q_i
 *       dV_j  =         sum_{h in group} sum_i P_ij dO_i
 *
 * Layouts: Q, O, dO, dQ are [B][H][N][d]; K, V, dK, dV are [B][Hkv][N][d];
 * LSE and D are [B][H][N].  All doubles, contiguous.
 *
 * Pins (tests/test_oracle.py): closed forms for Q = 0 and for row 0, rows of
 * P summing to one, finite-difference gradients with the pages' epsilon and
 * threshold, constant-V and N = 1 special cases, the dV / dK sum identities,
 * and reduction to textbook softmax attention and to MHA with repeated K/V.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX4(b, h, n, k, Hn, N, d) ((((size_t)(b) * (Hn) + (h)) * (N) + (n)) * (d) + (k))

/* Number of keys row i may attend to. */
static int support_len(int i, int N, int causal) { return causal ? i + 1 : N; }

/*
 * One query row of the forward: fills p[0..len) with the softmax row and
 * returns its max and log-sum-exp.  q, kv point at a row of Q and at the
 * first row of this head's K.
 */
static void softmax_row(const double *q, const double *K, int len, int d,
                        double scale, double *p, double *m_out, double *lse_out) {
    double m = -INFINITY;
    for (int j = 0; j < len; ++j) {
        double s = 0.0;
        for (int k = 0; k < d; ++k) s += q[k] * K[(size_t)j * d + k];
        s *= scale;
        p[j] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int j = 0; j < len; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    for (int j = 0; j < len; ++j) p[j] /= l;
    *m_out = m;
    *lse_out = m + log(l);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward: O [B,H,N,d], LSE [B,H,N]. Returns 0, or -1 on bad sizes / OOM. */
int oracle_attn_fwd_f64(const double *Q, const double *K, const double *V,
                        double *O, double *LSE, int B, int H, int Hkv, int N,
                        int d, double scale, int causal) {
    if (B < 0 || H <= 0 || Hkv <= 0 || N < 0 || d <= 0 || H % Hkv != 0) return -1;
    const int G = H / Hkv;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H), g = h / G;
        double *p = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!p) {
#pragma omp atomic write
            err = 1;
            continue;
        }
        const double *Kg = K + IDX4(b, g, 0, 0, Hkv, N, d);
        const double *Vg = V + IDX4(b, g, 0, 0, Hkv, N, d);
        for (int i = 0; i < N; ++i) {
            const int len = support_len(i, N, causal);
            double m, lse;
            softmax_row(Q + IDX4(b, h, i, 0, H, N, d), Kg, len, d, scale, p, &m, &lse);
            double *o = O + IDX4(b, h, i, 0, H, N, d);
            for (int k = 0; k < d; ++k) o[k] = 0.0;
            for (int j = 0; j < len; ++j)
                for (int k = 0; k < d; ++k) o[k] += p[j] * Vg[(size_t)j * d + k];
            LSE[(size_t)bh * N + i] = lse;
        }
        free(p);
    }
    return err ? -1 : 0;
}

/*
 * Backward.  Recomputes P and O from the definition (it does not take the
 * forward's outputs), then forms the gradients listed in the header.
 * D [B,H,N] receives sum_k dO_ik O_ik and Dalt [B,H,N] receives
 * sum_j P_ij dP_ij; the two must agree (a pin).  Either may be NULL.
 */
int oracle_attn_bwd_f64(const double *Q, const double *K, const double *V,
                        const double *dO, double *dQ, double *dK, double *dV,
                        double *D, double *Dalt, int B, int H, int Hkv, int N,
                        int d, double scale, int causal) {
    if (B < 0 || H <= 0 || Hkv <= 0 || N < 0 || d <= 0 || H % Hkv != 0) return -1;
    const int G = H / Hkv;
    int err = 0;
    /* One (b, KV head) per task: every dK / dV row of the group is written
     * by that task alone. */
#pragma omp parallel for schedule(dynamic, 1)
    for (long bg = 0; bg < (long)B * Hkv; ++bg) {
        const int b = (int)(bg / Hkv), g = (int)(bg % Hkv);
        const size_t n1 = (size_t)(N > 0 ? N : 1);
        double *p = (double *)malloc(sizeof(double) * n1);
        double *dp = (double *)malloc(sizeof(double) * n1);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        if (!p || !dp || !o) {
            free(p); free(dp); free(o);
#pragma omp atomic write
            err = 1;
            continue;
        }
        const double *Kg = K + IDX4(b, g, 0, 0, Hkv, N, d);
        const double *Vg = V + IDX4(b, g, 0, 0, Hkv, N, d);
        double *dKg = dK + IDX4(b, g, 0, 0, Hkv, N, d);
        double *dVg = dV + IDX4(b, g, 0, 0, Hkv, N, d);
        memset(dKg, 0, sizeof(double) * (size_t)N * d);
        memset(dVg, 0, sizeof(double) * (size_t)N * d);
        for (int h = g * G; h < (g + 1) * G; ++h) {
            for (int i = 0; i < N; ++i) {
                const int len = support_len(i, N, causal);
                const double *q = Q + IDX4(b, h, i, 0, H, N, d);
                const double *dor = dO + IDX4(b, h, i, 0, H, N, d);
                double m, lse;
                softmax_row(q, Kg, len, d, scale, p, &m, &lse);
                /* O_i and dP_i */
                for (int k = 0; k < d; ++k) o[k] = 0.0;
                for (int j = 0; j < len; ++j) {
                    double acc = 0.0;
                    for (int k = 0; k < d; ++k) {
                        o[k] += p[j] * Vg[(size_t)j * d + k];
                        acc += dor[k] * Vg[(size_t)j * d + k];
                    }
                    dp[j] = acc;
                }
                double Di = 0.0, Di_alt = 0.0;
                for (int k = 0; k < d; ++k) Di += dor[k] * o[k];
                for (int j = 0; j < len; ++j) Di_alt += p[j] * dp[j];
                const size_t row = ((size_t)b * H + h) * N + i;
                if (D) D[row] = Di;
                if (Dalt) Dalt[row] = Di_alt;
                double *dq = dQ + IDX4(b, h, i, 0, H, N, d);
                for (int k = 0; k < d; ++k) dq[k] = 0.0;
                for (int j = 0; j < len; ++j) {
                    const double ds = p[j] * (dp[j] - Di);
                    for (int k = 0; k < d; ++k) {
                        dq[k] += scale * ds * Kg[(size_t)j * d + k];
                        dKg[(size_t)j * d + k] += scale * ds * q[k];
                        dVg[(size_t)j * d + k] += p[j] * dor[k];
                    }
                }
            }
        }
        free(p); free(dp); free(o);
    }
    return err ? -1 : 0;
}

/*
 * D_i = sum_k dO_ik O_ik over `rows` rows of width d: the backward's
 * per-row correction term, taken on whatever O the caller passes.
 */
int oracle_rowdot_f64(const double *O, const double *dO, double *D, long rows, int d) {
    if (rows < 0 || d <= 0) return -1;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int k = 0; k < d; ++k) acc += O[(size_t)r * d + k] * dO[(size_t)r * d + k];
        D[r] = acc;
    }
    return 0;
}

/*
 * Rotary position embedding of rows of width d (d even), fp64.
 *
 * "NanoEuler: modelo GPT-2 ... en C puro sin PyTorch" and "NanoEuler:
 * Hand-writing GPT-2 in Pure C/CUDA", FAQ on llm.c: the model uses RoPE, with
 * no formula given.  Taken here as the original rotary embedding: row r of a
 * [rows][d] array sits at position n = r % N (rows are [heads][N] flattened);
 * each pair (x_2i, x_2i+1) is turned by the angle n * theta_i with
 *     theta_i = base^(-2i/d),   i = 0 .. d/2 - 1,
 *     y_2i   = x_2i cos(a) - x_2i+1 sin(a)
 *     y_2i+1 = x_2i sin(a) + x_2i+1 cos(a).
 * `inverse` turns by -a instead (the transpose of the rotation): applied to
 * the gradient with respect to the rotated rows it gives the gradient with
 * respect to the unrotated ones.
 */
int oracle_rope_f64(const double *X, double *Y, long rows, int N, int d, double base,
                    int inverse) {
    if (rows < 0 || N < 1 || d < 2 || (d & 1) || !(base > 0.0)) return -1;
    const double sgn = inverse ? -1.0 : 1.0;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        const double n = (double)(r % N);
        for (int i = 0; i < d / 2; ++i) {
            const double theta = pow(base, -2.0 * i / d);
            const double a = sgn * n * theta;
            const double c = cos(a), s = sin(a);
            const double x0 = X[(size_t)r * d + 2 * i], x1 = X[(size_t)r * d + 2 * i + 1];
            Y[(size_t)r * d + 2 * i] = x0 * c - x1 * s;
            Y[(size_t)r * d + 2 * i + 1] = x0 * s + x1 * c;
        }
    }
    return 0;
}

/*
 * Decode attention over a key/value cache, fp64 (the inference use the pages
 * mention: "NanoEuler: Hand-writing GPT-2 in Pure C/CUDA", FAQ on production
 * inference -- inference works, without paged or batched caches).
 *
 * Reading taken: batch element b holds a contiguous cache of L_b = lens[b]
 * rows (1 <= L_b <= Lmax) that already includes the nq new tokens, so new
 * token t (0 <= t < nq, nq <= L_b) sits at position L_b - nq + t and, under
 * the decoder's causal mask, sees cache rows 0 .. L_b - nq + t.  Query head h
 * reads KV head h / (H / Hkv).  Row by row, the plain softmax:
 *     S_j = scale * q . k_j,  O = sum_j softmax(S)_j v_j,  LSE = ln sum_j e^S_j
 * Layouts: Q, O [B][H][nq][d]; Kc, Vc [B][Hkv][Lmax][d]; LSE [B][H][nq].
 */
int oracle_attn_decode_f64(const double *Q, const double *Kc, const double *Vc, const int *lens,
                           double *O, double *LSE, int B, int H, int Hkv, int nq, int Lmax,
                           int d, double scale) {
    if (B < 1 || H < 1 || Hkv < 1 || nq < 1 || Lmax < 1 || d < 1 || H % Hkv) return -1;
    for (int b = 0; b < B; ++b)
        if (lens[b] < nq || lens[b] > Lmax) return -1;
    const int G = H / Hkv;
    int err = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)Lmax);
        if (!p) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for collapse(2) schedule(dynamic)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < H; ++h) {
                if (!p) continue;
                const int g = h / G, L = lens[b];
                const double *K = Kc + ((size_t)b * Hkv + g) * Lmax * d;
                const double *V = Vc + ((size_t)b * Hkv + g) * Lmax * d;
                for (int t = 0; t < nq; ++t) {
                    const double *q = Q + (((size_t)b * H + h) * nq + t) * d;
                    const int len = L - nq + t + 1;
                    double m = -INFINITY;
                    for (int j = 0; j < len; ++j) {
                        double s = 0.0;
                        for (int k = 0; k < d; ++k) s += q[k] * K[(size_t)j * d + k];
                        p[j] = scale * s;
                        if (p[j] > m) m = p[j];
                    }
                    double l = 0.0;
                    for (int j = 0; j < len; ++j) {
                        p[j] = exp(p[j] - m);
                        l += p[j];
                    }
                    double *o = O + (((size_t)b * H + h) * nq + t) * d;
                    for (int k = 0; k < d; ++k) o[k] = 0.0;
                    for (int j = 0; j < len; ++j)
                        for (int k = 0; k < d; ++k) o[k] += p[j] / l * V[(size_t)j * d + k];
                    LSE[((size_t)b * H + h) * nq + t] = m + log(l);
                }
            }
        free(p);
    }
    return err ? -1 : 0;
}
