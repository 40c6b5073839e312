/*
 * wide_oracle.c -- plain, slow, obviously-correct CPU restatement of the
 * group-masked projections of WIDE (token-level dynamic width pruning).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library) shares no code, header, table or helper with this file.
 *
 * Source: "WIDE: Boosting Adaptive LLM Inference via Token-level Dynamic
 * Width Pruning" (arXiv 2607.28418, HTML version).
 *   - Sec. 3.3, Eq. 7: per-routing-column SortDesc giving the reordered mask
 *     and the gather/scatter index I.
 *   - App. B, "metadata shared by all three kernels": the index identity
 *     reordered[j,g] = M[I[j,g], g]; (B,T) flattened to M rows.
 *   - Sec. 3.1, Eq. 3: FFN unit, ((phi(X Wg^T) (.) (X Wu^T)) (.)_G M) Wd^T.
 *   - Sec. 3.1, Eq. 2: attention unit (q_proj pruned on out-features,
 *     o_proj on in-features), G = (Hq/Hk) d.
 *   - App. B, "Implementation of GEMM-K", Eq. 21:
 *     C[m,n] = sum_g M[m,g] sum_{k in K_g} A[m,k] B[n,k].
 *   - App. B "Implementation of Attention" (decoding paragraph) with Sec. 3.1
 *     Eq. 2: routed decode attention, one routing group per GQA group
 *     (G = (Hq/Hk) d), softmax(q K^T / sqrt(d)) V for active groups.
 *   - App. B "Implementation of Attention" (prefill, Algorithm 4): routed
 *     causal attention over the query rows of active (token, group) pairs,
 *     dense K/V, zeros for inactive rows.
 *   - Sec. 3.1 "Routing Components", Eq. 4-5: bottleneck router
 *     R = reshape(X W1 W2) in R^{T x N_G x 2}, inference mask
 *     M = 1[argmax_c R[...,c] = 0] (class 0 executes, class 1 skips).
 *
 * Arithmetic: every bf16 input is decoded exactly to double and every sum
 * is accumulated in double (the pages fix no precision; double makes the
 * rounding of this file negligible against the GPU's bf16/fp32 path).
 * Loops run in the order of the definitions; the only parallelism is an
 * OpenMP loop over independent tokens (rows).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - phi is SiLU, x * sigmoid(x) (Llama backbones, Sec. 4.1).
 *   - SortDesc is stable: active rows first, then inactive rows, each part
 *     in ascending original row index; I is a full permutation.
 *   - A mask byte != 0 means "active".
 *   - Channel f belongs to group floor(f / G) (contiguous groups, Sec. 3.1).
 *   - Weights are stored [out_features, in_features] (B in R^{N x K}, Sec. 3.3);
 *     the router's W1 (D x r on the page) is stored [r, D] and W2 (r x 2N_G)
 *     is stored [2N_G, r].
 *   - The reshape of the 2N_G router outputs to (N_G, 2) is row-major: output
 *     column 2g + c is class c of group g.
 *   - argmax over the two classes returns the first maximum, so a tie
 *     (R[t,g,0] == R[t,g,1]) selects class 0: the group executes.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* Exact bf16 -> double: a bf16 value is the upper half of an IEEE float. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* SiLU, the reading of the element-wise activation phi of Eq. 3. */
static double silu(double a)
{
    return a / (1.0 + exp(-a));
}

int oracle_version(void) { return 1; }

/*
 * Eq. 7 (Sec. 3.3) and App. B Algorithm 1: for every routing column g,
 * SortDesc(M[:,g]) -- a stable partition of the rows, active first.
 *   mask   : uint8 [T, n_groups] row-major, != 0 means active
 *   perm   : int32 [n_groups, T]  (perm[g*T + j] = I[j, g])
 *   counts : int32 [n_groups]     (length of the active prefix)
 */
void oracle_reorder(const uint8_t *mask, int T, int n_groups,
                    int32_t *perm, int32_t *counts)
{
    for (int g = 0; g < n_groups; ++g) {
        int c = 0;
        for (int t = 0; t < T; ++t)
            if (mask[(size_t)t * n_groups + g] != 0)
                perm[(size_t)g * T + c++] = t;
        counts[g] = c;
        for (int t = 0; t < T; ++t)
            if (mask[(size_t)t * n_groups + g] == 0)
                perm[(size_t)g * T + c++] = t;
    }
}

/*
 * GEMM-MN without activation (Sec. 3.1 Eq. 2 for q_proj; App. B
 * "Implementation of GEMM-MN"): Y[t, n] = M[t, n/G] * sum_k X[t,k] W[n,k].
 *   X : bf16 [T, K], W : bf16 [N, K], mask : uint8 [T, N/G], Y : double [R, N]
 *   rows : optional list of R token indices to evaluate (NULL = all T rows,
 *          R = T); output row i is token rows[i].
 */
void oracle_proj_mn(const uint16_t *X, const uint16_t *W, const uint8_t *mask,
                    int T, int K, int N, int G,
                    const int32_t *rows, int n_rows, double *Y)
{
    const int n_groups = N / G;
    const int R = rows ? n_rows : T;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < R; ++i) {
        const int t = rows ? rows[i] : i;
        for (int n = 0; n < N; ++n) {
            double y = 0.0;
            if (mask[(size_t)t * n_groups + n / G] != 0) {
                for (int k = 0; k < K; ++k)
                    y += bf16_to_double(X[(size_t)t * K + k]) *
                         bf16_to_double(W[(size_t)n * K + k]);
            }
            Y[(size_t)i * N + n] = y;
        }
    }
}

/*
 * FFN up/gate half of Eq. 3 (Sec. 3.1), GEMM-MN with the fused activation:
 *   H[t, f] = M[t, f/G] * silu(sum_d X[t,d] Wg[f,d]) * (sum_d X[t,d] Wu[f,d])
 *   X : bf16 [T, D], Wg, Wu : bf16 [F, D], mask : uint8 [T, F/G],
 *   H : double [R, F] (rows as in oracle_proj_mn).
 */
void oracle_gate_up(const uint16_t *X, const uint16_t *Wg, const uint16_t *Wu,
                    const uint8_t *mask, int T, int D, int F, int G,
                    const int32_t *rows, int n_rows, double *H)
{
    const int n_groups = F / G;
    const int R = rows ? n_rows : T;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < R; ++i) {
        const int t = rows ? rows[i] : i;
        for (int f = 0; f < F; ++f) {
            double h = 0.0;
            if (mask[(size_t)t * n_groups + f / G] != 0) {
                double a = 0.0, b = 0.0;
                for (int d = 0; d < D; ++d) {
                    const double x = bf16_to_double(X[(size_t)t * D + d]);
                    a += x * bf16_to_double(Wg[(size_t)f * D + d]);
                    b += x * bf16_to_double(Wu[(size_t)f * D + d]);
                }
                h = silu(a) * b;
            }
            H[(size_t)i * F + f] = h;
        }
    }
}

/*
 * GEMM-K, App. B Eq. 21 (down_proj / o_proj, pruned on in-features):
 *   Y[t, n] = sum_g M[t,g] sum_{k in K_g} A[t,k] W[n,k],  K_g = [gG, (g+1)G)
 *   A : bf16 [T, K], W : bf16 [N, K], mask : uint8 [T, K/G],
 *   Y : double [R, N].  Entries of A in inactive groups never contribute.
 */
void oracle_proj_k(const uint16_t *A, const uint16_t *W, const uint8_t *mask,
                   int T, int K, int N, int G,
                   const int32_t *rows, int n_rows, double *Y)
{
    const int n_groups = K / G;
    const int R = rows ? n_rows : T;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < R; ++i) {
        const int t = rows ? rows[i] : i;
        for (int n = 0; n < N; ++n) {
            double y = 0.0;
            for (int g = 0; g < n_groups; ++g) {
                if (mask[(size_t)t * n_groups + g] == 0)
                    continue;
                for (int k = g * G; k < (g + 1) * G; ++k)
                    y += bf16_to_double(A[(size_t)t * K + k]) *
                         bf16_to_double(W[(size_t)n * K + k]);
            }
            Y[(size_t)i * N + n] = y;
        }
    }
}

/*
 * Whole masked FFN of Eq. 3: Y = ((silu(X Wg^T) (.) X Wu^T) (.)_G M) Wd^T,
 * with the intermediate kept in double (never rounded).
 *   X : bf16 [T, D], Wg, Wu : bf16 [F, D], Wd : bf16 [D, F],
 *   mask : uint8 [T, F/G], Y : double [R, D].
 */
void oracle_ffn(const uint16_t *X, const uint16_t *Wg, const uint16_t *Wu,
                const uint16_t *Wd, const uint8_t *mask,
                int T, int D, int F, int G,
                const int32_t *rows, int n_rows, double *Y,
                double *scratch /* [R, F] */)
{
    const int R = rows ? n_rows : T;
    const int n_groups = F / G;
    oracle_gate_up(X, Wg, Wu, mask, T, D, F, G, rows, n_rows, scratch);
    #pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < R; ++i) {
        const int t = rows ? rows[i] : i;
        for (int n = 0; n < D; ++n) {
            double y = 0.0;
            for (int g = 0; g < n_groups; ++g) {
                if (mask[(size_t)t * n_groups + g] == 0)
                    continue;
                for (int f = g * G; f < (g + 1) * G; ++f)
                    y += scratch[(size_t)i * F + f] *
                         bf16_to_double(Wd[(size_t)n * F + f]);
            }
            Y[(size_t)i * D + n] = y;
        }
    }
}

/*
 * Router of Sec. 3.1 (Eq. 4) and its inference mask (Eq. 5):
 *   z[t, j]    = sum_d X[t,d] W1[j,d]                 (j < r)
 *   R[t, g, c] = sum_j z[t,j] W2[2g+c, j]             (c in {0, 1})
 *   mask[t, g] = 1 if argmax_c R[t,g,c] == 0, i.e. R[t,g,0] >= R[t,g,1]
 *   X : bf16 [T, D];  W1 : bf16 [r, D];  W2 : bf16 [2*n_groups, r]
 *   logits : double [T, 2*n_groups] (R, column 2g + c);  mask : uint8 [T, n_groups]
 *   The decision is taken on the logits rounded to float, the precision the
 *   GPU kernel decides in; logits are returned unrounded.
 */
void oracle_router(const uint16_t *X, const uint16_t *W1, const uint16_t *W2,
                   int T, int D, int r, int n_groups, double *logits, uint8_t *mask)
{
    const int nc = 2 * n_groups;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) {
        double z[1024];
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += bf16_to_double(X[(size_t)t * D + d]) * bf16_to_double(W1[(size_t)j * D + d]);
            z[j] = acc;
        }
        for (int c = 0; c < nc; ++c) {
            double acc = 0.0;
            for (int j = 0; j < r; ++j)
                acc += z[j] * bf16_to_double(W2[(size_t)c * r + j]);
            logits[(size_t)t * nc + c] = acc;
        }
        for (int g = 0; g < n_groups; ++g) {
            const float r0 = (float)logits[(size_t)t * nc + 2 * g];
            const float r1 = (float)logits[(size_t)t * nc + 2 * g + 1];
            mask[(size_t)t * n_groups + g] = (uint8_t)(r0 >= r1 ? 1 : 0);
        }
    }
}

/*
 * Routed decode attention (App. B "Implementation of Attention", decoding;
 * Sec. 3.1 Eq. 2: the attention groups are GQA-aligned, G = (Hq/Hk) d, so
 * group g is KV head g and the Hq/Hk query heads that share it).  One query
 * token per sequence b attends to the lens[b] cached keys (the last position,
 * so no causal cut inside the cache):
 *   s[j]      = (q[b,h,:] . K[b,g,j,:]) / sqrt(d),   g = h / (Hq/Hk)
 *   O[b,h,:]  = mask[b,g] * sum_j softmax(s)[j] V[b,g,j,:]
 * An inactive group, or a sequence with no cached key, gives zeros.
 *   Q : bf16 [B, Hq, d];  K, V : bf16 [B, Hk, L_max, d];  lens : int32 [B]
 *   mask : uint8 [B, Hk];  O : double [B, Hq, d]
 */
void oracle_attn_decode(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                        const int32_t *lens, const uint8_t *mask, int B, int Hq, int Hk,
                        int d, int L_max, double *O)
{
    const int qpk = Hq / Hk;
    const double scale = 1.0 / sqrt((double)d);
    #pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * Hq; ++bh) {
        const int b = bh / Hq, h = bh % Hq, g = h / qpk;
        double *o = O + (size_t)bh * d;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        const int L = lens[b];
        if (mask[(size_t)b * Hk + g] == 0 || L <= 0) continue;
        const uint16_t *q = Q + (size_t)bh * d;
        const uint16_t *Kb = K + ((size_t)b * Hk + g) * (size_t)L_max * d;
        const uint16_t *Vb = V + ((size_t)b * Hk + g) * (size_t)L_max * d;
        double m = -INFINITY;
        for (int j = 0; j < L; ++j) {
            double sj = 0.0;
            for (int e = 0; e < d; ++e)
                sj += bf16_to_double(q[e]) * bf16_to_double(Kb[(size_t)j * d + e]);
            sj *= scale;
            if (sj > m) m = sj;
        }
        double l = 0.0;
        for (int j = 0; j < L; ++j) {
            double sj = 0.0;
            for (int e = 0; e < d; ++e)
                sj += bf16_to_double(q[e]) * bf16_to_double(Kb[(size_t)j * d + e]);
            const double p = exp(sj * scale - m);
            l += p;
            for (int e = 0; e < d; ++e) o[e] += p * bf16_to_double(Vb[(size_t)j * d + e]);
        }
        for (int e = 0; e < d; ++e) o[e] /= l;
    }
}

/*
 * Routed prefill attention (App. B "Implementation of Attention", prefill,
 * Algorithm 4; GQA-aligned groups of Sec. 3.1 Eq. 2: query head h reads KV
 * head g = h / (Hq/Hk), which is also its routing group):
 *   O[b,t,h,:] = mask[b,t,g] * sum_{j <= t (causal) or all j}
 *                softmax_j(Q[b,t,h,:] . K[b,g,j,:] / sqrt(d)) V[b,g,j,:]
 *   Q : bf16 [B, T, Hq, d];  K, V : bf16 [B, Hk, T, d];  mask : uint8 [B, T, Hk]
 *   O : double [B, T, Hq, d]; inactive (token, group) rows are zero.
 */
void oracle_attn_prefill(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                         const uint8_t *mask, int B, int T, int Hq, int Hk, int d,
                         int causal, const int32_t *rows, int n_rows, double *O)
{
    /* rows: optional list of n_rows token positions t to evaluate (all heads,
       every sequence); NULL = every position.  O is [B, R, Hq, d]. */
    const int qpk = Hq / Hk;
    const double scale = 1.0 / sqrt((double)d);
    const int R = rows ? n_rows : T;
    #pragma omp parallel for schedule(dynamic, 1)
    for (long long row = 0; row < (long long)B * R * Hq; ++row) {
        const int h = (int)(row % Hq);
        const int i = (int)((row / Hq) % R);
        const int b = (int)(row / ((long long)Hq * R));
        const int t = rows ? rows[i] : i;
        const int g = h / qpk;
        const size_t qrow = ((size_t)b * T + t) * Hq + h;
        double *o = O + (size_t)row * d;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        if (mask[((size_t)b * T + t) * Hk + g] == 0) continue;
        const uint16_t *q = Q + qrow * d;
        const uint16_t *Kb = K + ((size_t)b * Hk + g) * (size_t)T * d;
        const uint16_t *Vb = V + ((size_t)b * Hk + g) * (size_t)T * d;
        const int n = causal ? t + 1 : T;
        double m = -INFINITY;
        for (int j = 0; j < n; ++j) {
            double sj = 0.0;
            for (int e = 0; e < d; ++e)
                sj += bf16_to_double(q[e]) * bf16_to_double(Kb[(size_t)j * d + e]);
            sj *= scale;
            if (sj > m) m = sj;
        }
        double l = 0.0;
        for (int j = 0; j < n; ++j) {
            double sj = 0.0;
            for (int e = 0; e < d; ++e)
                sj += bf16_to_double(q[e]) * bf16_to_double(Kb[(size_t)j * d + e]);
            const double p = exp(sj * scale - m);
            l += p;
            for (int e = 0; e < d; ++e) o[e] += p * bf16_to_double(Vb[(size_t)j * d + e]);
        }
        for (int e = 0; e < d; ++e) o[e] /= l;
    }
}
