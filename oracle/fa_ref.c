/*
 * fa_ref.c -- plain, slow fp64 CPU oracle for attention forward and the
 * FlashAttention-2 backward (preprocess D, then dQ / dK / dV).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only tests/, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (all arithmetic in double precision, inputs already
 * upcast exactly by the caller):
 *
 *   layout (boostr flash_bwd.rs, shape checks in flash_attention_bwd_impl;
 *   rustytorch backward.rs, doc comment of flash_attention_backward):
 *     Q, O, dO, dQ : [B, H,    S_q, d]   row-major, contiguous
 *     K, V, dK, dV : [B, H_kv, S_k, d]
 *     LSE, D       : [B, H,    S_q]
 *   query head h reads key/value head hk = h / (H / H_kv)  (consecutive
 *   grouping; the pages only fix that dK, dV have H_kv heads).
 *
 *   mask(i, j): query i sits at key position p_i = i + (S_k - S_q)
 *   (bottom-right alignment; p_i = i when S_q == S_k).
 *     non-causal -> every j < S_k;  causal -> j <= p_i.
 *     sliding window w > 0 (boostr autograd_attention.rs, window_size in
 *     FlashAttentionConfig; 0 means no window): additionally p_i - j < w,
 *     and when not causal also j - p_i < w.  A causal query therefore sees
 *     at most its w most recent keys, itself included; a non-causal one
 *     the keys less than w positions away on either side.  The pages name
 *     the parameter but not its exact band; this is the plain reading.
 *
 *   forward:   S_ij   = scale * <Q_i, K_j>
 *              LSE_i  = log sum_{j allowed} exp(S_ij)   (natural log,
 *                       -inf for a row with no allowed key)
 *              O_i    = sum_j exp(S_ij - LSE_i) V_j      (0 for such a row)
 *
 *   backward (boostr flash_bwd.rs doc comment, "Two-step process"):
 *     step 1   D_i    = sum_c dO_ic * O_ic                 (preprocess)
 *     step 2   P_ij   = allowed ? exp(S_ij - LSE_i) : 0
 *              dP_ij  = <dO_i, V_j>
 *              dS_ij  = P_ij * (dP_ij - D_i)
 *              dQ_i   = scale * sum_j dS_ij K_j
 *              dK_j  += scale * sum_i dS_ij Q_i   (summed over the group)
 *              dV_j  += sum_i P_ij dO_i           (summed over the group)
 *   These are the chain rule of O = softmax(scale * Q K^T) V with the saved
 *   LSE standing in for the softmax normaliser; D_i equals sum_j P_ij dP_ij
 *   when O is the exact forward output.
 *
 * No blocking, fusion or reordering beyond the definition: each query row is
 * visited once, its full score row is formed, and the sums above are taken
 * in index order.  OpenMP only splits independent (batch, kv head) pairs or
 * independent sampled rows across threads.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX4(b, h, i, c, NH, S, d) ((((size_t)(b) * (NH) + (h)) * (S) + (i)) * (size_t)(d) + (c))
#define IDX3(b, h, i, NH, S) ((((size_t)(b) * (NH) + (h)) * (S)) + (i))

/* Is key j visible to query i?  Bottom-right alignment; window 0 = none. */
static int allowed(long i, long j, int S_q, int S_k, int causal, int window) {
    if (j < 0 || j >= S_k) return 0;
    const long p = i + (long)(S_k - S_q);
    if (window > 0 && (p - j >= window || (!causal && j - p >= window))) return 0;
    if (!causal) return 1;
    return j <= p;
}

static double dot(const double* a, const double* b, int d) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

int fa_ref_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward: O and LSE from Q, K, V (definition above). */
void fa_ref_fwd(const double* Q, const double* K, const double* V, double* O, double* LSE,
                int B, int H, int H_kv, int S_q, int S_k, int d, double scale, int causal,
                int window) {
    const int g = H / H_kv;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const int hk = h / g;
            double* s = (double*)malloc(sizeof(double) * (size_t)(S_k > 0 ? S_k : 1));
            for (int i = 0; i < S_q; ++i) {
                const double* q = Q + IDX4(b, h, i, 0, H, S_q, d);
                double m = -INFINITY;
                for (int j = 0; j < S_k; ++j) {
                    if (!allowed(i, j, S_q, S_k, causal, window)) { s[j] = -INFINITY; continue; }
                    s[j] = scale * dot(q, K + IDX4(b, hk, j, 0, H_kv, S_k, d), d);
                    if (s[j] > m) m = s[j];
                }
                double* o = O + IDX4(b, h, i, 0, H, S_q, d);
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                if (m == -INFINITY) { LSE[IDX3(b, h, i, H, S_q)] = -INFINITY; continue; }
                double z = 0.0;
                for (int j = 0; j < S_k; ++j)
                    if (s[j] != -INFINITY) z += exp(s[j] - m);
                const double lse = m + log(z);
                LSE[IDX3(b, h, i, H, S_q)] = lse;
                for (int j = 0; j < S_k; ++j) {
                    if (s[j] == -INFINITY) continue;
                    const double p = exp(s[j] - lse);
                    const double* v = V + IDX4(b, hk, j, 0, H_kv, S_k, d);
                    for (int c = 0; c < d; ++c) o[c] += p * v[c];
                }
            }
            free(s);
        }
}

/* Step 1 of the backward (boostr flash_bwd.rs, "Step 1: Preprocessing"):
 * D_r = sum_c dO_rc * O_rc for each of the R = B*H*S_q query rows. */
void fa_ref_preprocess(const double* dO, const double* O, double* D, long R, int d) {
#pragma omp parallel for schedule(static)
    for (long r = 0; r < R; ++r) D[r] = dot(dO + (size_t)r * d, O + (size_t)r * d, d);
}

/* Full backward: dQ, dK, dV (definition above).  D is optional output. */
void fa_ref_bwd(const double* dO, const double* Q, const double* K, const double* V,
                const double* O, const double* LSE, double* dQ, double* dK, double* dV,
                double* D_out, int B, int H, int H_kv, int S_q, int S_k, int d, double scale,
                int causal, int window) {
    const int g = H / H_kv;
    memset(dQ, 0, sizeof(double) * (size_t)B * H * S_q * d);
    memset(dK, 0, sizeof(double) * (size_t)B * H_kv * S_k * d);
    memset(dV, 0, sizeof(double) * (size_t)B * H_kv * S_k * d);
    /* one thread owns one (b, hk): its dK and dV rows are written by nobody else */
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int hk = 0; hk < H_kv; ++hk) {
            double* p = (double*)malloc(sizeof(double) * (size_t)(S_k > 0 ? S_k : 1));
            double* ds = (double*)malloc(sizeof(double) * (size_t)(S_k > 0 ? S_k : 1));
            for (int h = hk * g; h < (hk + 1) * g; ++h)
                for (int i = 0; i < S_q; ++i) {
                    const double* q = Q + IDX4(b, h, i, 0, H, S_q, d);
                    const double* o = O + IDX4(b, h, i, 0, H, S_q, d);
                    const double* g_o = dO + IDX4(b, h, i, 0, H, S_q, d);
                    const double lse = LSE[IDX3(b, h, i, H, S_q)];
                    const double Di = dot(g_o, o, d);
                    if (D_out) D_out[IDX3(b, h, i, H, S_q)] = Di;
                    for (int j = 0; j < S_k; ++j) {
                        if (!allowed(i, j, S_q, S_k, causal, window)) { p[j] = 0.0; ds[j] = 0.0; continue; }
                        const double sij = scale * dot(q, K + IDX4(b, hk, j, 0, H_kv, S_k, d), d);
                        p[j] = exp(sij - lse);
                        const double dpij = dot(g_o, V + IDX4(b, hk, j, 0, H_kv, S_k, d), d);
                        ds[j] = p[j] * (dpij - Di);
                    }
                    double* dq = dQ + IDX4(b, h, i, 0, H, S_q, d);
                    for (int j = 0; j < S_k; ++j) {
                        if (p[j] == 0.0 && ds[j] == 0.0) continue;
                        const double* k = K + IDX4(b, hk, j, 0, H_kv, S_k, d);
                        double* dk = dK + IDX4(b, hk, j, 0, H_kv, S_k, d);
                        double* dv = dV + IDX4(b, hk, j, 0, H_kv, S_k, d);
                        for (int c = 0; c < d; ++c) {
                            dq[c] += scale * ds[j] * k[c];
                            dk[c] += scale * ds[j] * q[c];
                            dv[c] += p[j] * g_o[c];
                        }
                    }
                }
            free(p);
            free(ds);
        }
}

/* Sampled dQ rows: rows[r] is a flat query-row index (b*H + h)*S_q + i.
 * Same definition as fa_ref_bwd, restricted to the requested rows. */
void fa_ref_dq_rows(const double* dO, const double* Q, const double* K, const double* V,
                    const double* O, const double* LSE, const long* rows, int nrows,
                    double* dQ_rows, int B, int H, int H_kv, int S_q, int S_k, int d,
                    double scale, int causal, int window) {
    (void)B;
    const int g = H / H_kv;
#pragma omp parallel for schedule(dynamic)
    for (int r = 0; r < nrows; ++r) {
        const long flat = rows[r];
        const int i = (int)(flat % S_q);
        const int h = (int)((flat / S_q) % H);
        const int b = (int)(flat / ((long)S_q * H));
        const int hk = h / g;
        const double* q = Q + IDX4(b, h, i, 0, H, S_q, d);
        const double* g_o = dO + IDX4(b, h, i, 0, H, S_q, d);
        const double lse = LSE[IDX3(b, h, i, H, S_q)];
        const double Di = dot(g_o, O + IDX4(b, h, i, 0, H, S_q, d), d);
        double* dq = dQ_rows + (size_t)r * d;
        for (int c = 0; c < d; ++c) dq[c] = 0.0;
        for (int j = 0; j < S_k; ++j) {
            if (!allowed(i, j, S_q, S_k, causal, window)) continue;
            const double* k = K + IDX4(b, hk, j, 0, H_kv, S_k, d);
            const double pij = exp(scale * dot(q, k, d) - lse);
            const double dsij = pij * (dot(g_o, V + IDX4(b, hk, j, 0, H_kv, S_k, d), d) - Di);
            for (int c = 0; c < d; ++c) dq[c] += scale * dsij * k[c];
        }
    }
}

/* Sampled dK / dV rows: rows[r] is a flat key-row index (b*H_kv + hk)*S_k + j.
 * Each requested row sums over every query row of every head in its group. */
void fa_ref_dkv_rows(const double* dO, const double* Q, const double* K, const double* V,
                     const double* O, const double* LSE, const long* rows, int nrows,
                     double* dK_rows, double* dV_rows, int B, int H, int H_kv, int S_q,
                     int S_k, int d, double scale, int causal, int window) {
    (void)B;
    const int g = H / H_kv;
#pragma omp parallel for schedule(dynamic)
    for (int r = 0; r < nrows; ++r) {
        const long flat = rows[r];
        const int j = (int)(flat % S_k);
        const int hk = (int)((flat / S_k) % H_kv);
        const int b = (int)(flat / ((long)S_k * H_kv));
        const double* k = K + IDX4(b, hk, j, 0, H_kv, S_k, d);
        const double* v = V + IDX4(b, hk, j, 0, H_kv, S_k, d);
        double* dk = dK_rows + (size_t)r * d;
        double* dv = dV_rows + (size_t)r * d;
        for (int c = 0; c < d; ++c) { dk[c] = 0.0; dv[c] = 0.0; }
        for (int h = hk * g; h < (hk + 1) * g; ++h)
            for (int i = 0; i < S_q; ++i) {
                if (!allowed(i, j, S_q, S_k, causal, window)) continue;
                const double* q = Q + IDX4(b, h, i, 0, H, S_q, d);
                const double* g_o = dO + IDX4(b, h, i, 0, H, S_q, d);
                const double Di = dot(g_o, O + IDX4(b, h, i, 0, H, S_q, d), d);
                const double pij = exp(scale * dot(q, k, d) - LSE[IDX3(b, h, i, H, S_q)]);
                const double dsij = pij * (dot(g_o, v, d) - Di);
                for (int c = 0; c < d; ++c) {
                    dk[c] += scale * dsij * q[c];
                    dv[c] += pij * g_o[c];
                }
            }
    }
}
