/*
 * Materialised-softmax attention oracle: plain C, binary64 throughout.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker of the
 * CUDA path.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline load it; the product library never links, calls or includes it,
 * and it shares no code with the kernels.
 *
 * What it computes is the plain definition that the streaming kernels reach
 * up to rounding order:
 *
 *   StreamingAttentionSM86.alpha (lsalpha source view), module header of the
 *   forward pass: causal attention softmax(Q K^T scale) V of one head, the
 *   log-sum-exp kept per row in base 2 (L = m + log2 l, which is
 *   (max + ln sum) / ln 2 of the natural-unit scores).
 *
 *   Same file, header of the backward pass: P recomputed from L,
 *   dP = dO V^T, D = rowsum(dO * O), dS = P * (dP - D), dQ = s dS K,
 *   dK = s dS^T Q, dV = P^T dO, s the natural score scale.
 *
 *   Same file, "the program" section: query head h reads K/V head
 *   h / (heads / kv_heads) (grouped-query attention).
 *
 *   Gist "snippet.py" (self_attn_fwd): a per-sequence length masks query
 *   rows and keys at or beyond it; rows with no valid key output zero.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes): L of a fully masked row is -inf; D and dQ of such a row are
 * zero; dK and dV are per K/V head, summed over the query heads of its group;
 * the diagonal is kept (a key equal to the query is valid).
 *
 * Layouts are the boundary's: q, dout [B][H][T][d]; k [B][Hkv][T][d];
 * vt [B][Hkv][d][T]; o [B][T][H*d]; lse, delta [B][H][T];
 * dq [B][H][T][d]; dk [B][Hkv][T][d]; dvt [B][Hkv][d][T].
 * Inputs are binary64 arrays (the caller widens binary16 exactly).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t batch, seq, heads, kv_heads, head_dim, causal;
    double scale;
} oracle_shape;

static const double LN2 = 0.69314718055994530942;

static int shape_ok(const oracle_shape* s) {
    if (!s) return 0;
    if (s->batch < 1 || s->seq < 1 || s->heads < 1 || s->kv_heads < 1 ||
        s->head_dim < 1)
        return 0;
    if (s->heads % s->kv_heads != 0) return 0;
    return 1;
}

static int seq_len(const oracle_shape* s, const int32_t* lens, int b) {
    if (!lens) return s->seq;
    int n = lens[b];
    if (n < 0) n = 0;
    if (n > s->seq) n = s->seq;
    return n;
}

/* valid(i, j): key j takes part in query row i's softmax. */
static int valid(const oracle_shape* s, int len, int i, int j) {
    if (i >= len || j >= len) return 0;
    if (s->causal && j > i) return 0;
    return 1;
}

static double dot(const double* a, const double* b, int n) {
    double acc = 0.0;
    for (int t = 0; t < n; ++t) acc += a[t] * b[t];
    return acc;
}

/* Pointers to the planes of one (batch, head). */
static const double* q_row(const oracle_shape* s, const double* q, int b, int h, int i) {
    return q + (((size_t)b * s->heads + h) * s->seq + i) * s->head_dim;
}
static const double* k_row(const oracle_shape* s, const double* k, int b, int kv, int j) {
    return k + (((size_t)b * s->kv_heads + kv) * s->seq + j) * s->head_dim;
}
static const double* vt_plane(const oracle_shape* s, const double* vt, int b, int kv) {
    return vt + ((size_t)b * s->kv_heads + kv) * (size_t)s->head_dim * s->seq;
}

/*
 * One query row of the materialised softmax.  Fills p[0..T) with the
 * probabilities P_ij (zero where invalid), o_row[0..d) with sum_j P_ij v_j,
 * and returns the row's max score M and normaliser Z = sum exp(s - M)
 * (Z = 0 and M = -inf when no key is valid).
 */
static void row_softmax(const oracle_shape* s, int len, const double* q, const double* k,
                        const double* vt, int b, int h, int i, double* p, double* o_row,
                        double* M_out, double* Z_out) {
    const int T = s->seq, d = s->head_dim;
    const int kv = h / (s->heads / s->kv_heads);
    const double* qi = q_row(s, q, b, h, i);
    const double* vp = vt_plane(s, vt, b, kv);
    double M = -INFINITY;
    for (int j = 0; j < T; ++j) {
        if (valid(s, len, i, j)) {
            p[j] = s->scale * dot(qi, k_row(s, k, b, kv, j), d);
            if (p[j] > M) M = p[j];
        } else {
            p[j] = 0.0;
        }
    }
    for (int c = 0; c < d; ++c) o_row[c] = 0.0;
    if (M == -INFINITY) {
        *M_out = -INFINITY;
        *Z_out = 0.0;
        return;
    }
    double Z = 0.0;
    for (int j = 0; j < T; ++j) {
        if (valid(s, len, i, j)) {
            p[j] = exp(p[j] - M);
            Z += p[j];
        }
    }
    for (int j = 0; j < T; ++j) p[j] /= Z; /* invalid entries stay 0 */
    for (int c = 0; c < d; ++c) {
        const double* vrow = vp + (size_t)c * T;
        double acc = 0.0;
        for (int j = 0; j < T; ++j) acc += p[j] * vrow[j];
        o_row[c] = acc;
    }
    *M_out = M;
    *Z_out = Z;
}

static double base2_lse(double M, double Z) {
    if (Z == 0.0) return -INFINITY;
    return (M + log(Z)) / LN2;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Forward pass: O [B][T][H*d] and base-2 log-sum-exp L [B][H][T]. */
int oracle_forward(const oracle_shape* s, const int32_t* lens, const double* q,
                   const double* k, const double* vt, double* o, double* lse) {
    if (!shape_ok(s) || !q || !k || !vt || !o || !lse) return -1;
    const int B = s->batch, H = s->heads, T = s->seq, d = s->head_dim;
    const long total = (long)B * H * T;
    int err = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)T);
        double* orow = (double*)malloc(sizeof(double) * (size_t)d);
        if (!p || !orow) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (long r = 0; r < total; ++r) {
                const int i = (int)(r % T);
                const int h = (int)((r / T) % H);
                const int b = (int)(r / ((long)T * H));
                const int len = seq_len(s, lens, b);
                double M, Z;
                row_softmax(s, len, q, k, vt, b, h, i, p, orow, &M, &Z);
                double* dst = o + (((size_t)b * T + i) * H + h) * d;
                memcpy(dst, orow, sizeof(double) * (size_t)d);
                lse[((size_t)b * H + h) * T + i] = base2_lse(M, Z);
            }
        }
        free(p);
        free(orow);
    }
    return err ? -2 : 0;
}

/*
 * Row-local part of the backward pass for one query row i of head h:
 * O_i, L_i, D_i = dO_i . O_i and dQ_i = s sum_j P_ij (dP_ij - D_i) k_j.
 * Returns M and Z of the row through the pointers (for the key-side sums).
 */
static void row_backward(const oracle_shape* s, int len, const double* q, const double* k,
                         const double* vt, const double* dout, int b, int h, int i,
                         double* p, double* o_row, double* dq_row, double* lse_out,
                         double* delta_out, double* M_out, double* Z_out) {
    const int T = s->seq, d = s->head_dim;
    const int kv = h / (s->heads / s->kv_heads);
    double M, Z;
    row_softmax(s, len, q, k, vt, b, h, i, p, o_row, &M, &Z);
    const double* doi = q_row(s, dout, b, h, i);
    const double* vp = vt_plane(s, vt, b, kv);
    for (int c = 0; c < d; ++c) dq_row[c] = 0.0;
    double D = 0.0;
    if (Z > 0.0) {
        D = dot(doi, o_row, d);
        for (int j = 0; j < T; ++j) {
            if (!valid(s, len, i, j)) continue;
            double dP = 0.0;
            for (int c = 0; c < d; ++c) dP += doi[c] * vp[(size_t)c * T + j];
            const double dS = p[j] * (dP - D);
            const double* kj = k_row(s, k, b, kv, j);
            for (int c = 0; c < d; ++c) dq_row[c] += dS * kj[c];
        }
        for (int c = 0; c < d; ++c) dq_row[c] *= s->scale;
    }
    *lse_out = base2_lse(M, Z);
    *delta_out = D;
    *M_out = M;
    *Z_out = Z;
}

/*
 * Key-side sums for key j of K/V head kv, given every row's M, Z and D of the
 * group's query heads (arrays [G][T]):
 *   dK_j = s sum_{h in group} sum_i dS_ij q_i,   dV_j = sum_h sum_i P_ij dO_i,
 * with P_ij = exp(s_ij - M_i) / Z_i the same materialised probability.
 */
static void key_sums(const oracle_shape* s, int len, const double* q, const double* k,
                     const double* vt, const double* dout, int b, int kv, int j,
                     const double* Mg, const double* Zg, const double* Dg, double* dk_row,
                     double* dv_row) {
    const int T = s->seq, d = s->head_dim;
    const int G = s->heads / s->kv_heads;
    const double* kj = k_row(s, k, b, kv, j);
    const double* vp = vt_plane(s, vt, b, kv);
    double* vjp = (double*)malloc(sizeof(double) * (size_t)d);
    if (!vjp) return;
    for (int c = 0; c < d; ++c) vjp[c] = vp[(size_t)c * T + j];
    for (int c = 0; c < d; ++c) {
        dk_row[c] = 0.0;
        dv_row[c] = 0.0;
    }
    for (int g = 0; g < G; ++g) {
        const int h = kv * G + g;
        for (int i = 0; i < T; ++i) {
            if (!valid(s, len, i, j)) continue;
            const double Z = Zg[(size_t)g * T + i];
            if (Z == 0.0) continue;
            const double* qi = q_row(s, q, b, h, i);
            const double* doi = q_row(s, dout, b, h, i);
            const double sij = s->scale * dot(qi, kj, d);
            const double P = exp(sij - Mg[(size_t)g * T + i]) / Z;
            const double dP = dot(doi, vjp, d);
            const double dS = P * (dP - Dg[(size_t)g * T + i]);
            for (int c = 0; c < d; ++c) {
                dk_row[c] += dS * qi[c];
                dv_row[c] += P * doi[c];
            }
        }
    }
    for (int c = 0; c < d; ++c) dk_row[c] *= s->scale;
    free(vjp);
}

/*
 * Full forward and backward pass.  Outputs: o, lse, delta (D), dq, dk, dvt.
 * Pass 1 walks query rows (row-local terms), pass 2 walks keys (the sums over
 * query rows that dK and dV need), each parallel over independent units.
 */
int oracle_backward(const oracle_shape* s, const int32_t* lens, const double* q,
                    const double* k, const double* vt, const double* dout, double* o,
                    double* lse, double* delta, double* dq, double* dk, double* dvt) {
    if (!shape_ok(s) || !q || !k || !vt || !dout || !o || !lse || !delta || !dq || !dk ||
        !dvt)
        return -1;
    const int B = s->batch, H = s->heads, Hkv = s->kv_heads, T = s->seq, d = s->head_dim;
    const int G = H / Hkv;
    const size_t nrows = (size_t)B * H * T;
    double* Ms = (double*)malloc(sizeof(double) * nrows);
    double* Zs = (double*)malloc(sizeof(double) * nrows);
    if (!Ms || !Zs) {
        free(Ms);
        free(Zs);
        return -2;
    }
    int err = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)T);
        double* orow = (double*)malloc(sizeof(double) * (size_t)d);
        if (!p || !orow) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (long r = 0; r < (long)nrows; ++r) {
                const int i = (int)(r % T);
                const int h = (int)((r / T) % H);
                const int b = (int)(r / ((long)T * H));
                const int len = seq_len(s, lens, b);
                const size_t lr = ((size_t)b * H + h) * T + i;
                row_backward(s, len, q, k, vt, dout, b, h, i, p,
                             orow, dq + lr * d, &lse[lr], &delta[lr], &Ms[lr], &Zs[lr]);
                memcpy(o + (((size_t)b * T + i) * H + h) * d, orow, sizeof(double) * (size_t)d);
            }
        }
        free(p);
        free(orow);
    }
    if (!err) {
        const long nkeys = (long)B * Hkv * T;
#pragma omp parallel
        {
            double* dkr = (double*)malloc(sizeof(double) * (size_t)d);
            double* dvr = (double*)malloc(sizeof(double) * (size_t)d);
            if (!dkr || !dvr) {
#pragma omp atomic write
                err = 1;
            } else {
#pragma omp for schedule(dynamic, 8)
                for (long r = 0; r < nkeys; ++r) {
                    const int j = (int)(r % T);
                    const int kv = (int)((r / T) % Hkv);
                    const int b = (int)(r / ((long)T * Hkv));
                    const int len = seq_len(s, lens, b);
                    const size_t g0 = ((size_t)b * H + (size_t)kv * G) * T;
                    key_sums(s, len, q, k, vt, dout, b, kv, j, Ms + g0, Zs + g0, delta + g0,
                             dkr, dvr);
                    double* dkdst = dk + (((size_t)b * Hkv + kv) * T + j) * d;
                    double* dvplane = dvt + ((size_t)b * Hkv + kv) * (size_t)d * T;
                    for (int c = 0; c < d; ++c) {
                        dkdst[c] = dkr[c];
                        dvplane[(size_t)c * T + j] = dvr[c];
                    }
                }
            }
            free(dkr);
            free(dvr);
        }
    }
    free(Ms);
    free(Zs);
    return err ? -2 : 0;
}

/*
 * Sampled query rows of head h in batch b: o_rows [n][d], lse_rows [n],
 * delta_rows [n], dq_rows [n][d].  Each row costs O(T d): every quantity here
 * depends on its own row only.
 */
int oracle_query_rows(const oracle_shape* s, const int32_t* lens, const double* q,
                      const double* k, const double* vt, const double* dout, int b, int h,
                      const int32_t* rows, int n, double* o_rows, double* lse_rows,
                      double* delta_rows, double* dq_rows) {
    if (!shape_ok(s) || !rows || n < 0 || b < 0 || b >= s->batch || h < 0 ||
        h >= s->heads)
        return -1;
    for (int t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= s->seq) return -1;
    const int T = s->seq, d = s->head_dim;
    const int len = seq_len(s, lens, b);
    int err = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)T);
        if (!p) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int t = 0; t < n; ++t) {
                double M, Z;
                row_backward(s, len, q, k, vt, dout, b, h, rows[t], p, o_rows + (size_t)t * d,
                             dq_rows + (size_t)t * d, &lse_rows[t], &delta_rows[t], &M, &Z);
            }
        }
        free(p);
    }
    return err ? -2 : 0;
}

/*
 * Sampled keys of K/V head kv in batch b: dk_rows [n][d], dv_rows [n][d].
 * The rows' M, Z and D of every query head in the group are computed first
 * (row-local, O(T^2 d) per head), then each sampled key's sums (O(G T d)).
 */
int oracle_key_rows(const oracle_shape* s, const int32_t* lens, const double* q,
                    const double* k, const double* vt, const double* dout, int b, int kv,
                    const int32_t* keys, int n, double* dk_rows, double* dv_rows) {
    if (!shape_ok(s) || !keys || n < 0 || b < 0 || b >= s->batch || kv < 0 ||
        kv >= s->kv_heads)
        return -1;
    for (int t = 0; t < n; ++t)
        if (keys[t] < 0 || keys[t] >= s->seq) return -1;
    const int T = s->seq, d = s->head_dim;
    const int G = s->heads / s->kv_heads;
    const int len = seq_len(s, lens, b);
    double* Mg = (double*)malloc(sizeof(double) * (size_t)G * T);
    double* Zg = (double*)malloc(sizeof(double) * (size_t)G * T);
    double* Dg = (double*)malloc(sizeof(double) * (size_t)G * T);
    if (!Mg || !Zg || !Dg) {
        free(Mg);
        free(Zg);
        free(Dg);
        return -2;
    }
    int err = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)T);
        double* orow = (double*)malloc(sizeof(double) * (size_t)d);
        double* dqr = (double*)malloc(sizeof(double) * (size_t)d);
        if (!p || !orow || !dqr) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (long r = 0; r < (long)G * T; ++r) {
                const int i = (int)(r % T);
                const int g = (int)(r / T);
                double L;
                row_backward(s, len, q, k, vt, dout, b, kv * G + g, i, p, orow, dqr, &L,
                             &Dg[r], &Mg[r], &Zg[r]);
            }
        }
        free(p);
        free(orow);
        free(dqr);
    }
    if (!err) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int t = 0; t < n; ++t)
            key_sums(s, len, q, k, vt, dout, b, kv, keys[t], Mg, Zg, Dg,
                     dk_rows + (size_t)t * d, dv_rows + (size_t)t * d);
    }
    free(Mg);
    free(Zg);
    free(Dg);
    return err ? -2 : 0;
}

/* The probability row P_i. of head h (for the invariant checks). */
int oracle_probs_row(const oracle_shape* s, const int32_t* lens, const double* q,
                     const double* k, const double* vt, int b, int h, int i, double* p_row) {
    if (!shape_ok(s) || !p_row || b < 0 || b >= s->batch || h < 0 || h >= s->heads || i < 0 ||
        i >= s->seq)
        return -1;
    double* orow = (double*)malloc(sizeof(double) * (size_t)s->head_dim);
    if (!orow) return -2;
    double M, Z;
    row_softmax(s, seq_len(s, lens, b), q, k, vt, b, h, i, p_row, orow, &M, &Z);
    free(orow);
    return 0;
}
