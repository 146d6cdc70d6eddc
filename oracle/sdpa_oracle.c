/*
 * sdpa_oracle.c -- float64 CPU oracle for scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this file's library. The product
 * path (the CUDA library) never calls it, and the two share no code.
 *
 * What it computes is the plain definition of softmax attention, the
 * "unfused" attention that materialises the score matrix (TransformerEngine
 * PR #3527, section "Performance"), evaluated in float64 with no blocking,
 * no online softmax and no reordering beyond the definition:
 *
 *   s_ij  = scale * sum_d q_id k_jd
 *   allowed(i,j) by mask type and window (below); masked s_ij = -inf
 *   LSE_i = ln sum_{allowed j} exp(s_ij)      (natural log; PR #3705,
 *                                              "Execution and supported scope":
 *                                              Stats are FP32 natural logs)
 *   p_ij  = exp(s_ij - LSE_i)
 *   o_i   = sum_j p_ij v_j
 *
 * Backward (the textbook derivative; the pages print no formula):
 *
 *   delta_i = sum_d dO_id o_id
 *   dP_ij   = sum_d dO_id v_jd
 *   dS_ij   = p_ij (dP_ij - delta_i)
 *   dQ_i    = scale * sum_j dS_ij k_j
 *   dK_j    = scale * sum_{heads h of kv head g} sum_i dS_ij q_i
 *   dV_j    = sum_{heads h of kv head g} sum_i p_ij dO_i
 *
 * Masks (PR #3527, "Approach" and "Scope": no_mask / causal /
 * causal_bottom_right; PR #3693 passes a (left, right) window pair):
 *   top-left causal:      the diagonal of row i is column i
 *   bottom-right causal:  the diagonal of row i is column i + Lk - Lq
 *   no mask:              the diagonal (for a window only) is column i
 *   allowed iff 0 <= j < Lk, j <= diag + right, j >= diag - left, where a
 *   causal mask sets right = 0 and a negative bound means unbounded.
 * A row with no allowed key has o = 0, LSE = -inf and contributes nothing
 * to any gradient.
 *
 * Grouped-query attention: q head h reads kv head h / (Hq / Hkv).
 *
 * Head dims: q and k rows have head_dim entries, v and o rows head_dim_v
 * (0 = head_dim). The definition above never mixes the two widths: s_ij
 * sums over the q/k width and o_i is a combination of v rows. The pages
 * list the (192, 128) pair among the forward engine's native shapes
 * (TransformerEngine PR #3527, "Scope"), and the backward there requires
 * d_qk == d_v, so the backward entry points here reject unequal widths.
 *
 * Layouts (PR #3527 "Scope": bshd, sbhd; PR #3705: compact thd with
 * zero-based cumulative sequence lengths):
 *   BSHD  x[b][s][h][d]       token row = b*S + s
 *   SBHD  x[s][b][h][d]       token row = s*B + b
 *   THD   x[t][h][d]          token row = cu_seqlens[b] + s
 * LSE is token-major: lse[token_row][h] (PR #3705: "packed token-major
 * FP32"; PR #3693 lists Stats [tq, h, 1] for thd).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_BSHD 0
#define OR_SBHD 1
#define OR_THD 2

#define OR_MASK_NONE 0
#define OR_MASK_CAUSAL_TOP_LEFT 1
#define OR_MASK_CAUSAL_BOTTOM_RIGHT 2

typedef struct {
    int layout;
    int mask_type;
    int batch;
    int seqlen_q;   /* BSHD/SBHD: the sequence length; THD: unused */
    int seqlen_kv;
    int num_heads_q;
    int num_heads_kv;
    int head_dim;
    int window_left;  /* < 0: unbounded */
    int window_right; /* < 0: unbounded; forced to 0 by a causal mask */
    double scale;
    int head_dim_v;   /* width of v and o rows; 0 = head_dim */
} oracle_problem;

/* ---- geometry --------------------------------------------------------- */

static int seq_len(const oracle_problem* p, const int32_t* cu, int b, int is_q) {
    if (p->layout == OR_THD) return cu[b + 1] - cu[b];
    return is_q ? p->seqlen_q : p->seqlen_kv;
}

/* token row of position s of sequence b (the leading index of the layout) */
static int64_t token_row(const oracle_problem* p, const int32_t* cu, int b, int s, int is_q) {
    switch (p->layout) {
        case OR_BSHD: return (int64_t)b * (is_q ? p->seqlen_q : p->seqlen_kv) + s;
        case OR_SBHD: return (int64_t)s * p->batch + b;
        default: return (int64_t)cu[b] + s;
    }
}

static const double* qrow(const oracle_problem* p, const double* x, const int32_t* cu, int b, int s, int h) {
    return x + (token_row(p, cu, b, s, 1) * p->num_heads_q + h) * p->head_dim;
}
static const double* kvrow(const oracle_problem* p, const double* x, const int32_t* cu, int b, int s, int g) {
    return x + (token_row(p, cu, b, s, 0) * p->num_heads_kv + g) * p->head_dim;
}

static int dv_of(const oracle_problem* p) { return p->head_dim_v > 0 ? p->head_dim_v : p->head_dim; }

/* row s of kv head g of v (rows of dv_of(p) entries) */
static const double* vrow(const oracle_problem* p, const double* x, const int32_t* cu, int b, int s, int g) {
    return x + (token_row(p, cu, b, s, 0) * p->num_heads_kv + g) * dv_of(p);
}

static int kv_head_of(const oracle_problem* p, int h) {
    return h / (p->num_heads_q / p->num_heads_kv);
}

static int allowed(const oracle_problem* p, int i, int j, int lq, int lk) {
    if (j < 0 || j >= lk) return 0;
    long diag = i;
    long right = p->window_right;
    if (p->mask_type == OR_MASK_CAUSAL_BOTTOM_RIGHT) diag = (long)i + lk - lq;
    if (p->mask_type != OR_MASK_NONE) right = 0;
    if (right >= 0 && j > diag + right) return 0;
    if (p->window_left >= 0 && j < diag - p->window_left) return 0;
    return 1;
}

static double dot(const double* a, const double* b, int n) {
    double s = 0.0;
    for (int d = 0; d < n; ++d) s += a[d] * b[d];
    return s;
}

/* Scores of one query row against all keys of its sequence; returns LSE
 * (natural log) and fills s[j] (-inf where masked). */
static double row_scores(const oracle_problem* p, const double* q, const double* k, const int32_t* cu_q,
                         const int32_t* cu_kv, int b, int h, int i, double* s) {
    int lq = seq_len(p, cu_q, b, 1), lk = seq_len(p, cu_kv, b, 0);
    int g = kv_head_of(p, h);
    const double* qi = qrow(p, q, cu_q, b, i, h);
    double m = -INFINITY;
    for (int j = 0; j < lk; ++j) {
        if (allowed(p, i, j, lq, lk)) {
            s[j] = p->scale * dot(qi, kvrow(p, k, cu_kv, b, j, g), p->head_dim);
            if (s[j] > m) m = s[j];
        } else {
            s[j] = -INFINITY;
        }
    }
    if (m == -INFINITY) return -INFINITY;
    double sum = 0.0;
    for (int j = 0; j < lk; ++j)
        if (s[j] != -INFINITY) sum += exp(s[j] - m);
    return m + log(sum);
}

/* o_i and LSE_i for one (b, h, i). */
static void row_forward(const oracle_problem* p, const double* q, const double* k, const double* v,
                        const int32_t* cu_q, const int32_t* cu_kv, int b, int h, int i, double* s,
                        double* o_out, double* lse_out) {
    int lk = seq_len(p, cu_kv, b, 0);
    int g = kv_head_of(p, h);
    int dv = dv_of(p);
    double lse = row_scores(p, q, k, cu_q, cu_kv, b, h, i, s);
    for (int d = 0; d < dv; ++d) o_out[d] = 0.0;
    if (lse != -INFINITY) {
        for (int j = 0; j < lk; ++j) {
            if (s[j] == -INFINITY) continue;
            double pij = exp(s[j] - lse);
            const double* vj = vrow(p, v, cu_kv, b, j, g);
            for (int d = 0; d < dv; ++d) o_out[d] += pij * vj[d];
        }
    }
    *lse_out = lse;
}

static int max_len(const oracle_problem* p, const int32_t* cu, int is_q) {
    if (p->layout != OR_THD) return is_q ? p->seqlen_q : p->seqlen_kv;
    int m = 0;
    for (int b = 0; b < p->batch; ++b) {
        int l = cu[b + 1] - cu[b];
        if (l > m) m = l;
    }
    return m;
}

static int64_t rows_total(const oracle_problem* p, const int32_t* cu, int is_q) {
    if (p->layout == OR_THD) return cu[p->batch];
    return (int64_t)p->batch * (is_q ? p->seqlen_q : p->seqlen_kv);
}

static int valid(const oracle_problem* p) {
    if (p->num_heads_kv <= 0 || p->num_heads_q <= 0 || p->head_dim <= 0 || p->batch < 0) return 0;
    if (p->head_dim_v < 0 || p->num_heads_q % p->num_heads_kv) return 0;
    return 1;
}

/* the backward is defined here for d_qk == d_v only */
static int valid_bwd(const oracle_problem* p) { return valid(p) && dv_of(p) == p->head_dim; }

/* ---- entry points ------------------------------------------------------ */

/* Full forward: o in Q's layout with head_dim_v columns, lse[token_row][Hq].
 * Returns 0 on success. */
int sdpa_oracle_fwd(const oracle_problem* p, const double* q, const double* k, const double* v,
                    const int32_t* cu_q, const int32_t* cu_kv, double* o, double* lse) {
    if (!valid(p)) return 1;
    int hq = p->num_heads_q, D = dv_of(p);
    int lkmax = max_len(p, cu_kv, 0);
    for (int b = 0; b < p->batch; ++b) {
        int lq = seq_len(p, cu_q, b, 1);
#pragma omp parallel
        {
            double* s = (double*)malloc(sizeof(double) * (size_t)(lkmax > 0 ? lkmax : 1));
#pragma omp for collapse(2) schedule(dynamic, 4)
            for (int h = 0; h < hq; ++h)
                for (int i = 0; i < lq; ++i) {
                    int64_t r = token_row(p, cu_q, b, i, 1);
                    row_forward(p, q, k, v, cu_q, cu_kv, b, h, i, s, o + (r * hq + h) * D, lse + r * hq + h);
                }
            free(s);
        }
    }
    return 0;
}

/* Forward for a list of n (b, h, i) triplets: o_rows[n][head_dim_v], lse_rows[n]. */
int sdpa_oracle_fwd_rows(const oracle_problem* p, const double* q, const double* k, const double* v,
                         const int32_t* cu_q, const int32_t* cu_kv, int n, const int32_t* bhi,
                         double* o_rows, double* lse_rows) {
    if (!valid(p)) return 1;
    int lkmax = max_len(p, cu_kv, 0);
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(lkmax > 0 ? lkmax : 1));
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n; ++r)
            row_forward(p, q, k, v, cu_q, cu_kv, bhi[3 * r], bhi[3 * r + 1], bhi[3 * r + 2], s,
                        o_rows + (size_t)r * dv_of(p), lse_rows + r);
        free(s);
    }
    return 0;
}

/*
 * Backward restricted to batch entries [b_lo, b_hi) and kv heads [g_lo, g_hi)
 * (all q heads of those groups). Writes dq (Q layout), dk, dv (K/V layout)
 * for those rows only, plus o, lse and delta (delta[token_row][Hq]) for the
 * q rows touched. Any of o/lse/delta may be NULL.
 * Pass 1 runs over query rows (LSE, o, delta, dQ); pass 2 over key rows
 * (dK, dV) recomputes p and dP from the stored LSE and delta.
 */
int sdpa_oracle_bwd_part(const oracle_problem* p, const double* q, const double* k, const double* v,
                         const double* dout, const int32_t* cu_q, const int32_t* cu_kv, int b_lo,
                         int b_hi, int g_lo, int g_hi, double* dq, double* dk, double* dv, double* o,
                         double* lse, double* delta) {
    if (!valid_bwd(p)) return 1;
    int hq = p->num_heads_q, hkv = p->num_heads_kv, D = p->head_dim;
    int group = hq / hkv;
    int lqmax = max_len(p, cu_q, 1), lkmax = max_len(p, cu_kv, 0);
    int64_t nrows = rows_total(p, cu_q, 1);
    double* lse_w = (double*)malloc(sizeof(double) * (size_t)(nrows * hq + 1));
    double* del_w = (double*)malloc(sizeof(double) * (size_t)(nrows * hq + 1));
    if (!lse_w || !del_w) {
        free(lse_w);
        free(del_w);
        return 2;
    }
    (void)lqmax;
    for (int b = b_lo; b < b_hi; ++b) {
        int lq = seq_len(p, cu_q, b, 1), lk = seq_len(p, cu_kv, b, 0);
        int nh = (g_hi - g_lo) * group;
        /* pass 1: rows of Q */
#pragma omp parallel
        {
            double* s = (double*)malloc(sizeof(double) * (size_t)(lkmax > 0 ? lkmax : 1));
            double* oi = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for collapse(2) schedule(dynamic, 4)
            for (int hh = 0; hh < nh; ++hh)
                for (int i = 0; i < lq; ++i) {
                    int h = g_lo * group + hh, g = kv_head_of(p, h);
                    int64_t r = token_row(p, cu_q, b, i, 1);
                    double li;
                    row_forward(p, q, k, v, cu_q, cu_kv, b, h, i, s, oi, &li);
                    const double* doi = qrow(p, dout, cu_q, b, i, h);
                    double di = dot(doi, oi, D);
                    lse_w[r * hq + h] = li;
                    del_w[r * hq + h] = di;
                    if (o) memcpy(o + (r * hq + h) * D, oi, sizeof(double) * (size_t)D);
                    if (lse) lse[r * hq + h] = li;
                    if (delta) delta[r * hq + h] = di;
                    double* dqi = dq + (r * hq + h) * D;
                    for (int d = 0; d < D; ++d) dqi[d] = 0.0;
                    if (li == -INFINITY) continue;
                    for (int j = 0; j < lk; ++j) {
                        if (s[j] == -INFINITY) continue;
                        const double* vj = kvrow(p, v, cu_kv, b, j, g);
                        const double* kj = kvrow(p, k, cu_kv, b, j, g);
                        double pij = exp(s[j] - li);
                        double dsij = pij * (dot(doi, vj, D) - di);
                        for (int d = 0; d < D; ++d) dqi[d] += p->scale * dsij * kj[d];
                    }
                }
            free(s);
            free(oi);
        }
        /* pass 2: rows of K / V */
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
        for (int g = g_lo; g < g_hi; ++g)
            for (int j = 0; j < lk; ++j) {
                int64_t rk = token_row(p, cu_kv, b, j, 0);
                double* dkj = dk + (rk * hkv + g) * D;
                double* dvj = dv + (rk * hkv + g) * D;
                for (int d = 0; d < D; ++d) dkj[d] = dvj[d] = 0.0;
                const double* kj = kvrow(p, k, cu_kv, b, j, g);
                const double* vj = kvrow(p, v, cu_kv, b, j, g);
                for (int h = g * group; h < (g + 1) * group; ++h)
                    for (int i = 0; i < lq; ++i) {
                        if (!allowed(p, i, j, lq, lk)) continue;
                        int64_t r = token_row(p, cu_q, b, i, 1);
                        double li = lse_w[r * hq + h];
                        if (li == -INFINITY) continue;
                        const double* qi = qrow(p, q, cu_q, b, i, h);
                        const double* doi = qrow(p, dout, cu_q, b, i, h);
                        double pij = exp(p->scale * dot(qi, kj, D) - li);
                        double dsij = pij * (dot(doi, vj, D) - del_w[r * hq + h]);
                        for (int d = 0; d < D; ++d) {
                            dvj[d] += pij * doi[d];
                            dkj[d] += p->scale * dsij * qi[d];
                        }
                    }
            }
    }
    free(lse_w);
    free(del_w);
    return 0;
}

/* Full backward: every batch entry and kv head. */
int sdpa_oracle_bwd(const oracle_problem* p, const double* q, const double* k, const double* v,
                    const double* dout, const int32_t* cu_q, const int32_t* cu_kv, double* dq, double* dk,
                    double* dv, double* o, double* lse, double* delta) {
    return sdpa_oracle_bwd_part(p, q, k, v, dout, cu_q, cu_kv, 0, p->batch, 0, p->num_heads_kv, dq, dk, dv, o,
                                lse, delta);
}

/*
 * dQ for a list of n (b, h, i) triplets, given nothing but the inputs:
 * every row is independent (its LSE, o and delta come from the row itself).
 */
int sdpa_oracle_dq_rows(const oracle_problem* p, const double* q, const double* k, const double* v,
                        const double* dout, const int32_t* cu_q, const int32_t* cu_kv, int n,
                        const int32_t* bhi, double* dq_rows) {
    if (!valid_bwd(p)) return 1;
    int D = p->head_dim;
    int lkmax = max_len(p, cu_kv, 0);
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(lkmax > 0 ? lkmax : 1));
        double* oi = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n; ++r) {
            int b = bhi[3 * r], h = bhi[3 * r + 1], i = bhi[3 * r + 2], g = kv_head_of(p, h);
            int lk = seq_len(p, cu_kv, b, 0);
            double li;
            double* dqi = dq_rows + (size_t)r * D;
            row_forward(p, q, k, v, cu_q, cu_kv, b, h, i, s, oi, &li);
            for (int d = 0; d < D; ++d) dqi[d] = 0.0;
            if (li == -INFINITY) continue;
            const double* doi = qrow(p, dout, cu_q, b, i, h);
            double di = dot(doi, oi, D);
            for (int j = 0; j < lk; ++j) {
                if (s[j] == -INFINITY) continue;
                double pij = exp(s[j] - li);
                double dsij = pij * (dot(doi, kvrow(p, v, cu_kv, b, j, g), D) - di);
                const double* kj = kvrow(p, k, cu_kv, b, j, g);
                for (int d = 0; d < D; ++d) dqi[d] += p->scale * dsij * kj[d];
            }
        }
        free(s);
        free(oi);
    }
    return 0;
}

/*
 * dK and dV rows for a list of n (b, g, j) triplets (kv head g, key j of
 * sequence b). Each needs LSE_i and delta_i of every query row of the heads
 * that read kv head g, so those are computed first (one pass over the query
 * rows of each distinct (b, g) in the list); then each key row sums its
 * column of dS and P as in pass 2 of the backward above.
 */
int sdpa_oracle_dkdv_rows(const oracle_problem* p, const double* q, const double* k, const double* v,
                          const double* dout, const int32_t* cu_q, const int32_t* cu_kv, int n,
                          const int32_t* bgj, double* dk_rows, double* dv_rows) {
    if (!valid_bwd(p)) return 1;
    int hq = p->num_heads_q, D = p->head_dim;
    int group = hq / p->num_heads_kv;
    int lkmax = max_len(p, cu_kv, 0);
    int64_t nrows = rows_total(p, cu_q, 1);
    double* lse_w = (double*)malloc(sizeof(double) * (size_t)(nrows * hq + 1));
    double* del_w = (double*)malloc(sizeof(double) * (size_t)(nrows * hq + 1));
    char* done = (char*)calloc((size_t)p->batch * p->num_heads_kv + 1, 1);
    if (!lse_w || !del_w || !done) {
        free(lse_w);
        free(del_w);
        free(done);
        return 2;
    }
    for (int r = 0; r < n; ++r) {
        int b = bgj[3 * r], g = bgj[3 * r + 1];
        if (done[b * p->num_heads_kv + g]) continue;
        done[b * p->num_heads_kv + g] = 1;
        int lq = seq_len(p, cu_q, b, 1);
#pragma omp parallel
        {
            double* s = (double*)malloc(sizeof(double) * (size_t)(lkmax > 0 ? lkmax : 1));
            double* oi = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for collapse(2) schedule(dynamic, 4)
            for (int hh = 0; hh < group; ++hh)
                for (int i = 0; i < lq; ++i) {
                    int h = g * group + hh;
                    int64_t row = token_row(p, cu_q, b, i, 1);
                    double li;
                    row_forward(p, q, k, v, cu_q, cu_kv, b, h, i, s, oi, &li);
                    lse_w[row * hq + h] = li;
                    del_w[row * hq + h] = dot(qrow(p, dout, cu_q, b, i, h), oi, D);
                }
            free(s);
            free(oi);
        }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n; ++r) {
        int b = bgj[3 * r], g = bgj[3 * r + 1], j = bgj[3 * r + 2];
        int lq = seq_len(p, cu_q, b, 1), lk = seq_len(p, cu_kv, b, 0);
        double* dkj = dk_rows + (size_t)r * D;
        double* dvj = dv_rows + (size_t)r * D;
        for (int d = 0; d < D; ++d) dkj[d] = dvj[d] = 0.0;
        const double* kj = kvrow(p, k, cu_kv, b, j, g);
        const double* vj = kvrow(p, v, cu_kv, b, j, g);
        for (int h = g * group; h < (g + 1) * group; ++h)
            for (int i = 0; i < lq; ++i) {
                if (!allowed(p, i, j, lq, lk)) continue;
                int64_t row = token_row(p, cu_q, b, i, 1);
                double li = lse_w[row * hq + h];
                if (li == -INFINITY) continue;
                const double* qi = qrow(p, q, cu_q, b, i, h);
                const double* doi = qrow(p, dout, cu_q, b, i, h);
                double pij = exp(p->scale * dot(qi, kj, D) - li);
                double dsij = pij * (dot(doi, vj, D) - del_w[row * hq + h]);
                for (int d = 0; d < D; ++d) {
                    dvj[d] += pij * doi[d];
                    dkj[d] += p->scale * dsij * qi[d];
                }
            }
    }
    free(lse_w);
    free(del_w);
    free(done);
    return 0;
}

/*
 * Merge of partial attention results over a split of the keys (the
 * context-parallel LSE handling of TransformerEngine PR #3527 and PR #3693,
 * "neutral statistics for empty ragged ring blocks"). Written out as the
 * log-sum-exp identity that makes attention over the union of key blocks
 * equal to the combination of the blocks' own results: for every item
 * (a row of one head),
 *   LSE = ln sum_k exp(LSE_k),   O = sum_k exp(LSE_k - LSE) O_k.
 * A block that saw no keys carries LSE_k = -inf and contributes nothing;
 * when every block is empty, O = 0 and LSE = -inf (the forward's convention
 * for a row without keys).
 * o_parts[n_parts][items][d], lse_parts[n_parts][items] -> o[items][d], lse[items].
 */
int sdpa_oracle_merge(int n_parts, int64_t items, int d, const double* o_parts, const double* lse_parts, double* o,
                      double* lse) {
    if (n_parts < 1 || items < 0 || d < 1) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t it = 0; it < items; ++it) {
        double m = -INFINITY;
        for (int k = 0; k < n_parts; ++k)
            if (lse_parts[(int64_t)k * items + it] > m) m = lse_parts[(int64_t)k * items + it];
        double* oi = o + it * d;
        for (int c = 0; c < d; ++c) oi[c] = 0.0;
        if (m == -INFINITY) {
            lse[it] = -INFINITY;
            continue;
        }
        double s = 0.0;
        for (int k = 0; k < n_parts; ++k) s += exp(lse_parts[(int64_t)k * items + it] - m);
        const double l = m + log(s);
        lse[it] = l;
        for (int k = 0; k < n_parts; ++k) {
            const double w = exp(lse_parts[(int64_t)k * items + it] - l);
            const double* ok = o_parts + ((int64_t)k * items + it) * d;
            for (int c = 0; c < d; ++c) oi[c] += w * ok[c];
        }
    }
    return 0;
}

/* The softmax probabilities of the definition, p_ij = exp(s_ij - LSE_i) for
 * every allowed key j of row i's sequence and 0 elsewhere, written to
 * probs[(token_row * Hq + h) * lk_max + j] (lk_max = the longest key
 * sequence). Returns 0 on success. */
int sdpa_oracle_probs(const oracle_problem* p, const double* q, const double* k, const int32_t* cu_q,
                      const int32_t* cu_kv, double* probs) {
    if (!valid(p)) return 1;
    int hq = p->num_heads_q, lkmax = max_len(p, cu_kv, 0);
    for (int b = 0; b < p->batch; ++b) {
        int lq = seq_len(p, cu_q, b, 1), lk = seq_len(p, cu_kv, b, 0);
#pragma omp parallel
        {
            double* srow = (double*)malloc(sizeof(double) * (size_t)(lkmax > 0 ? lkmax : 1));
#pragma omp for collapse(2) schedule(dynamic, 4)
            for (int h = 0; h < hq; ++h)
                for (int i = 0; i < lq; ++i) {
                    double* prow = probs + (token_row(p, cu_q, b, i, 1) * hq + h) * lkmax;
                    double l = row_scores(p, q, k, cu_q, cu_kv, b, h, i, srow);
                    for (int j = 0; j < lkmax; ++j)
                        prow[j] = (j < lk && l != -INFINITY && srow[j] != -INFINITY) ? exp(srow[j] - l) : 0.0;
                }
            free(srow);
        }
    }
    return 0;
}

/*
 * FP8 E4M3 forward (the FP8 variant of this kernel family). Reading of
 * TransformerEngine PR #3705's closing note ("Amax S"): with E4M3 inputs the
 * softmax output is stored in E4M3 under a fixed scale, 448 (the format's
 * largest value) without dropout, so no amax of it is ever needed. A fixed
 * scale does that only if the stored probabilities are normalised by the
 * row's largest one (then the largest is stored as 448 exactly); they are
 * divided by the row sum after the product with V. Written out:
 *   Q, K, V are E4M3 codes with per-tensor descales d_q, d_k, d_v (the real
 *   value of a code c is decode(c) * d);
 *   s_ij  = scale * d_q * d_k * sum_d decode(q_id) decode(k_jd), masked as above;
 *   m_i   = max_j s_ij;  L_i = sum_j exp(s_ij - m_i);  LSE_i = m_i + ln L_i;
 *   P8_ij = e4m3(exp(s_ij - m_i) * scale_s);
 *   o_i   = sum_j P8_ij decode(v_j) * d_v / (scale_s * L_i).
 * The softmax is exact (float64); only the stored P is rounded.
 */

/* E4M3, the finite-only variant of the OCP 8-bit float: sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits. Exponent field 0 holds the subnormals
 * m/8 * 2^-6; S.1111.111 is NaN; there is no infinity; the largest finite
 * magnitude is 1.75 * 2^8 = 448. */
double sdpa_oracle_e4m3_decode(uint8_t c) {
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);          /* m/8 * 2^-6 */
    else
        v = ldexp(8.0 + m, e - 10);        /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Nearest E4M3 value, ties to the even mantissa; magnitudes of 448 and more
 * saturate to 448 (NaN stays NaN). Between 2^k and 2^(k+1) (k >= -6) the
 * representable values are 2^(k-3) apart; below 2^-6 (subnormals) 2^-9. */
double sdpa_oracle_e4m3_round(double x) {
    if (isnan(x)) return x;
    double a = fabs(x);
    if (a >= 448.0) return copysign(448.0, x);
    int k;
    frexp(a, &k);                          /* a in [2^(k-1), 2^k) */
    int ex = k - 1 < -6 ? -6 : k - 1;
    double spacing = ldexp(1.0, ex - 3);
    return copysign(nearbyint(a / spacing) * spacing, x);  /* round-to-nearest-even mode */
}

void sdpa_oracle_e4m3_round_array(int64_t n, const double* x, double* y) {
    for (int64_t i = 0; i < n; ++i) y[i] = sdpa_oracle_e4m3_round(x[i]);
}

void sdpa_oracle_e4m3_decode_array(int64_t n, const uint8_t* c, double* y) {
    for (int64_t i = 0; i < n; ++i) y[i] = sdpa_oracle_e4m3_decode(c[i]);
}

/* o in Q's layout with head_dim_v columns, lse[token_row][Hq]; q8/k8/v8 are
 * E4M3 codes in their layouts. Returns 0 on success. */
int sdpa_oracle_fwd_fp8(const oracle_problem* p, const uint8_t* q8, const uint8_t* k8, const uint8_t* v8,
                        double descale_q, double descale_k, double descale_v, double scale_s,
                        const int32_t* cu_q, const int32_t* cu_kv, double* o, double* lse) {
    if (!valid(p) || !(scale_s > 0.0)) return 1;
    int hq = p->num_heads_q, D = p->head_dim, DV = dv_of(p);
    int64_t nq = rows_total(p, cu_q, 1) * hq * D;
    int64_t nk = rows_total(p, cu_kv, 0) * p->num_heads_kv * D;
    int64_t nv = rows_total(p, cu_kv, 0) * p->num_heads_kv * DV;
    double* qd = (double*)malloc(sizeof(double) * (size_t)(nq > 0 ? nq : 1));
    double* kd = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    double* vd = (double*)malloc(sizeof(double) * (size_t)(nv > 0 ? nv : 1));
    if (!qd || !kd || !vd) {
        free(qd);
        free(kd);
        free(vd);
        return 2;
    }
    sdpa_oracle_e4m3_decode_array(nq, q8, qd);
    sdpa_oracle_e4m3_decode_array(nk, k8, kd);
    sdpa_oracle_e4m3_decode_array(nv, v8, vd);
    oracle_problem ps = *p;
    ps.scale = p->scale * descale_q * descale_k;   /* s_ij on the decoded codes */
    int lkmax = max_len(p, cu_kv, 0);
    for (int b = 0; b < p->batch; ++b) {
        int lq = seq_len(p, cu_q, b, 1), lk = seq_len(p, cu_kv, b, 0);
#pragma omp parallel
        {
            double* srow = (double*)malloc(sizeof(double) * (size_t)(lkmax > 0 ? lkmax : 1));
#pragma omp for collapse(2) schedule(dynamic, 4)
            for (int h = 0; h < hq; ++h)
                for (int i = 0; i < lq; ++i) {
                    int64_t r = token_row(p, cu_q, b, i, 1);
                    double* orow = o + (r * hq + h) * DV;
                    double l = row_scores(&ps, qd, kd, cu_q, cu_kv, b, h, i, srow);
                    for (int d = 0; d < DV; ++d) orow[d] = 0.0;
                    lse[r * hq + h] = l;
                    if (l == -INFINITY) continue;
                    int g = kv_head_of(p, h);
                    double m = -INFINITY, sum = 0.0;
                    for (int j = 0; j < lk; ++j)
                        if (srow[j] > m) m = srow[j];
                    for (int j = 0; j < lk; ++j) {
                        if (srow[j] == -INFINITY) continue;
                        sum += exp(srow[j] - m);
                        double p8 = sdpa_oracle_e4m3_round(exp(srow[j] - m) * scale_s);
                        const double* vj = vrow(p, vd, cu_kv, b, j, g);
                        for (int d = 0; d < DV; ++d) orow[d] += p8 * vj[d];
                    }
                    for (int d = 0; d < DV; ++d) orow[d] *= descale_v / (scale_s * sum);
                }
            free(srow);
        }
    }
    free(qd);
    free(kd);
    free(vd);
    return 0;
}

int sdpa_oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
