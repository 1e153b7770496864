/*
 * nsa_oracle.c -- plain fp64 CPU oracle for NSA selected attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA path is compared
 * against.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * load it; the product path never calls it and shares no code with it.
 *
 * What it computes (selected-attention branch of Native Sparse Attention, as
 * described in "FSA: An Alternative Efficient Implementation of Native Sparse
 * Attention Kernel", key designs 1-4, and the Flash-Sparse-Attention README,
 * "Method"):  every query token t of KV head h picks T KV blocks of B_K keys
 * (the selection tensor, h_K x N x T); each of the g query heads of that KV
 * head attends, causally, to the union of the keys of those blocks, with one
 * softmax per query over that union.  FSA "does not change the NSA algorithm",
 * so the oracle is the plain definition written out:
 *
 *   B(t)   = { b in sel[h,t,:] : 0 <= b <= c(t), b < ceil(len/B_K) }  (a set)
 *   K(t)   = { b*B_K + i : b in B(t), 0 <= i < B_K, b*B_K + i <= tau }
 *   s_j    = scale * <q_t, k_j>                     (fp64)
 *   lse_t  = m + ln sum_j exp(s_j - m),  m = max_j s_j
 *   o_t    = sum_j exp(s_j - lse_t) v_j
 *
 * tau is the token's position inside its own packed sequence and c(t) = tau / B_K;
 * block indices are local to the sequence.  Empty key sets give o = 0,
 * lse = -inf.  Backward is the direct derivative of the above:
 *   P_j = exp(s_j - lse), dP_j = <dO_t, v_j>, D_t = sum_j P_j dP_j,
 *   dS_j = P_j (dP_j - D_t), dq_t = scale sum_j dS_j k_j,
 *   dk_j += scale dS_j q_t, dv_j += P_j dO_t   (summed over all tokens and the g heads).
 *
 * The index tensors of key design 2 (I_i: the tokens that selected KV block i;
 * O_i: where each (token, slot) pair's partial result lives in the compact
 * buffer) are produced by nsa_oracle_index in the order that makes them unique:
 * KV head major, then global block id, tokens ascending inside a block, slots
 * ascending inside a token, first occurrence of a duplicate wins.
 *
 * Layouts: q/out/dq/dout [N, h_q, d]; k/v/dk/dv [N, h_k, d]; sel [h_k, N, T];
 * lse [h_q, N]; cu_seqlens [S+1]; query head hq reads KV head hq / g.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_MAX_TOPK 64

static void set_threads(int num_threads) {
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
}

int nsa_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sequence containing packed token t: largest s with cu[s] <= t. */
static int seq_of(const int32_t *cu, int num_seqs, int64_t t) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/* Valid slots of one selection row.  keep[k] = 1 when slot k names a block that is
 * in range (0 <= b <= c, b < nblk) and did not occur in an earlier slot. */
static int valid_slots(const int32_t *row, int topk, int c, int nblk, int *keep) {
    int n = 0;
    for (int k = 0; k < topk; ++k) {
        int b = row[k];
        keep[k] = 0;
        if (b < 0 || b > c || b >= nblk) continue;
        int dup = 0;
        for (int k2 = 0; k2 < k; ++k2)
            if (keep[k2] && row[k2] == b) { dup = 1; break; }
        if (dup) continue;
        keep[k] = 1;
        ++n;
    }
    return n;
}

/* B(t) in ascending block order. */
static int token_blocks(const int32_t *row, int topk, int c, int nblk, int *blocks) {
    int keep[ORC_MAX_TOPK];
    int n = 0;
    valid_slots(row, topk, c, nblk, keep);
    for (int k = 0; k < topk; ++k)
        if (keep[k]) blocks[n++] = row[k];
    for (int i = 1; i < n; ++i) {           /* insertion sort */
        int x = blocks[i], j = i - 1;
        while (j >= 0 && blocks[j] > x) { blocks[j + 1] = blocks[j]; --j; }
        blocks[j + 1] = x;
    }
    return n;
}

/* Local key indices K(t) (ascending); returns |K(t)|.  With window > 0 (the
 * sliding-window branch, window_size of the Flash-Sparse-Attention README) a key is
 * also required to lie in the window: kappa > tau - window. */
static int token_keys(const int32_t *row, int topk, int tau, int len, int block, int window,
                      int *keys) {
    int blocks[ORC_MAX_TOPK];
    int c = tau / block, nblk = (len + block - 1) / block;
    int nb = token_blocks(row, topk, c, nblk, blocks), n = 0;
    for (int i = 0; i < nb; ++i)
        for (int j = 0; j < block; ++j) {
            int kappa = blocks[i] * block + j;
            if (kappa > tau) break;
            if (window > 0 && kappa <= tau - window) continue;
            keys[n++] = kappa;
        }
    return n;
}

static double dot(const double *a, const double *b, int d) {
    double s = 0.0;
    for (int i = 0; i < d; ++i) s += a[i] * b[i];
    return s;
}

static int check_args(int num_seqs, const int32_t *cu, int h_k, int g, int d, int block, int topk) {
    if (num_seqs < 1 || h_k < 1 || g < 1 || d < 1 || block < 1 || topk < 1 || topk > ORC_MAX_TOPK)
        return 1;
    if (cu[0] != 0) return 1;
    for (int s = 0; s < num_seqs; ++s)
        if (cu[s + 1] < cu[s]) return 1;
    return 0;
}

/* Forward for one (token, query head): writes o[d] and returns lse.  Scratch: keys
 * and scores of size topk*block. */
static double fwd_one(const int32_t *cu, int num_seqs, int h_k, int g, int d, int block, int topk,
                      int window, const int32_t *sel, const double *q, const double *k,
                      const double *v, double scale, int64_t t, int hq, double *o, int *keys,
                      double *sc) {
    const int64_t N = cu[num_seqs];
    const int h_q = h_k * g, h = hq / g;
    const int s = seq_of(cu, num_seqs, t);
    const int tau = (int)(t - cu[s]), len = cu[s + 1] - cu[s];
    const int nk =
        token_keys(sel + ((int64_t)h * N + t) * topk, topk, tau, len, block, window, keys);
    const double *qt = q + (t * h_q + hq) * d;
    for (int i = 0; i < d; ++i) o[i] = 0.0;
    if (nk == 0) return -INFINITY;
    double m = -INFINITY;
    for (int j = 0; j < nk; ++j) {
        int64_t kt = cu[s] + keys[j];
        sc[j] = scale * dot(qt, k + (kt * h_k + h) * d, d);
        if (sc[j] > m) m = sc[j];
    }
    double l = 0.0;
    for (int j = 0; j < nk; ++j) l += exp(sc[j] - m);
    const double lse = m + log(l);
    for (int j = 0; j < nk; ++j) {
        const double p = exp(sc[j] - lse);
        const double *vj = v + ((cu[s] + keys[j]) * h_k + h) * d;
        for (int i = 0; i < d; ++i) o[i] += p * vj[i];
    }
    return lse;
}

int nsa_oracle_fwd_w(int num_seqs, const int32_t *cu, int h_k, int g, int d, int block, int topk,
                     int window, const int32_t *sel, const double *q, const double *k,
                     const double *v, double scale, double *out, double *lse, int num_threads) {
    if (check_args(num_seqs, cu, h_k, g, d, block, topk)) return 1;
    set_threads(num_threads);
    const int64_t N = cu[num_seqs];
    const int h_q = h_k * g;
    int bad = 0;
#pragma omp parallel reduction(|: bad)
    {
        int *keys = (int *)malloc(sizeof(int) * (size_t)topk * block);
        double *sc = (double *)malloc(sizeof(double) * (size_t)topk * block);
        if (!keys || !sc) bad = 1;
#pragma omp for schedule(dynamic, 64)
        for (int64_t i = 0; i < N * h_q; ++i) {
            if (!keys || !sc) continue;
            int64_t t = i / h_q;
            int hq = (int)(i % h_q);
            lse[(int64_t)hq * N + t] = fwd_one(cu, num_seqs, h_k, g, d, block, topk, window, sel,
                                               q, k, v, scale, t, hq, out + (t * h_q + hq) * d,
                                               keys, sc);
        }
        free(keys);
        free(sc);
    }
    return bad ? 2 : 0;
}

int nsa_oracle_fwd(int num_seqs, const int32_t *cu, int h_k, int g, int d, int block, int topk,
                   const int32_t *sel, const double *q, const double *k, const double *v,
                   double scale, double *out, double *lse, int num_threads) {
    return nsa_oracle_fwd_w(num_seqs, cu, h_k, g, d, block, topk, 0, sel, q, k, v, scale, out,
                            lse, num_threads);
}

/* Forward on selected (token, query head) pairs only: rows[2*i] = t, rows[2*i+1] = hq;
 * out_rows [n_rows, d], lse_rows [n_rows].  Same arithmetic as nsa_oracle_fwd. */
int nsa_oracle_fwd_rows(int num_seqs, const int32_t *cu, int h_k, int g, int d, int block, int topk,
                        const int32_t *sel, const double *q, const double *k, const double *v,
                        double scale, int64_t n_rows, const int64_t *rows, double *out_rows,
                        double *lse_rows, int num_threads) {
    if (check_args(num_seqs, cu, h_k, g, d, block, topk)) return 1;
    set_threads(num_threads);
    const int64_t N = cu[num_seqs];
    for (int64_t i = 0; i < n_rows; ++i)
        if (rows[2 * i] < 0 || rows[2 * i] >= N || rows[2 * i + 1] < 0 || rows[2 * i + 1] >= h_k * g)
            return 1;
    int bad = 0;
#pragma omp parallel reduction(|: bad)
    {
        int *keys = (int *)malloc(sizeof(int) * (size_t)topk * block);
        double *sc = (double *)malloc(sizeof(double) * (size_t)topk * block);
        if (!keys || !sc) bad = 1;
#pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < n_rows; ++i) {
            if (!keys || !sc) continue;
            lse_rows[i] = fwd_one(cu, num_seqs, h_k, g, d, block, topk, 0, sel, q, k, v, scale,
                                  rows[2 * i], (int)rows[2 * i + 1], out_rows + i * d, keys, sc);
        }
        free(keys);
        free(sc);
    }
    return bad ? 2 : 0;
}

/*
 * Backward by direct differentiation.  Pass 1, per (token, query head): the
 * softmax statistics lse_t, D_t = sum_j P_j dP_j and dq_t.  Pass 2, per (KV head,
 * key block): dk_j and dv_j as the sums over every (token, query head) whose key
 * set K(t) contains key j.  No blocking beyond the definition; the pass split only
 * keeps the parallel loops free of write conflicts.
 */
int nsa_oracle_bwd_w(int num_seqs, const int32_t *cu, int h_k, int g, int d, int block, int topk,
                     int window, const int32_t *sel, const double *q, const double *k,
                     const double *v, const double *dout, double scale, double *dq, double *dk,
                     double *dv, int num_threads) {
    if (check_args(num_seqs, cu, h_k, g, d, block, topk)) return 1;
    set_threads(num_threads);
    const int64_t N = cu[num_seqs];
    const int h_q = h_k * g;
    double *lse = (double *)malloc(sizeof(double) * (size_t)(N * h_q));
    double *Dt = (double *)malloc(sizeof(double) * (size_t)(N * h_q));
    if (!lse || !Dt) { free(lse); free(Dt); return 2; }
    int bad = 0;
    /* pass 1: lse, D and dq per (t, hq) */
#pragma omp parallel reduction(|: bad)
    {
        int *keys = (int *)malloc(sizeof(int) * (size_t)topk * block);
        double *sc = (double *)malloc(sizeof(double) * (size_t)topk * block);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        if (!keys || !sc || !o) bad = 1;
#pragma omp for schedule(dynamic, 64)
        for (int64_t i = 0; i < N * h_q; ++i) {
            if (!keys || !sc || !o) continue;
            const int64_t t = i / h_q;
            const int hq = (int)(i % h_q), h = hq / g;
            const int s = seq_of(cu, num_seqs, t);
            const int tau = (int)(t - cu[s]), len = cu[s + 1] - cu[s];
            double *dqt = dq + (t * h_q + hq) * d;
            for (int x = 0; x < d; ++x) dqt[x] = 0.0;
            const int nk = token_keys(sel + ((int64_t)h * N + t) * topk, topk, tau, len, block,
                                      window, keys);
            if (nk == 0) { lse[i] = -INFINITY; Dt[i] = 0.0; continue; }
            const double *qt = q + (t * h_q + hq) * d;
            const double *dot_ = dout + (t * h_q + hq) * d;
            double m = -INFINITY, l = 0.0;
            for (int j = 0; j < nk; ++j) {
                sc[j] = scale * dot(qt, k + ((cu[s] + keys[j]) * h_k + h) * d, d);
                if (sc[j] > m) m = sc[j];
            }
            for (int j = 0; j < nk; ++j) l += exp(sc[j] - m);
            const double L = m + log(l);
            double D = 0.0;
            for (int j = 0; j < nk; ++j) {
                const double p = exp(sc[j] - L);
                const double dp = dot(dot_, v + ((cu[s] + keys[j]) * h_k + h) * d, d);
                D += p * dp;
            }
            for (int j = 0; j < nk; ++j) {
                const int64_t kt = cu[s] + keys[j];
                const double p = exp(sc[j] - L);
                const double dp = dot(dot_, v + (kt * h_k + h) * d, d);
                const double ds = p * (dp - D);
                const double *kj = k + (kt * h_k + h) * d;
                for (int x = 0; x < d; ++x) dqt[x] += scale * ds * kj[x];
            }
            lse[i] = L;
            Dt[i] = D;
        }
        free(keys);
        free(sc);
        free(o);
    }
    if (bad) { free(lse); free(Dt); return 2; }
    /* pass 2: dk, dv per (KV head, sequence block) */
    int64_t nb_total = 0;
    for (int s = 0; s < num_seqs; ++s) nb_total += (cu[s + 1] - cu[s] + block - 1) / block;
    for (int64_t i = 0; i < N * h_k * d; ++i) { dk[i] = 0.0; dv[i] = 0.0; }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < nb_total * h_k; ++w) {
        const int h = (int)(w % h_k);
        int64_t gb = w / h_k;
        int s = 0;
        while (gb >= (cu[s + 1] - cu[s] + block - 1) / block) {
            gb -= (cu[s + 1] - cu[s] + block - 1) / block;
            ++s;
        }
        const int b = (int)gb, len = cu[s + 1] - cu[s];
        for (int tau = b * block; tau < len; ++tau) {          /* only later tokens can use block b */
            const int64_t t = cu[s] + tau;
            /* b <= c(t) and b < nblk hold here, so b is in B(t) iff some slot names it */
            const int32_t *row = sel + ((int64_t)h * N + t) * topk;
            int has = 0;
            for (int x = 0; x < topk; ++x) has |= (row[x] == b);
            if (!has) continue;
            for (int j = 0; j < g; ++j) {
                const int hq = h * g + j;
                const double L = lse[t * h_q + hq], D = Dt[t * h_q + hq];
                const double *qt = q + (t * h_q + hq) * d;
                const double *dot_ = dout + (t * h_q + hq) * d;
                for (int i = 0; i < block; ++i) {
                    const int kappa = b * block + i;
                    if (kappa > tau) break;
                    if (window > 0 && kappa <= tau - window) continue;
                    const int64_t kt = cu[s] + kappa;
                    const double *kj = k + (kt * h_k + h) * d, *vj = v + (kt * h_k + h) * d;
                    const double p = exp(scale * dot(qt, kj, d) - L);
                    const double ds = p * (dot(dot_, vj, d) - D);
                    double *dkj = dk + (kt * h_k + h) * d, *dvj = dv + (kt * h_k + h) * d;
                    for (int x = 0; x < d; ++x) {
                        dkj[x] += scale * ds * qt[x];
                        dvj[x] += p * dot_[x];
                    }
                }
            }
        }
    }
    free(lse);
    free(Dt);
    return 0;
}

int nsa_oracle_bwd(int num_seqs, const int32_t *cu, int h_k, int g, int d, int block, int topk,
                   const int32_t *sel, const double *q, const double *k, const double *v,
                   const double *dout, double scale, double *dq, double *dk, double *dv,
                   int num_threads) {
    return nsa_oracle_bwd_w(num_seqs, cu, h_k, g, d, block, topk, 0, sel, q, k, v, dout, scale,
                            dq, dk, dv, num_threads);
}

/* Selection rows of the sliding window: token t (local position tau) names the blocks
 * that hold keys of (tau - window, tau], newest first (c, c - 1, ...), the rest -1.
 * Returns 1 when topk is too small for some token. */
int nsa_oracle_window_select(int num_seqs, const int32_t *cu, int h_k, int block, int topk,
                             int window, int32_t *sel) {
    const int64_t N = cu[num_seqs];
    for (int s = 0; s < num_seqs; ++s)
        for (int tau = 0; tau < cu[s + 1] - cu[s]; ++tau) {
            const int64_t t = cu[s] + tau;
            const int c = tau / block;
            const int first = tau - window + 1 > 0 ? (tau - window + 1) / block : 0;
            if (c - first + 1 > topk) return 1;
            for (int h = 0; h < h_k; ++h) {
                int32_t *row = sel + ((int64_t)h * N + t) * topk;
                for (int k = 0; k < topk; ++k) row[k] = (c - k >= first) ? c - k : -1;
            }
        }
    return 0;
}

/* Number of KV blocks per head over the packed batch: sum_s ceil(len_s / B_K). */
int64_t nsa_oracle_num_blocks(int num_seqs, const int32_t *cu, int block) {
    int64_t nb = 0;
    for (int s = 0; s < num_seqs; ++s) nb += (cu[s + 1] - cu[s] + block - 1) / block;
    return nb;
}

/*
 * Index tensors.  counts[h*NB + gb] = number of tokens whose valid, de-duplicated
 * selection contains global block gb (= local block + blocks of earlier sequences);
 * offsets = exclusive prefix sum of counts (h-major), offsets[h_k*NB] = total;
 * q_list[offsets[h*NB+gb] + r] = r-th such token in ascending order (I_i);
 * slot_map[(h*N + t)*T + k] = that position for a kept slot, -1 otherwise (O_i).
 * q_list must hold h_k*N*T entries.  Returns the total number of pairs, or -1.
 */
int64_t nsa_oracle_index(int num_seqs, const int32_t *cu, int h_k, int block, int topk,
                         const int32_t *sel, int32_t *counts, int32_t *offsets, int32_t *q_list,
                         int32_t *slot_map) {
    if (check_args(num_seqs, cu, h_k, 1, 1, block, topk)) return -1;
    const int64_t N = cu[num_seqs];
    const int64_t NB = nsa_oracle_num_blocks(num_seqs, cu, block);
    int64_t *blk_start = (int64_t *)malloc(sizeof(int64_t) * (size_t)(num_seqs + 1));
    int64_t *fill = (int64_t *)malloc(sizeof(int64_t) * (size_t)(h_k * NB + 1));
    if (!blk_start || !fill) { free(blk_start); free(fill); return -1; }
    blk_start[0] = 0;
    for (int s = 0; s < num_seqs; ++s)
        blk_start[s + 1] = blk_start[s] + (cu[s + 1] - cu[s] + block - 1) / block;
    for (int64_t i = 0; i < h_k * NB; ++i) counts[i] = 0;
    int keep[ORC_MAX_TOPK];
    for (int h = 0; h < h_k; ++h)
        for (int64_t t = 0; t < N; ++t) {
            const int s = seq_of(cu, num_seqs, t);
            const int tau = (int)(t - cu[s]), len = cu[s + 1] - cu[s];
            const int32_t *row = sel + ((int64_t)h * N + t) * topk;
            valid_slots(row, topk, tau / block, (len + block - 1) / block, keep);
            for (int k = 0; k < topk; ++k)
                if (keep[k]) counts[h * NB + blk_start[s] + row[k]] += 1;
        }
    int64_t run = 0;
    for (int64_t i = 0; i < h_k * NB; ++i) {
        offsets[i] = (int32_t)run;
        fill[i] = run;
        run += counts[i];
    }
    offsets[h_k * NB] = (int32_t)run;
    for (int h = 0; h < h_k; ++h)
        for (int64_t t = 0; t < N; ++t) {
            const int s = seq_of(cu, num_seqs, t);
            const int tau = (int)(t - cu[s]), len = cu[s + 1] - cu[s];
            const int32_t *row = sel + ((int64_t)h * N + t) * topk;
            int32_t *sm = slot_map + ((int64_t)h * N + t) * topk;
            valid_slots(row, topk, tau / block, (len + block - 1) / block, keep);
            for (int k = 0; k < topk; ++k) {
                if (!keep[k]) { sm[k] = -1; continue; }
                const int64_t pos = fill[h * NB + blk_start[s] + row[k]]++;
                q_list[pos] = (int32_t)t;
                sm[k] = (int32_t)pos;
            }
        }
    free(blk_start);
    free(fill);
    return run;
}
