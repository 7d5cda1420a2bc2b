/*
 * gqa_oracle.c -- plain, slow, fp64 CPU oracle for causal grouped-query
 * scaled-dot-product attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the test suite, the package's smoke check and the
 * CPU-baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (one head at a time, every step a full T x T matrix):
 *   S_ij   = scale * sum_d Q_id K_jd                      score matrix
 *   M_ij   = causal ? (j <= i) : 1                        mask (diagonal kept)
 *   LSE_i  = log sum_{j: M_ij} exp(S_ij)                  natural log
 *   P_ij   = M_ij * exp(S_ij - LSE_i)                     row softmax
 *   O_i    = sum_j P_ij V_j
 * and, for the scalar L = sum(dO * O):
 *   dP_ij  = sum_d dO_id V_jd
 *   Delta_i= sum_j P_ij dP_ij
 *   dS_ij  = P_ij (dP_ij - Delta_i)
 *   dQ_i   = scale * sum_j dS_ij K_j
 *   dK_j  += scale * sum_i dS_ij Q_i      (summed over the query heads of a group)
 *   dV_j  += sum_i P_ij dO_i              (summed over the query heads of a group)
 *
 * Sources: the softmax / ScaledDotProductAttention / MultiHeadAttention
 * components of "Project Overview" (llm-from-scratch), section "Core Stack:
 * llm/ -- llm/transformer.py"; the materialising "slower, easier-to-read
 * reference path" of its section "Performance Layer: kernel/ and parallel/";
 * "Decoder-only MHA/GQA ... causal attention" and the causal GQA backward of
 * the microLLM-rocm README, section "Why this project exists".  The pages do
 * not print the equations; the lines above are the textbook definition they
 * name.  Readings of points the pages leave open:
 *   - query head h uses key/value head floor(h / G), G = Hq / Hkv;
 *   - key j is visible to query i iff j <= i (diagonal included), Tq == Tk;
 *   - LSE is a natural logarithm;
 *   - a row with no visible key (not reachable with the masks above) gives
 *     O = 0 and LSE = -inf.
 *
 * Layout: every tensor is addressed through (row stride, head stride) so the
 * same per-head routine serves the dense [B,H,T,D] layout and the packed
 * variable-length layout [total,H,D].  LSE / Delta: dense [B,H,T], packed
 * [H,total].
 *
 * Parallelism: OpenMP over the rows of each step inside one head (rows are
 * independent in every step listed above).  No blocking, fusion or
 * reordering of the arithmetic beyond the definition.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One head's view: element (t, d) at base[t * rs + d]. */
typedef struct {
    const double* base;
    long rs;
} cview;

typedef struct {
    double* base;
    long rs;
} mview;

/* PLANT selects a deliberately wrong variant, compiled only by the test that
 * checks the pins catch such mistakes (0 = the oracle as stated above). */
#ifndef PLANT
#define PLANT 0
#endif

static int visible(long i, long j, int causal) {
    if (PLANT == 1) return causal ? (j < i) : 1;      /* planted: diagonal dropped */
    return causal ? (j <= i) : 1;
}

static long kv_head(long h, long G, long Hkv) {
    if (PLANT == 2) return h % Hkv;                     /* planted: interleaved groups */
    (void)Hkv;
    return h / G;
}

/* S = scale * Q K^T restricted to the mask; masked entries are -inf. */
static void scores(cview q, cview k, long T, long D, int causal, double scale, double* S) {
    long i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < T; ++i) {
        for (long j = 0; j < T; ++j) {
            double acc = 0.0;
            if (visible(i, j, causal)) {
                for (long d = 0; d < D; ++d) acc += q.base[i * q.rs + d] * k.base[j * k.rs + d];
                S[i * T + j] = scale * acc;
            } else {
                S[i * T + j] = -INFINITY;
            }
        }
    }
}

/* LSE_i = log sum_j exp(S_ij) (max-subtracted), then P = exp(S - LSE) in place. */
static void softmax_rows(double* S, long T, double* lse_row /* T, stride 1 */) {
    long i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < T; ++i) {
        double* s = S + i * T;
        double m = -INFINITY;
        for (long j = 0; j < T; ++j) if (s[j] > m) m = s[j];
        if (m == -INFINITY) {              /* no visible key */
            for (long j = 0; j < T; ++j) s[j] = 0.0;
            lse_row[i] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (long j = 0; j < T; ++j) sum += exp(s[j] - m);
        double l = m + (PLANT == 5 ? log2(sum) : log(sum)); /* 5: planted wrong base */
        lse_row[i] = l;
        for (long j = 0; j < T; ++j) s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - l);
    }
}

/* Out = A V with A a T x T matrix:  Out_i = sum_j A_ij V_j. */
static void rows_times(const double* A, cview v, long T, long D, mview out, int accumulate) {
    long i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < T; ++i) {
        for (long d = 0; d < D; ++d) {
            double acc = 0.0;
            for (long j = 0; j < T; ++j) acc += A[i * T + j] * v.base[j * v.rs + d];
            if (accumulate) out.base[i * out.rs + d] += acc; else out.base[i * out.rs + d] = acc;
        }
    }
}

/* Out_j (+)= c * sum_i A_ij X_i   (A transposed times X). */
static void cols_times(const double* A, cview x, long T, long D, double c, mview out) {
    long j;
#pragma omp parallel for schedule(static)
    for (j = 0; j < T; ++j) {
        for (long d = 0; d < D; ++d) {
            double acc = 0.0;
            for (long i = 0; i < T; ++i) acc += A[i * T + j] * x.base[i * x.rs + d];
            out.base[j * out.rs + d] += c * acc;
        }
    }
}

/* One head forward: O (T x D) and LSE (T).  P (T x T scratch) holds the
 * probabilities on return. */
static void head_fwd(cview q, cview k, cview v, long T, long D, int causal, double scale,
                     mview o, double* lse_row, double* P) {
    scores(q, k, T, D, causal, scale, P);
    softmax_rows(P, T, lse_row);
    rows_times(P, v, T, D, o, 0);
}

/* One head backward.  Adds this query head's share into dk, dv (the
 * group sum) and writes dq.  P, dS: T x T scratch.  Optionally returns O, LSE
 * and Delta of the head. */
static void head_bwd(cview q, cview k, cview v, cview dout, long T, long D, int causal, double scale,
                     mview dq, mview dk, mview dv, double* P, double* dS,
                     double* lse_row, double* delta_row, mview o) {
    head_fwd(q, k, v, T, D, causal, scale, o, lse_row, P);
    long i;
    /* dP = dO V^T, then Delta_i = sum_j P_ij dP_ij, then dS = P o (dP - Delta). */
#pragma omp parallel for schedule(static)
    for (i = 0; i < T; ++i) {
        double delta = 0.0;
        for (long j = 0; j < T; ++j) {
            double dp = 0.0;
            for (long d = 0; d < D; ++d) dp += dout.base[i * dout.rs + d] * v.base[j * v.rs + d];
            dS[i * T + j] = dp;                 /* dP for now */
            delta += P[i * T + j] * dp;
        }
        delta_row[i] = delta;
        if (PLANT == 4) delta = -delta;                 /* planted: sign error */
        for (long j = 0; j < T; ++j) dS[i * T + j] = P[i * T + j] * (dS[i * T + j] - delta);
    }
    /* dQ = scale * dS K */
    rows_times(dS, k, T, D, dq, 0);
#pragma omp parallel for schedule(static)
    for (i = 0; i < T; ++i)
        for (long d = 0; d < D; ++d) dq.base[i * dq.rs + d] *= scale;
    /* dK += scale * dS^T Q ;  dV += P^T dO */
    cols_times(dS, q, T, D, PLANT == 3 ? 1.0 : scale, dk);   /* 3: planted missing scale */
    cols_times(P, dout, T, D, 1.0, dv);
}

/* Rounding-error scale of the backward outputs when P, dS and the stored O
 * are bf16 operands (unit roundoff u) and everything else is exact.  Each
 * rounding is an independent relative error of at most u, so an output's
 * error is a sum of independent terms whose size is u times the root of the
 * summed squares of what each rounding multiplies (probabilistic rounding-
 * error analysis).  With
 *   w2_i  = sum_d dO_id^2 (O_id^2 + sum_j P_ij^2 V_jd^2)   (Delta_i from a rounded O)
 * the squared terms are (two roundings touch each dS_ij: P and dS itself)
 *   eq2_id  = scale^2 (2 sum_j dS_ij^2 K_jd^2 + (sum_j P_ij K_jd)^2 w2_i)
 *   ek2_jd += scale^2 sum_i Q_id^2 (2 dS_ij^2 + P_ij^2 w2_i)
 *   ev2_jd += sum_i P_ij^2 dO_id^2
 * (a row's Delta error is common to all its dS entries, hence the squared
 * sum in eq2).  The caller takes square roots.  P and dS are the head's
 * T x T matrices. */
static void head_err_terms(cview q, cview k, cview v, cview dout, cview o, long T, long D, double scale,
                           const double* P, const double* dS, double* w2, mview eq2, mview ek2, mview ev2) {
    long i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < T; ++i) {
        double w = 0.0;
        for (long d = 0; d < D; ++d) {
            double pv = 0.0;
            for (long j = 0; j < T; ++j) {
                double x = P[i * T + j] * v.base[j * v.rs + d];
                pv += x * x;
            }
            double g = dout.base[i * dout.rs + d], od = o.base[i * o.rs + d];
            w += g * g * (od * od + pv);
        }
        w2[i] = w;
        for (long d = 0; d < D; ++d) {
            double ss = 0.0, pk = 0.0;
            for (long j = 0; j < T; ++j) {
                double kd = k.base[j * k.rs + d];
                ss += dS[i * T + j] * dS[i * T + j] * kd * kd;
                pk += P[i * T + j] * kd;
            }
            eq2.base[i * eq2.rs + d] = scale * scale * (2.0 * ss + pk * pk * w);
        }
    }
    long j;
#pragma omp parallel for schedule(static)
    for (j = 0; j < T; ++j) {
        for (long d = 0; d < D; ++d) {
            double ak = 0.0, av = 0.0;
            for (long i2 = 0; i2 < T; ++i2) {
                double qd = q.base[i2 * q.rs + d], gd = dout.base[i2 * dout.rs + d];
                double p = P[i2 * T + j], ds = dS[i2 * T + j];
                ak += qd * qd * (2.0 * ds * ds + p * p * w2[i2]);
                av += p * p * gd * gd;
            }
            ek2.base[j * ek2.rs + d] += scale * scale * ak;
            ev2.base[j * ev2.rs + d] += av;
        }
    }
}

static int check_shape(long Hq, long Hkv, long D) {
    if (Hq < 1 || Hkv < 1 || D < 1) return 2;
    if (Hq % Hkv) return 2;
    return 0;
}

/* ---------------------------------------------------------------- dense */
/* q,o,dout,dq: [B,Hq,T,D]; k,v,dk,dv: [B,Hkv,T,D]; lse, delta: [B,Hq,T]. */

int oracle_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
               long B, long Hq, long Hkv, long T, long D, int causal, double scale) {
    int st = check_shape(Hq, Hkv, D);
    if (st || B < 0 || T < 0) return st ? st : 2;
    if (B == 0 || T == 0) return 0;
    long G = Hq / Hkv;
    double* P = (double*)malloc(sizeof(double) * T * T);
    if (!P) return 10;
    for (long b = 0; b < B; ++b)
        for (long h = 0; h < Hq; ++h) {
            long g = kv_head(h, G, Hkv);
            cview qh = {q + (b * Hq + h) * T * D, D};
            cview kh = {k + (b * Hkv + g) * T * D, D};
            cview vh = {v + (b * Hkv + g) * T * D, D};
            mview oh = {o + (b * Hq + h) * T * D, D};
            head_fwd(qh, kh, vh, T, D, causal, scale, oh, lse + (b * Hq + h) * T, P);
        }
    free(P);
    return 0;
}

/* o, lse, delta are outputs too (may be NULL).  edq, edk, edv (all or none):
 * the squared rounding-error terms of head_err_terms, laid out like dq, dk, dv. */
int oracle_bwd(const double* q, const double* k, const double* v, const double* dout,
               double* dq, double* dk, double* dv, double* o, double* lse, double* delta,
               double* edq, double* edk, double* edv,
               long B, long Hq, long Hkv, long T, long D, int causal, double scale) {
    int st = check_shape(Hq, Hkv, D);
    if (st || B < 0 || T < 0) return st ? st : 2;
    if (B == 0 || T == 0) return 0;
    long G = Hq / Hkv;
    double* P = (double*)malloc(sizeof(double) * T * T);
    double* dS = (double*)malloc(sizeof(double) * T * T);
    double* lse_tmp = (double*)malloc(sizeof(double) * T);
    double* delta_tmp = (double*)malloc(sizeof(double) * T);
    double* o_tmp = (double*)malloc(sizeof(double) * T * D);
    if (!P || !dS || !lse_tmp || !delta_tmp || !o_tmp) {
        free(P); free(dS); free(lse_tmp); free(delta_tmp); free(o_tmp);
        return 10;
    }
    memset(dk, 0, sizeof(double) * B * Hkv * T * D);
    memset(dv, 0, sizeof(double) * B * Hkv * T * D);
    double* E = NULL;
    if (edq) {
        memset(edk, 0, sizeof(double) * B * Hkv * T * D);
        memset(edv, 0, sizeof(double) * B * Hkv * T * D);
        E = (double*)malloc(sizeof(double) * T * T);
        if (!E) { free(P); free(dS); free(lse_tmp); free(delta_tmp); free(o_tmp); return 10; }
    }
    for (long b = 0; b < B; ++b)
        for (long h = 0; h < Hq; ++h) {
            long g = kv_head(h, G, Hkv);
            cview qh = {q + (b * Hq + h) * T * D, D};
            cview kh = {k + (b * Hkv + g) * T * D, D};
            cview vh = {v + (b * Hkv + g) * T * D, D};
            cview doh = {dout + (b * Hq + h) * T * D, D};
            mview dqh = {dq + (b * Hq + h) * T * D, D};
            mview dkh = {dk + (b * Hkv + g) * T * D, D};
            mview dvh = {dv + (b * Hkv + g) * T * D, D};
            mview oh = {o ? o + (b * Hq + h) * T * D : o_tmp, D};
            double* lr = lse ? lse + (b * Hq + h) * T : lse_tmp;
            double* dr = delta ? delta + (b * Hq + h) * T : delta_tmp;
            head_bwd(qh, kh, vh, doh, T, D, causal, scale, dqh, dkh, dvh, P, dS, lr, dr, oh);
            if (E) {
                cview oc = {oh.base, oh.rs};
                mview eq = {edq + (b * Hq + h) * T * D, D};
                mview ek = {edk + (b * Hkv + g) * T * D, D};
                mview ev = {edv + (b * Hkv + g) * T * D, D};
                head_err_terms(qh, kh, vh, doh, oc, T, D, scale, P, dS, E, eq, ek, ev);
            }
        }
    free(P); free(dS); free(lse_tmp); free(delta_tmp); free(o_tmp); free(E);
    return 0;
}

/* ------------------------------------------------------ variable length */
/* Packed layout: q,o,dout,dq [total,Hq,D]; k,v,dk,dv [total,Hkv,D];
 * lse, delta [Hq,total].  cu_seqlens: host int32 [num_seqs+1], cu[0] = 0,
 * non-decreasing, cu[num_seqs] = total.  Each slice [cu[s], cu[s+1]) is an
 * independent causal problem. */

static int check_cu(const int* cu, long num_seqs, long total) {
    if (num_seqs < 0 || total < 0) return 2;
    if (num_seqs == 0) return total == 0 ? 0 : 5;
    if (cu[0] != 0) return 5;
    for (long s = 0; s < num_seqs; ++s) if (cu[s + 1] < cu[s]) return 5;
    if (cu[num_seqs] != total) return 5;
    return 0;
}

static long max_len(const int* cu, long num_seqs) {
    long m = 0;
    for (long s = 0; s < num_seqs; ++s) if (cu[s + 1] - cu[s] > m) m = cu[s + 1] - cu[s];
    return m;
}

int oracle_varlen_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                      const int* cu, long num_seqs, long total, long Hq, long Hkv, long D,
                      int causal, double scale) {
    int st = check_shape(Hq, Hkv, D);
    if (st) return st;
    if ((st = check_cu(cu, num_seqs, total))) return st;
    long G = Hq / Hkv, L = max_len(cu, num_seqs);
    if (L == 0) return 0;
    double* P = (double*)malloc(sizeof(double) * L * L);
    if (!P) return 10;
    for (long s = 0; s < num_seqs; ++s) {
        long off = cu[s], T = cu[s + 1] - cu[s];
        if (T == 0) continue;
        for (long h = 0; h < Hq; ++h) {
            long g = kv_head(h, G, Hkv);
            cview qh = {q + (off * Hq + h) * D, Hq * D};
            cview kh = {k + (off * Hkv + g) * D, Hkv * D};
            cview vh = {v + (off * Hkv + g) * D, Hkv * D};
            mview oh = {o + (off * Hq + h) * D, Hq * D};
            head_fwd(qh, kh, vh, T, D, causal, scale, oh, lse + h * total + off, P);
        }
    }
    free(P);
    return 0;
}

int oracle_varlen_bwd(const double* q, const double* k, const double* v, const double* dout,
                      double* dq, double* dk, double* dv, double* o, double* lse, double* delta,
                      double* edq, double* edk, double* edv, const int* cu, long num_seqs, long total, long Hq, long Hkv, long D,
                      int causal, double scale) {
    int st = check_shape(Hq, Hkv, D);
    if (st) return st;
    if ((st = check_cu(cu, num_seqs, total))) return st;
    long G = Hq / Hkv, L = max_len(cu, num_seqs);
    memset(dk, 0, sizeof(double) * total * Hkv * D);
    memset(dv, 0, sizeof(double) * total * Hkv * D);
    if (edq) {
        memset(edk, 0, sizeof(double) * total * Hkv * D);
        memset(edv, 0, sizeof(double) * total * Hkv * D);
    }
    if (L == 0) return 0;
    double* P = (double*)malloc(sizeof(double) * L * L);
    double* dS = (double*)malloc(sizeof(double) * L * L);
    double* lse_tmp = (double*)malloc(sizeof(double) * L);
    double* delta_tmp = (double*)malloc(sizeof(double) * L);
    double* o_tmp = (double*)malloc(sizeof(double) * L * D);
    if (!P || !dS || !lse_tmp || !delta_tmp || !o_tmp) {
        free(P); free(dS); free(lse_tmp); free(delta_tmp); free(o_tmp);
        return 10;
    }
    double* E = NULL;
    if (edq && !(E = (double*)malloc(sizeof(double) * L * L))) {
        free(P); free(dS); free(lse_tmp); free(delta_tmp); free(o_tmp);
        return 10;
    }
    for (long s = 0; s < num_seqs; ++s) {
        long off = cu[s], T = cu[s + 1] - cu[s];
        if (T == 0) continue;
        for (long h = 0; h < Hq; ++h) {
            long g = kv_head(h, G, Hkv);
            cview qh = {q + (off * Hq + h) * D, Hq * D};
            cview kh = {k + (off * Hkv + g) * D, Hkv * D};
            cview vh = {v + (off * Hkv + g) * D, Hkv * D};
            cview doh = {dout + (off * Hq + h) * D, Hq * D};
            mview dqh = {dq + (off * Hq + h) * D, Hq * D};
            mview dkh = {dk + (off * Hkv + g) * D, Hkv * D};
            mview dvh = {dv + (off * Hkv + g) * D, Hkv * D};
            mview oh = {o ? o + (off * Hq + h) * D : o_tmp, o ? Hq * D : D};
            double* lr = lse ? lse + h * total + off : lse_tmp;
            double* dr = delta ? delta + h * total + off : delta_tmp;
            head_bwd(qh, kh, vh, doh, T, D, causal, scale, dqh, dkh, dvh, P, dS, lr, dr, oh);
            if (E) {
                cview oc = {oh.base, oh.rs};
                mview eq = {edq + (off * Hq + h) * D, Hq * D};
                mview ek = {edk + (off * Hkv + g) * D, Hkv * D};
                mview ev = {edv + (off * Hkv + g) * D, Hkv * D};
                head_err_terms(qh, kh, vh, doh, oc, T, D, scale, P, dS, E, eq, ek, ev);
            }
        }
    }
    free(P); free(dS); free(lse_tmp); free(delta_tmp); free(o_tmp); free(E);
    return 0;
}

/* ------------------------------------------------- decode over a KV cache */
/* Cached attention (the "cached GQA" / per-row-prefix cached attention of the
 * microLLM-rocm README, section "Why this project exists"): row b holds
 * cache_lens[b] keys; its Tq queries are the newest Tq positions, so query t
 * sits at absolute position len_b - Tq + t and sees keys j <= that position
 * (the causal mask aligned to the end of the cache).
 * q, o [B,Hq,Tq,D]; k_cache, v_cache [B,Hkv,S,D] (S = cache capacity);
 * lse [B,Hq,Tq]; lens: host int32 [B], Tq <= lens[b] <= S. */
int oracle_decode_fwd(const double* q, const double* k, const double* v, const int* lens, double* o, double* lse,
                      long B, long Hq, long Hkv, long Tq, long S, long D, double scale) {
    int st = check_shape(Hq, Hkv, D);
    if (st || B < 0 || Tq < 1 || S < 1) return st ? st : 2;
    for (long b = 0; b < B; ++b)
        if (lens[b] < Tq || lens[b] > S) return 5;
    long G = Hq / Hkv;
    double* row = (double*)malloc(sizeof(double) * S);
    if (!row) return 10;
    for (long b = 0; b < B; ++b)
        for (long h = 0; h < Hq; ++h) {
            long g = kv_head(h, G, Hkv), len = lens[b];
            const double* kh = k + (b * Hkv + g) * S * D;
            const double* vh = v + (b * Hkv + g) * S * D;
            for (long t = 0; t < Tq; ++t) {
                const double* qr = q + ((b * Hq + h) * Tq + t) * D;
                long last = len - Tq + t;               /* newest visible key */
                double m = -INFINITY;
                for (long j = 0; j <= last; ++j) {
                    double acc = 0.0;
                    for (long d = 0; d < D; ++d) acc += qr[d] * kh[j * D + d];
                    row[j] = scale * acc;
                    if (row[j] > m) m = row[j];
                }
                double sum = 0.0;
                for (long j = 0; j <= last; ++j) sum += exp(row[j] - m);
                double l = m + log(sum);
                lse[(b * Hq + h) * Tq + t] = l;
                double* orow = o + ((b * Hq + h) * Tq + t) * D;
                for (long d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (long j = 0; j <= last; ++j) acc += exp(row[j] - l) * vh[j * D + d];
                    orow[d] = acc;
                }
            }
        }
    free(row);
    return 0;
}

int oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
