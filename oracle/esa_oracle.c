/*
 * CPU oracle for gated fine-grained sparse attention — TEST INFRASTRUCTURE.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this code. It is deliberately plain and slow: every quantity follows
 * its definition on the pages, in 64-bit integers or fp64, with no tiling,
 * no fusion and no reordering.
 *
 * Sources (the pages this follows):
 *  - "超大规模MoE架构中稀疏注意力机制的演进与实践" (Gated DSA), section 二.1
 *    (Indexer + Top-K: an indexer scores the query against every history
 *    position, the K best positions go on to full attention), section 二.2
 *    (the indexer uses no RoPE), section 二.3 and the pseudo-code of section
 *    四.1 (matmul scores, top-k, gather, scaled dot-product attention, then
 *    final = g*attn + (1-g)*linear_output).
 *  - "混合注意力架构演进：从线性注意力到稀疏门控的技术权衡", section 三
 *    (sparse_attention: indexer_score, topk, gather, softmax(Q K_sel^T/sqrt(d)) V_sel).
 *  - "Elastic Attention：动态路由优化大模型长文本处理", sections 2.2 and 3.1
 *    (per-head routing: a head runs either full or sparse attention).
 *  - The linear branch: the Gated DSA page, sections 一, 二.3 and 三, names it
 *    KDA, a gated linear attention kept in most layers that folds the history
 *    into a recurrent state, and mixes its output with the sparse attention
 *    output; the page prints no formula, so oracle_kda follows the published
 *    Kimi Delta Attention recurrence (a delta-rule state update with one
 *    forgetting factor per key channel).
 *
 * Readings taken where the pages are silent (each is restated in the tests):
 *  the prefix of query position p is keys 0..p inclusive; the indexer is a
 *  plain weighted sum over indexer heads of int8 dot products (no
 *  nonlinearity; a ReLU per indexer head is an option), with one indexer key
 *  per position shared by all indexer heads; per-head index sets (an option)
 *  score each indexer head alone, unweighted, and query head h attends to
 *  the set of indexer head h / (Hq/H_I); ties in the score go to the lower position; the index set is
 *  returned in ascending position order, padded with -1, with
 *  cnt = min(K, p+1); one index set per (sequence, query) is shared by every
 *  query head; the gate is one value in (0,1) per query head; heads routed to
 *  full attention output the attention result without the gate mix; query
 *  head h reads key/value head floor(h / (Hq/Hkv)).
 *
 * Parity pins: every function here is pinned by the CPU tests against brute
 * force, closed forms, invariants and library routines (numpy, torch).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> exact double */
static double bf16_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* int8 dot product of indexer head h of query row (b, t) with the indexer
 * key at position j, in int64 */
static int64_t indexer_dot(const int8_t *qI, const int8_t *kI, long Tq, long Tk, int H_I, int D_I,
                           long b, long t, int h, long j) {
    int64_t dot = 0;
    for (int c = 0; c < D_I; c++) {
        int64_t a = qI[((b * Tq + t) * H_I + h) * D_I + c];
        int64_t k = kI[(b * Tk + j) * D_I + c];
        dot += a * k;
    }
    return dot;
}

/*
 * Indexer scores of query row (b, t) against keys 0..p, p = q_offset + t,
 * in int64 (no RoPE anywhere):
 *   head < 0 (one index set per query, the Gated DSA indexer):
 *       s_j = sum_h w_h * f(sum_c qI[b,t,h,c] * kI[b,j,c])
 *   head >= 0 (one index set per indexer head: the per-head [batch, heads,
 *   top_k] index shape of the Gated DSA pseudo-code, which scores each head's
 *   query against the shared history keys without weights):
 *       s_j = f(sum_c qI[b,t,head,c] * kI[b,j,c])
 * where f is the identity, or f(x) = max(x, 0) when relu is set (a ReLU on
 * each indexer head's dot product before the weighted sum).
 * Writes p+1 scores; returns p+1, or -1 when a score does not fit in int32
 * (the interface promises int32 scores).
 */
long oracle_indexer_row_mode(const int8_t *qI, const int8_t *kI, const int32_t *wI,
                             long B, long Tq, long Tk, long q_offset, int H_I, int D_I,
                             long b, long t, int relu, int head, int32_t *scores) {
    (void)B;
    long p = q_offset + t;
    long n = p + 1;
    if (n > Tk) return -2;
    for (long j = 0; j < n; j++) {
        int64_t s = 0;
        for (int h = 0; h < H_I; h++) {
            if (head >= 0 && h != head) continue;
            int64_t dot = indexer_dot(qI, kI, Tq, Tk, H_I, D_I, b, t, h, j);
            if (relu && dot < 0) dot = 0;
            if (head >= 0) s += dot;
            else s += (int64_t)wI[h] * dot;
        }
        if (s > INT32_MAX || s < INT32_MIN) return -1;
        scores[j] = (int32_t)s;
    }
    return n;
}

/* The Gated DSA indexer: weighted sum over heads, no nonlinearity. */
long oracle_indexer_row(const int8_t *qI, const int8_t *kI, const int32_t *wI,
                        long B, long Tq, long Tk, long q_offset, int H_I, int D_I,
                        long b, long t, int32_t *scores) {
    return oracle_indexer_row_mode(qI, kI, wI, B, Tq, Tk, q_offset, H_I, D_I, b, t, 0, -1, scores);
}

typedef struct {
    int32_t s;
    int32_t j;
} scored_pos;

/* (score descending, position ascending) */
static int by_score_then_position(const void *x, const void *y) {
    const scored_pos *a = (const scored_pos *)x, *b = (const scored_pos *)y;
    if (a->s != b->s) return (a->s > b->s) ? -1 : 1;
    return (a->j < b->j) ? -1 : (a->j > b->j);
}

static int ascending_i32(const void *x, const void *y) {
    int32_t a = *(const int32_t *)x, b = *(const int32_t *)y;
    return (a < b) ? -1 : (a > b);
}

/*
 * Top-K selection for a list of query rows (flat row id r = b*Tq + t).
 * For each row (and, with per-head sets, each indexer head of it): order
 * positions 0..p by (score descending, position ascending), keep the first
 * min(K, p+1), sort them ascending, pad with -1.
 * flags: bit 0 = ReLU per indexer head, bit 1 = one index set per indexer
 * head (scores as in oracle_indexer_row_mode).
 * idx is [n_rows, K] (or [n_rows, H_I, K] with per-head sets), cnt is
 * [n_rows] (or [n_rows, H_I]). Returns 0, or -1 on int32 overflow.
 */
int oracle_topk_rows_mode(const int8_t *qI, const int8_t *kI, const int32_t *wI,
                          long B, long Tq, long Tk, long q_offset, int H_I, int D_I,
                          int K, int flags, const int64_t *rows, long n_rows,
                          int32_t *idx, int32_t *cnt, int n_threads) {
    const int relu = flags & 1, per_head = (flags >> 1) & 1;
    const int nsets = per_head ? H_I : 1;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (long r = 0; r < n_rows; r++) {
        long b = rows[r] / Tq, t = rows[r] % Tq;
        long n = q_offset + t + 1;
        int32_t *sc = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
        scored_pos *order = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)n);
        for (int set = 0; set < nsets; set++) {
            const long out = r * nsets + set;
            if (oracle_indexer_row_mode(qI, kI, wI, B, Tq, Tk, q_offset, H_I, D_I, b, t, relu, per_head ? set : -1,
                                        sc) != n) {
                bad |= 1;
                continue;
            }
            for (long j = 0; j < n; j++) {
                order[j].s = sc[j];
                order[j].j = (int32_t)j;
            }
            qsort(order, (size_t)n, sizeof(scored_pos), by_score_then_position);
            long kk = n < K ? n : K;
            int32_t *row = idx + out * (long)K;
            for (long i = 0; i < kk; i++) row[i] = order[i].j;
            qsort(row, (size_t)kk, sizeof(int32_t), ascending_i32);
            for (long i = kk; i < K; i++) row[i] = -1;
            cnt[out] = (int32_t)kk;
        }
        free(sc);
        free(order);
    }
    return bad ? -1 : 0;
}

/* The Gated DSA selection: one index set per query row. */
int oracle_topk_rows(const int8_t *qI, const int8_t *kI, const int32_t *wI,
                     long B, long Tq, long Tk, long q_offset, int H_I, int D_I,
                     int K, const int64_t *rows, long n_rows,
                     int32_t *idx, int32_t *cnt, int n_threads) {
    return oracle_topk_rows_mode(qI, kI, wI, B, Tq, Tk, q_offset, H_I, D_I, K, 0, rows, n_rows, idx, cnt, n_threads);
}

/*
 * Attention for a list of query rows, all query heads, in fp64.
 *  - Head h of row (b,t) reads key/value head kh = h / (Hq/Hkv).
 *  - Key set: when route is given and route[b*Hq+h] == 0 (a full head), all
 *    positions 0..p; otherwise the index set of head h: with nsets = 1 the
 *    row's one set idx[r, 0..cnt[r]); with nsets > 1 (one set per indexer
 *    head) the set s = h / (Hq/nsets), idx[r, s, 0..cnt[r, s]).
 *  - logit_j = scale * sum_c q[b,t,h,c] * k[b,j,kh,c];  m = max logit;
 *    o = sum_j e^(logit_j - m) v[b,j,kh,:] / sum_j e^(logit_j - m);
 *    lse = m + ln sum_j e^(logit_j - m).
 *  - An empty key set (cnt = 0) gives o = 0 and lse = -inf.
 *  - Sparse heads with g given: out = g[h]*o + (1-g[h])*lin[b,t,h,:];
 *    full heads (and sparse heads without g): out = o.
 * q, lin: [B,Tq,Hq,D] bf16 bits; k, v: [B,Tk,Hkv,D] bf16 bits; idx/cnt are
 * per listed row. out [n_rows,Hq,D], lse [n_rows,Hq] (lse may be NULL).
 * Returns 0, or -1 when an index lies outside 0..p.
 */
int oracle_attention_rows_sets(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               const int32_t *idx, const int32_t *cnt, int K, int nsets,
                               long B, long Tq, long Tk, long q_offset,
                               int Hq, int Hkv, int D, double scale,
                               const float *g, const uint16_t *lin, const uint8_t *route,
                               const int64_t *rows, long n_rows,
                               double *out, double *lse, int n_threads) {
    (void)B;
    int bad = 0;
    int G = Hq / Hkv;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (long r = 0; r < n_rows; r++) {
        long b = rows[r] / Tq, t = rows[r] % Tq;
        long p = q_offset + t;
        double *logit = (double *)malloc(sizeof(double) * (size_t)(p + 1));
        int32_t *keys = (int32_t *)malloc(sizeof(int32_t) * (size_t)(p + 1));
        double *acc = (double *)malloc(sizeof(double) * (size_t)D);
        for (int h = 0; h < Hq; h++) {
            int kh = h / G;
            long set = r * nsets + h / (Hq / nsets);  /* the index set of head h */
            int full = (route != NULL) && (route[b * Hq + h] == 0);
            long nk;
            if (full) {
                nk = p + 1;
                for (long j = 0; j < nk; j++) keys[j] = (int32_t)j;
            } else {
                nk = cnt[set];
                for (long i = 0; i < nk; i++) {
                    int32_t j = idx[set * (long)K + i];
                    if (j < 0 || j > p) {
                        bad |= 1;
                        j = 0;
                    }
                    keys[i] = j;
                }
            }
            const uint16_t *qrow = q + ((b * Tq + t) * Hq + h) * (long)D;
            double m = -INFINITY;
            for (long i = 0; i < nk; i++) {
                const uint16_t *krow = k + ((b * Tk + keys[i]) * Hkv + kh) * (long)D;
                double dot = 0.0;
                for (int c = 0; c < D; c++) dot += bf16_to_double(qrow[c]) * bf16_to_double(krow[c]);
                logit[i] = dot * scale;
                if (logit[i] > m) m = logit[i];
            }
            double den = 0.0;
            for (int c = 0; c < D; c++) acc[c] = 0.0;
            for (long i = 0; i < nk; i++) {
                double e = exp(logit[i] - m);
                den += e;
                const uint16_t *vrow = v + ((b * Tk + keys[i]) * Hkv + kh) * (long)D;
                for (int c = 0; c < D; c++) acc[c] += e * bf16_to_double(vrow[c]);
            }
            double *o = out + (r * Hq + h) * (long)D;
            const uint16_t *lrow = lin ? lin + ((b * Tq + t) * Hq + h) * (long)D : NULL;
            for (int c = 0; c < D; c++) {
                /* an empty key set (cnt = 0) attends to nothing: o = 0 */
                double oc = nk > 0 ? acc[c] / den : 0.0;
                if (!full && g != NULL && lrow != NULL) {
                    double gh = (double)g[h];
                    oc = gh * oc + (1.0 - gh) * bf16_to_double(lrow[c]);
                }
                o[c] = oc;
            }
            if (lse) lse[r * Hq + h] = m + log(den);
        }
        free(logit);
        free(keys);
        free(acc);
    }
    return bad ? -1 : 0;
}

/* Attention with one index set per query row (nsets = 1). */
int oracle_attention_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const int32_t *idx, const int32_t *cnt, int K,
                          long B, long Tq, long Tk, long q_offset,
                          int Hq, int Hkv, int D, double scale,
                          const float *g, const uint16_t *lin, const uint8_t *route,
                          const int64_t *rows, long n_rows,
                          double *out, double *lse, int n_threads) {
    return oracle_attention_rows_sets(q, k, v, idx, cnt, K, 1, B, Tq, Tk, q_offset, Hq, Hkv, D, scale, g, lin, route,
                                      rows, n_rows, out, lse, n_threads);
}

/*
 * Attention router (Elastic Attention page, section 2.2: a 2-layer MLP on the
 * current key hidden states decides, per attention head, full or sparse).
 * Reading taken: per sequence b the key states are averaged over the Tk
 * cached positions and concatenated over key/value heads,
 *   x[c] = (1/Tk) sum_j k[b, j, c / D, c % D],      c < Hkv*D,
 * then hid[f] = max(0, b1[f] + sum_c W1[f, c] x[c]) for f < F, and for
 * query head h the logits z_o = b2[2h+o] + sum_f W2[2h+o, f] hid[f]
 * (o = 0: full, o = 1: sparse); route[b, h] = 1 (sparse) iff z_1 >= z_0.
 * W1 fp32 [F, Hkv*D], b1 [F], W2 fp32 [2*Hq, F], b2 [2*Hq]; k bf16 bits.
 * All sums in fp64. margin[b*Hq + h] = z_1 - z_0 (for the test's tie band).
 */
int oracle_route_heads(const uint16_t *k, long B, long Tk, int Hkv, int D, int Hq, int F,
                       const float *W1, const float *b1, const float *W2, const float *b2,
                       uint8_t *route, double *margin) {
    const long C = (long)Hkv * D;
    double *x = (double *)malloc(sizeof(double) * (size_t)C);
    double *hid = (double *)malloc(sizeof(double) * (size_t)F);
    for (long b = 0; b < B; b++) {
        for (long c = 0; c < C; c++) {
            double acc = 0.0;
            for (long j = 0; j < Tk; j++) acc += bf16_to_double(k[(b * Tk + j) * C + c]);
            x[c] = Tk > 0 ? acc / (double)Tk : 0.0;
        }
        for (int f = 0; f < F; f++) {
            double acc = (double)b1[f];
            for (long c = 0; c < C; c++) acc += (double)W1[(long)f * C + c] * x[c];
            hid[f] = acc > 0.0 ? acc : 0.0;
        }
        for (int h = 0; h < Hq; h++) {
            double z[2];
            for (int o = 0; o < 2; o++) {
                double acc = (double)b2[2 * h + o];
                for (int f = 0; f < F; f++) acc += (double)W2[(long)(2 * h + o) * F + f] * hid[f];
                z[o] = acc;
            }
            route[b * Hq + h] = (uint8_t)(z[1] >= z[0] ? 1 : 0);
            if (margin) margin[b * Hq + h] = z[1] - z[0];
        }
    }
    free(x);
    free(hid);
    return 0;
}

/* The linear-attention branch (KDA) whose output is the linear_output of the
 * gate mix. Per sequence b and head h, a state S of Dk x Dv values (row i: key
 * channel i; column c: value channel c) starts from state_in (fp32
 * [B, H, Dk, Dv]) or from zero, and for t = 0 .. T-1:
 *   forget:  S[i][c] *= alpha_t[i]                (one factor per key channel)
 *   read:    u[c]  = sum_i k_t[i] S[i][c]          (what S returns for k_t)
 *   write:   S[i][c] += beta_t k_t[i] (v_t[c] - u[c])   (delta rule)
 *   output:  o_t[c] = scale * sum_i q_t[i] S[i][c]
 * q, k bf16 [B, T, H, Dk]; v bf16 [B, T, H, Dv]; alpha fp32 [B, T, H, Dk];
 * beta fp32 [B, T, H]; o fp64 [B, T, H, Dv]; the final S goes to state_out
 * (fp64 [B, H, Dk, Dv]) when it is not NULL. Returns 0. */
int oracle_kda(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
               const float *state_in, long B, long T, int H, int Dk, int Dv, double scale, double *o,
               double *state_out, int n_threads) {
    const long BH = B * H;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#else
    (void)n_threads;
#endif
    for (long bh = 0; bh < BH; bh++) {
        const long b = bh / H;
        const int h = (int)(bh % H);
        double *S = (double *)malloc(sizeof(double) * (size_t)Dk * (size_t)Dv);
        double *u = (double *)malloc(sizeof(double) * (size_t)Dv);
        for (int i = 0; i < Dk; i++)
            for (int c = 0; c < Dv; c++)
                S[i * Dv + c] = state_in ? (double)state_in[(bh * Dk + i) * Dv + c] : 0.0;
        for (long t = 0; t < T; t++) {
            const long row = (b * T + t) * H + h;
            const uint16_t *kt = k + row * Dk, *qt = q + row * Dk, *vt = v + row * Dv;
            const float *at = alpha + row * Dk;
            const double bt = (double)beta[row];
            for (int i = 0; i < Dk; i++)
                for (int c = 0; c < Dv; c++) S[i * Dv + c] *= (double)at[i];
            for (int c = 0; c < Dv; c++) {
                double acc = 0.0;
                for (int i = 0; i < Dk; i++) acc += bf16_to_double(kt[i]) * S[i * Dv + c];
                u[c] = acc;
            }
            for (int i = 0; i < Dk; i++)
                for (int c = 0; c < Dv; c++)
                    S[i * Dv + c] += bt * bf16_to_double(kt[i]) * (bf16_to_double(vt[c]) - u[c]);
            for (int c = 0; c < Dv; c++) {
                double acc = 0.0;
                for (int i = 0; i < Dk; i++) acc += bf16_to_double(qt[i]) * S[i * Dv + c];
                o[row * Dv + c] = scale * acc;
            }
        }
        if (state_out)
            for (long e = 0; e < (long)Dk * Dv; e++) state_out[bh * Dk * Dv + e] = S[e];
        free(S);
        free(u);
    }
    return 0;
}

/*
 * Threshold form of the index sets of a list of query rows (flat row id
 * r = b*Tq + t; one index set per row, scored as in oracle_indexer_row_mode
 * with head = -1). The top-K set of a row under the tie rule "lower position
 * wins" is described by two integers:
 *   T = the score of the K-th position in (score descending, position
 *       ascending) order, and P = that K-th position itself;
 *   key j <= p is in the set iff s_j > T, or s_j == T and j <= P
 * (the positions scoring T that the set holds are exactly the lowest ones,
 * and the K-th of the order is the last of them). When the prefix holds at
 * most K keys the set is the whole prefix: T = INT32_MIN, P = p. The routed
 * attention (Elastic Attention page, section 3.1: sparse heads inside the
 * fused kernel) rebuilds its sparse heads' sets from this form.
 * flags as in oracle_topk_rows_mode: with per-head sets (bit 1) every
 * indexer head of a row has its own set, scored by that head alone.
 * thr is [n_rows][2] = (T, P), or [n_rows][H_I][2] with per-head sets.
 * Returns 0, or -1 on int32 overflow.
 */
int oracle_threshold_rows(const int8_t *qI, const int8_t *kI, const int32_t *wI,
                          long B, long Tq, long Tk, long q_offset, int H_I, int D_I,
                          int K, int flags, const int64_t *rows, long n_rows,
                          int32_t *thr, int n_threads) {
    const int relu = flags & 1, per_head = (flags >> 1) & 1;
    const int nsets = per_head ? H_I : 1;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (long r = 0; r < n_rows; r++) {
        const long b = rows[r] / Tq, t = rows[r] % Tq;
        const long p = q_offset + t, n = p + 1;  /* keys 0..p */
        for (int set = 0; set < nsets; set++) {
            int32_t *tr = thr + 2 * (r * nsets + set);
            if (n <= K) {
                tr[0] = INT32_MIN;
                tr[1] = (int32_t)p;
                continue;
            }
            int32_t *sc = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
            scored_pos *order = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)n);
            const int scored_head = per_head ? set : -1; /* the set's own head, or the weighted sum */
            if (oracle_indexer_row_mode(qI, kI, wI, B, Tq, Tk, q_offset, H_I, D_I, b, t, relu, scored_head, sc) != n) {
                bad |= 1;
            } else {
                for (long j = 0; j < n; j++) {
                    order[j].s = sc[j];
                    order[j].j = (int32_t)j;
                }
                qsort(order, (size_t)n, sizeof(scored_pos), by_score_then_position);
                const scored_pos kth = order[K - 1];
                tr[0] = kth.s;
                tr[1] = kth.j;
            }
            free(sc);
            free(order);
        }
    }
    return bad ? -1 : 0;
}
