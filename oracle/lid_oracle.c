/*
 * lid_oracle.c -- plain fp64 CPU oracle of the lightning-indexer top-k.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load this file's library. It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes (DeepSeek-V4-Flash lightning indexer, as described on
 *  - "Eval bug: DeepSeek-V4-Flash lightning-indexer materialises a
 *    ctx-proportional (4 GiB/layer) score buffer" (llama.cpp issue 25468),
 *    root-cause comment: the chain lid_kq = mul_mat(indexer_k, indexer_q)
 *    -> relu -> * weights -> sum_rows -> lid_score -> + mask -> lid_top_k,
 *    which keeps the top 512 keys per query;
 *  - "deepseek v4 support" (llama.cpp PR 22378), the commit that reverts
 *    collapse-Q: per query, top_k(sum_h relu(kv . indexer_q) * index_weights);
 *  - fairydreaming/llama.cpp PR 2, the note on the API change: the scale
 *    factors are gone and an f16 mask is added):
 *
 *   I[t,s] = sum_h w[t,h] * max(0, sum_d q[t,h,d] * k[s,d])  +  mask[t,s]
 *
 * and, per query t, the k keys of largest I[t,.].
 *
 * Every step is the plain definition, in this order, in fp64:
 *   1. decode bf16 (bits << 16 as an IEEE binary32) or f16 (IEEE 754
 *      binary16, decoded below from its definition) inputs to double;
 *   2. dot_h = sum over d in increasing order; I = sum over h in increasing
 *      order of w * max(0, dot_h); score = I + mask;
 *   3. sort all n_kv pairs (score, s) by score descending, ties by s
 *      ascending (+0 and -0 compare equal; -inf is an ordinary value);
 *   4. emit the first min(top_k, n_kv) pairs, pad the rest with (-1, -inf).
 * The readings behind steps 3 and 4 (tie order, padding, output order) are
 * not fixed by the pages; they are this project's stated choices.
 *
 * The same steps take quantised operands too (lid_oracle_topk_e4m3): E4M3
 * codes with one scale per row, decoded from the format's definition below
 * and multiplied by their scale in step 1.
 *
 * Parallelism: OpenMP over blocks of keys for the scores, then over rows for
 * the sorts. Nothing is blocked, fused or reordered beyond that.
 *
 * lid_oracle_sparse_attn (below) is the plain definition of the consumer of
 * the selection: softmax attention of each query head over its selected
 * latent rows.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16: the upper half of an IEEE binary32. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24); /* subnormal: m * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(m + 1024), e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

static double decode(uint16_t b, int is_f16) {
    return is_f16 ? f16_to_double(b) : bf16_to_double(b);
}

/*
 * OCP 8-bit floating point, E4M3 (the "fn" variant, without infinities):
 * 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits. Exponent field 0 is
 * subnormal, (m / 8) * 2^-6; S.1111.111 is NaN; every other code is the
 * finite value (1 + m / 8) * 2^(e - 7), the largest being 448.
 */
static double e4m3_to_double(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);      /* m/8 * 2^-6 */
    else
        v = ldexp((double)(m + 8), e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/*
 * The operands of a call. In the 16-bit form q and k hold bf16 or f16 bits.
 * In the 8-bit form q8 and k8 hold E4M3 codes and each element's value is its
 * row's scale times the code's value: q[t,h,d] = q_scale[t,h] * e4m3(q8[t,h,d])
 * and k[s,d] = k_scale[s] * e4m3(k8[s,d]).
 */
typedef struct {
    const uint16_t *q, *k;
    int is_f16;
    const uint8_t *q8, *k8;
    const float *q_scale, *k_scale;
} operands_t;

static double q_value(const operands_t *o, int64_t t, int H, int D, int64_t i) {
    if (o->q8) return (double)o->q_scale[t * H + i / D] * e4m3_to_double(o->q8[t * H * D + i]);
    return decode(o->q[t * H * D + i], o->is_f16);
}

static double k_value(const operands_t *o, int64_t s, int D, int d) {
    if (o->k8) return (double)o->k_scale[s] * e4m3_to_double(o->k8[s * D + d]);
    return decode(o->k[s * D + d], o->is_f16);
}

/*
 * fp64 scores of the listed query rows over keys [0, n_kv):
 * out[r * n_kv + s] = I[rows[r], s] + mask[rows[r], s].
 * q: [n_q][H][D], k: [n_kv][D] (see operands_t), w: [n_q][H] f32,
 * mask: [n_q][n_kv] f16 bits or NULL (all zero).
 * OpenMP splits the keys into blocks; every block takes every listed row.
 */
#define KEY_BLOCK 512
static int rows_scores(const operands_t *o, const float *w, const uint16_t *mask,
                       int64_t n_kv, int H, int D, const int64_t *rows, int64_t n_rows,
                       double *out) {
    double *qd = (double *)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1) * H * D);
    if (!qd) return 2;
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t i = 0; i < (int64_t)H * D; ++i)
            qd[r * H * D + i] = q_value(o, rows[r], H, D, i);
    int64_t n_blk = (n_kv + KEY_BLOCK - 1) / KEY_BLOCK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t b = 0; b < n_blk; ++b) {
        double krow[256];
        int64_t s_end = (b + 1) * KEY_BLOCK < n_kv ? (b + 1) * KEY_BLOCK : n_kv;
        for (int64_t s = b * KEY_BLOCK; s < s_end; ++s) {
            for (int d = 0; d < D; ++d) krow[d] = k_value(o, s, D, d);
            for (int64_t r = 0; r < n_rows; ++r) {
                int64_t t = rows[r];
                double I = 0.0;
                for (int h = 0; h < H; ++h) {
                    const double *qh = qd + (r * H + h) * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += qh[d] * krow[d];
                    double relu = dot > 0.0 ? dot : 0.0;
                    I += (double)w[t * H + h] * relu;
                }
                double m = mask ? f16_to_double(mask[t * n_kv + s]) : 0.0;
                out[r * n_kv + s] = I + m;
            }
        }
    }
    free(qd);
    return 0;
}

typedef struct {
    double score;
    int64_t idx;
} pair_t;

/* score descending, then index ascending (+0 == -0 under double compare) */
static int cmp_pair(const void *a, const void *b) {
    const pair_t *x = (const pair_t *)a, *y = (const pair_t *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

static int check_args(const void *q, const void *k, const float *w,
                      int64_t n_q, int64_t n_kv, int H, int D,
                      const int64_t *rows, int64_t n_rows) {
    if (!q || !k || !w || (!rows && n_rows > 0) || H <= 0 || D <= 0 || D > 256 ||
        n_kv < 0 || n_rows < 0)
        return 1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= n_q) return 1;
    return 0;
}

/*
 * Full fp64 score rows for the listed queries.
 * rows: int64 query indices (n_rows of them); out: [n_rows][n_kv] doubles.
 * Returns 0 on success, 1 on bad arguments, 2 when out of host memory.
 */
int lid_oracle_scores(const uint16_t *q, const uint16_t *k, const float *w,
                      const uint16_t *mask, int64_t n_q, int64_t n_kv, int H,
                      int D, int is_f16, const int64_t *rows, int64_t n_rows,
                      double *out) {
    if (check_args(q, k, w, n_q, n_kv, H, D, rows, n_rows) || !out) return 1;
    operands_t o = {q, k, is_f16, NULL, NULL, NULL, NULL};
    return rows_scores(&o, w, mask, n_kv, H, D, rows, n_rows, out);
}

/*
 * Top-k of the listed queries: the first min(top_k, n_kv) entries of each
 * row's full (score desc, index asc) order, then (-1, -inf) padding.
 * out_idx: [n_rows][top_k] int64, out_score: [n_rows][top_k] doubles.
 * Rows are processed in batches so that the fp64 rows held at once stay
 * within about 256 MB. Returns 0 / 1 (bad arguments) / 2 (out of memory).
 */
static int rows_topk(const operands_t *o, const float *w, const uint16_t *mask,
                     int64_t n_kv, int H, int D, int top_k, const int64_t *rows,
                     int64_t n_rows, int64_t *out_idx, double *out_score) {
    int64_t row_cap = n_kv > 0 ? (int64_t)(32 << 20) / n_kv : n_rows;
    if (row_cap < 1) row_cap = 1;
    if (row_cap > n_rows) row_cap = n_rows > 0 ? n_rows : 1;
    double *sc = (double *)malloc(sizeof(double) * (size_t)row_cap * (size_t)(n_kv > 0 ? n_kv : 1));
    if (!sc) return 2;
    int bad = 0;
    for (int64_t r0 = 0; r0 < n_rows && !bad; r0 += row_cap) {
        int64_t nr = n_rows - r0 < row_cap ? n_rows - r0 : row_cap;
        if (rows_scores(o, w, mask, n_kv, H, D, rows + r0, nr, sc)) {
            bad = 2;
            break;
        }
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t r = 0; r < nr; ++r) {
            pair_t *pairs = (pair_t *)malloc(sizeof(pair_t) * (size_t)(n_kv > 0 ? n_kv : 1));
            if (!pairs) {
#pragma omp atomic write
                bad = 2;
                continue;
            }
            for (int64_t s = 0; s < n_kv; ++s) {
                pairs[s].score = sc[r * n_kv + s];
                pairs[s].idx = s;
            }
            qsort(pairs, (size_t)n_kv, sizeof(pair_t), cmp_pair);
            int64_t o = (r0 + r) * top_k;
            for (int j = 0; j < top_k; ++j) {
                if (j < n_kv) {
                    out_idx[o + j] = pairs[j].idx;
                    out_score[o + j] = pairs[j].score;
                } else {
                    out_idx[o + j] = -1;
                    out_score[o + j] = -INFINITY;
                }
            }
            free(pairs);
        }
    }
    free(sc);
    return bad;
}

int lid_oracle_topk(const uint16_t *q, const uint16_t *k, const float *w,
                    const uint16_t *mask, int64_t n_q, int64_t n_kv, int H,
                    int D, int top_k, int is_f16, const int64_t *rows,
                    int64_t n_rows, int64_t *out_idx, double *out_score) {
    if (check_args(q, k, w, n_q, n_kv, H, D, rows, n_rows) || !out_idx ||
        !out_score || top_k <= 0)
        return 1;
    operands_t o = {q, k, is_f16, NULL, NULL, NULL, NULL};
    return rows_topk(&o, w, mask, n_kv, H, D, top_k, rows, n_rows, out_idx, out_score);
}

/*
 * The 8-bit form of the two calls above: q8 [n_q][H][D] and k8 [n_kv][D]
 * E4M3 codes, q_scale [n_q][H] and k_scale [n_kv] f32; element values are
 * scale * e4m3(code) (operands_t), everything else as in the 16-bit form.
 * This is the indexer with quantised operands. Sources: "llama.cpp DeepSeek
 * v4 Flash experimental inference", section "Plan: Implement CUDA Kernels for
 * DeepSeek v4 (DSV4) Operations", kernel 3 (dsv4_fp8_kv_quantize: rows
 * quantised to E4M3 against their amax); "deepseek v4 support" (llama.cpp PR
 * 22378), the batched-prefill commit (the indexer's queries are quantised on
 * its scoring path). The score is the same formula on the dequantised values.
 */
int lid_oracle_scores_e4m3(const uint8_t *q8, const float *q_scale, const uint8_t *k8,
                           const float *k_scale, const float *w, const uint16_t *mask,
                           int64_t n_q, int64_t n_kv, int H, int D, const int64_t *rows,
                           int64_t n_rows, double *out) {
    if (check_args(q8, k8, w, n_q, n_kv, H, D, rows, n_rows) || !out || !q_scale || !k_scale)
        return 1;
    operands_t o = {NULL, NULL, 0, q8, k8, q_scale, k_scale};
    return rows_scores(&o, w, mask, n_kv, H, D, rows, n_rows, out);
}

int lid_oracle_topk_e4m3(const uint8_t *q8, const float *q_scale, const uint8_t *k8,
                         const float *k_scale, const float *w, const uint16_t *mask,
                         int64_t n_q, int64_t n_kv, int H, int D, int top_k,
                         const int64_t *rows, int64_t n_rows, int64_t *out_idx,
                         double *out_score) {
    if (check_args(q8, k8, w, n_q, n_kv, H, D, rows, n_rows) || !out_idx || !out_score ||
        !q_scale || !k_scale || top_k <= 0)
        return 1;
    operands_t o = {NULL, NULL, 0, q8, k8, q_scale, k_scale};
    return rows_topk(&o, w, mask, n_kv, H, D, top_k, rows, n_rows, out_idx, out_score);
}

/*
 * Sparse attention over the selected keys (the consumer of the top-k):
 * "Eval bug: DeepSeek-V4-Flash lightning-indexer ..." (llama.cpp issue 25468),
 * root-cause comment: the top-512 selection feeds the CSA layers' attention;
 * "deepseek v4 support" (llama.cpp PR 22378), the batched-prefill commit:
 * Q*K^T -> softmax -> *V over the V4 MLA latent KV (K[0] = 512), where slots
 * masked to -INFINITY contribute zero to softmax/V.
 *
 * For each row t and head h, with J = { j : 0 <= idx[t,j] < n_kv and the
 * selection's score (if given) is not -inf }:
 *   s_j = sum_d qa[t,h,d] * kv[idx[t,j],d]          (increasing d)
 *   m = max_j scale * s_j,  e_j = exp(scale * s_j - m),  Z = sum_j e_j
 *   out[t,h,d] = sum_j (e_j / Z) * kv[idx[t,j],d]     (increasing j)
 *   lse[t,h] = m + log(Z)
 * and out = 0, lse = -inf when J is empty. Keys and values are the same
 * latent rows. Everything in fp64; OpenMP over rows.
 */
int lid_oracle_sparse_attn(const uint16_t *qa, const uint16_t *kv, const int32_t *idx, const float *sel_score,
                           int64_t n_q, int64_t n_kv, int Ha, int Dc, int top_k, int is_f16, double scale,
                           const int64_t *rows, int64_t n_rows, double *out, double *lse) {
    if (!qa || !idx || !rows || !out || !lse || n_q < 0 || n_kv < 0 || Ha <= 0 || Dc <= 0 || top_k <= 0)
        return 1;
    if (n_kv > 0 && !kv) return 1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= n_q) return 2;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t t = rows[r];
        int64_t *sel = (int64_t *)malloc(sizeof(int64_t) * (size_t)top_k);
        double *e = (double *)malloc(sizeof(double) * (size_t)top_k);
        if (!sel || !e) {
            free(sel);
            free(e);
#pragma omp atomic write
            err = 3;
            continue;
        }
        int nj = 0;
        for (int j = 0; j < top_k; ++j) {
            const int64_t s = idx[t * top_k + j];
            if (s < 0 || s >= n_kv) continue;
            if (sel_score && sel_score[t * top_k + j] == -INFINITY) continue;
            sel[nj++] = s;
        }
        for (int h = 0; h < Ha; ++h) {
            double *o = out + (r * Ha + h) * (int64_t)Dc;
            for (int d = 0; d < Dc; ++d) o[d] = 0.0;
            if (nj == 0) {
                lse[r * Ha + h] = -INFINITY;
                continue;
            }
            const uint16_t *qrow = qa + (t * Ha + h) * (int64_t)Dc;
            double m = -INFINITY;
            for (int j = 0; j < nj; ++j) {
                const uint16_t *krow = kv + sel[j] * (int64_t)Dc;
                double sj = 0.0;
                for (int d = 0; d < Dc; ++d) sj += decode(qrow[d], is_f16) * decode(krow[d], is_f16);
                e[j] = scale * sj;
                if (e[j] > m) m = e[j];
            }
            double z = 0.0;
            for (int j = 0; j < nj; ++j) {
                e[j] = exp(e[j] - m);
                z += e[j];
            }
            for (int j = 0; j < nj; ++j) {
                const uint16_t *vrow = kv + sel[j] * (int64_t)Dc;
                const double pj = e[j] / z;
                for (int d = 0; d < Dc; ++d) o[d] += pj * decode(vrow[d], is_f16);
            }
            lse[r * Ha + h] = m + log(z);
        }
        free(sel);
        free(e);
    }
    return err;
}

/* Decoders exposed so tests can pin them against library conversions. */
double lid_oracle_decode_bf16(uint16_t b) { return bf16_to_double(b); }
double lid_oracle_decode_f16(uint16_t b) { return f16_to_double(b); }
double lid_oracle_decode_e4m3(uint8_t b) { return e4m3_to_double(b); }

int lid_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
