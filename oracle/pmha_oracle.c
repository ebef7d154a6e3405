/*
 * Oracle for edge-packed multi-head attention: plain, slow, fp64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link,
 * load or call this file: only the test suite, the smoke check of the entry
 * module and the CPU-baseline leg of the benchmark use it. It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Source of every formula: the kpnn2 0.3.0 API reference page
 * "PackedMultiheadAttention" (constructor parameter table, the Notes section
 * with its five numbered steps, the forward() Returns table and the Examples),
 * and, for the dense limit, the continuiti "Multi head attention" page
 * (the MultiHead formula) and the PyTorch nn.MultiheadAttention tutorial page
 * ("Three projections in one tensor" and "Example").
 *
 * Every floating-point quantity is double. Loops run in the order the
 * definition states; OpenMP only splits independent output rows across
 * threads, so the arithmetic of each output element is the same whatever the
 * thread count.
 *
 * Parity status: every function here is pinned by tests that do not use this
 * file's arithmetic (torch.nn.MultiheadAttention in float64, a dense -inf
 * masked attention, brute-force loops on tiny inputs, the printed doctest of
 * the kpnn2 page, and softmax invariants). No function is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Status codes of the oracle. They are defined here on their own; tests map
 * them to the library's codes by meaning. */
enum {
    ORACLE_OK = 0,
    ORACLE_ERR_EMPTY = 1,     /* nnz < 1 */
    ORACLE_ERR_RANGE = 2,     /* an index outside [0, features) */
    ORACLE_ERR_DUPLICATE = 3, /* a (source, target) pair given twice */
    ORACLE_ERR_ARG = 4,       /* a size or option the layer rejects */
    ORACLE_ERR_NOMEM = 5
};

/* ------------------------------------------------------------------------ */
/* Index checks and the self-loop append.                                   */
/* kpnn2 PackedMultiheadAttention, parameter table: source_index must lie in */
/* [0, key_features), target_index in [0, query_features), both of length   */
/* nnz >= 1, and no (source, target) pair may repeat. add_self_loops appends */
/* every missing (i, i) after the given pairs and needs                      */
/* query_features == key_features.                                           */
/* ------------------------------------------------------------------------ */

static int cmp_i64(const void *a, const void *b)
{
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x > y) - (x < y);
}

int oracle_validate_edges(const int64_t *source_index, const int64_t *target_index,
                          int64_t nnz, int64_t query_features, int64_t key_features)
{
    if (query_features < 1 || key_features < 1) return ORACLE_ERR_ARG;
    if (nnz < 1) return ORACLE_ERR_EMPTY;
    for (int64_t e = 0; e < nnz; ++e) {
        if (source_index[e] < 0 || source_index[e] >= key_features) return ORACLE_ERR_RANGE;
        if (target_index[e] < 0 || target_index[e] >= query_features) return ORACLE_ERR_RANGE;
    }
    /* A pair is identified by the number target * key_features + source. */
    int64_t *pair = (int64_t *)malloc((size_t)nnz * sizeof(int64_t));
    if (!pair) return ORACLE_ERR_NOMEM;
    for (int64_t e = 0; e < nnz; ++e) pair[e] = target_index[e] * key_features + source_index[e];
    qsort(pair, (size_t)nnz, sizeof(int64_t), cmp_i64);
    int status = ORACLE_OK;
    for (int64_t e = 1; e < nnz; ++e)
        if (pair[e] == pair[e - 1]) { status = ORACLE_ERR_DUPLICATE; break; }
    free(pair);
    return status;
}

/* Writes the given pairs followed by every missing (i, i), i ascending, into
 * out_source / out_target (capacity nnz + n) and the new count into *out_nnz. */
int oracle_append_self_loops(const int64_t *source_index, const int64_t *target_index,
                             int64_t nnz, int64_t n, int64_t *out_source,
                             int64_t *out_target, int64_t *out_nnz)
{
    char *has_loop = (char *)calloc((size_t)n, 1);
    if (!has_loop) return ORACLE_ERR_NOMEM;
    for (int64_t e = 0; e < nnz; ++e) {
        out_source[e] = source_index[e];
        out_target[e] = target_index[e];
        if (source_index[e] == target_index[e]) has_loop[source_index[e]] = 1;
    }
    int64_t k = nnz;
    for (int64_t i = 0; i < n; ++i)
        if (!has_loop[i]) { out_source[k] = i; out_target[k] = i; ++k; }
    *out_nnz = k;
    free(has_loop);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Grouping of the edges by target (a CSR view).                             */
/* The pages gather per edge and never order the edges of one target; the   */
/* library orders them by (target, source). This is that order, written as a */
/* plain sort of (target, source, edge id) triples.                          */
/* row_ptr has query_features + 1 entries; col and perm have nnz entries:    */
/* col[i] is the source of the i-th edge in that order and perm[i] its       */
/* position in the caller's arrays.                                          */
/* ------------------------------------------------------------------------ */

typedef struct { int64_t target, source, id; } edge_triple;

static int cmp_triple(const void *a, const void *b)
{
    const edge_triple *x = (const edge_triple *)a, *y = (const edge_triple *)b;
    if (x->target != y->target) return (x->target > y->target) - (x->target < y->target);
    if (x->source != y->source) return (x->source > y->source) - (x->source < y->source);
    return (x->id > y->id) - (x->id < y->id);
}

int oracle_csr_by_target(const int64_t *source_index, const int64_t *target_index,
                         int64_t nnz, int64_t query_features,
                         int64_t *row_ptr, int64_t *col, int64_t *perm)
{
    edge_triple *t = (edge_triple *)malloc((size_t)(nnz > 0 ? nnz : 1) * sizeof(edge_triple));
    if (!t) return ORACLE_ERR_NOMEM;
    for (int64_t e = 0; e < nnz; ++e) {
        t[e].target = target_index[e];
        t[e].source = source_index[e];
        t[e].id = e;
    }
    qsort(t, (size_t)nnz, sizeof(edge_triple), cmp_triple);
    for (int64_t i = 0; i <= query_features; ++i) row_ptr[i] = 0;
    for (int64_t e = 0; e < nnz; ++e) row_ptr[t[e].target + 1] += 1;
    for (int64_t i = 0; i < query_features; ++i) row_ptr[i + 1] += row_ptr[i];
    for (int64_t e = 0; e < nnz; ++e) { col[e] = t[e].source; perm[e] = t[e].id; }
    free(t);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Projections. kpnn2 PackedMultiheadAttention, Notes step 1 and the         */
/* attribute table (four separate embed_dim -> embed_dim nn.Linear layers); */
/* nn.Linear stores its weight as (out_features, in_features), so            */
/*   Y[r, o] = sum_i X[r, i] * W[o, i] + b[o]                                 */
/* (the tutorial page writes the same as x @ W_q.T + b_q).                   */
/* bias may be NULL (bias=False).                                            */
/* ------------------------------------------------------------------------ */

void oracle_linear(int64_t rows, int64_t in_dim, int64_t out_dim, const double *X,
                   const double *W, const double *bias, double *Y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t o = 0; o < out_dim; ++o) {
            double acc = 0.0;
            for (int64_t i = 0; i < in_dim; ++i) acc += X[r * in_dim + i] * W[o * in_dim + i];
            if (bias) acc += bias[o];
            Y[r * out_dim + o] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Attention of one target over its live keys, all heads.                    */
/* kpnn2 PackedMultiheadAttention, Notes steps 2-4:                          */
/* (forward() parameter key_padding_mask: a masked key's edges take no part  */
/*  in the softmax; masked[j] != 0 marks edge j of this target as dropped,   */
/*  masked may be NULL)                                                      */
/*   score[e] = dot(q[t], k[s]) / sqrt(d)       per head, d = E / H channels */
/*   weight   = softmax of the scores over the edges into t only             */
/*   mixed[t] = sum_e weight[e] * v[s]                                       */
/* and the paragraph after the steps: a target with no live key mixes to     */
/* zeros (not NaN) and has no weights.                                       */
/* q has E entries; k_rows, v_rows are (n_edges, E) row-major, the projected */
/* key and value rows of the sources in edge order; mixed gets E entries;    */
/* weight (nullable) gets (n_edges, H): weight[j * H + h].                    */
/* The softmax is written with the maximum subtracted, which is the same     */
/* function and keeps exp() finite.                                          */
/* ------------------------------------------------------------------------ */

int oracle_attend_masked(int64_t embed_dim, int64_t num_heads, const double *q, int64_t n_edges,
                         const double *k_rows, const double *v_rows, const unsigned char *masked,
                         double *mixed, double *weight)
{
    if (num_heads < 1 || embed_dim % num_heads != 0) return ORACLE_ERR_ARG;
    const int64_t E = embed_dim, H = num_heads, d = E / H;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    for (int64_t c = 0; c < E; ++c) mixed[c] = 0.0;
    if (weight)
        for (int64_t j = 0; j < n_edges * H; ++j) weight[j] = 0.0;
    int64_t live = 0;
    for (int64_t j = 0; j < n_edges; ++j)
        if (!masked || !masked[j]) ++live;
    if (live == 0) return ORACLE_OK; /* no live key: mixes to zeros, weights 0 */
    double *score = (double *)malloc((size_t)n_edges * sizeof(double));
    if (!score) return ORACLE_ERR_NOMEM;
    for (int64_t h = 0; h < H; ++h) {
        /* step 2: one score per live edge */
        for (int64_t j = 0; j < n_edges; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c) dot += q[h * d + c] * k_rows[j * E + h * d + c];
            score[j] = dot * inv_sqrt_d;
        }
        /* step 3: softmax over the live edges into this target */
        double m = -INFINITY;
        for (int64_t j = 0; j < n_edges; ++j)
            if ((!masked || !masked[j]) && score[j] > m) m = score[j];
        double denom = 0.0;
        for (int64_t j = 0; j < n_edges; ++j)
            if (!masked || !masked[j]) denom += exp(score[j] - m);
        /* step 4: weighted sum of the value rows */
        for (int64_t j = 0; j < n_edges; ++j) {
            if (masked && masked[j]) continue;
            double w = exp(score[j] - m) / denom;
            if (weight) weight[j * H + h] = w;
            for (int64_t c = 0; c < d; ++c) mixed[h * d + c] += w * v_rows[j * E + h * d + c];
        }
    }
    free(score);
    return ORACLE_OK;
}

int oracle_attend(int64_t embed_dim, int64_t num_heads, const double *q, int64_t n_edges,
                  const double *k_rows, const double *v_rows, double *mixed, double *weight)
{
    return oracle_attend_masked(embed_dim, num_heads, q, n_edges, k_rows, v_rows, NULL, mixed, weight);
}

/* ------------------------------------------------------------------------ */
/* One full forward pass, batch-first.                                       */
/* kpnn2 PackedMultiheadAttention, Notes steps 1-5 and forward() Returns;    */
/* key_padding_mask (nullable) is (B, S) bytes, nonzero = key ignored in     */
/* that sample (forward() parameter key_padding_mask).                       */
/*   query (B, L, E), key and value (B, S, E); output (B, L, E);             */
/*   weight (B, nnz, H), one entry per live edge in the order of the index   */
/*   arrays (nullable).                                                      */
/* Step 5 joins the heads' slices (they already sit side by side in mixed)   */
/* and applies out_proj.                                                     */
/* The edges into each target are found by one pass over the index arrays   */
/* in their given order; no CSR from elsewhere is used.                      */
/* ------------------------------------------------------------------------ */

int oracle_forward_masked(int64_t batch, int64_t query_features, int64_t key_features,
                          int64_t embed_dim, int64_t num_heads,
                          const double *query, const double *key, const double *value,
                          const double *wq, const double *bq, const double *wk, const double *bk,
                          const double *wv, const double *bv, const double *wo, const double *bo,
                          int64_t nnz, const int64_t *source_index, const int64_t *target_index,
                          const unsigned char *key_padding_mask, double *output, double *weight)
{
    const int64_t B = batch, L = query_features, S = key_features, E = embed_dim, H = num_heads;
    if (B < 1 || L < 1 || S < 1 || E < 1 || H < 1 || E % H != 0) return ORACLE_ERR_ARG;
    int status = ORACLE_OK;

    /* step 1: projections of every token */
    double *q = (double *)malloc((size_t)(B * L * E) * sizeof(double));
    double *k = (double *)malloc((size_t)(B * S * E) * sizeof(double));
    double *v = (double *)malloc((size_t)(B * S * E) * sizeof(double));
    double *mixed = (double *)malloc((size_t)(B * L * E) * sizeof(double));
    /* edges into each target, in the order of the index arrays */
    int64_t *first = (int64_t *)malloc((size_t)(L + 1) * sizeof(int64_t));
    int64_t *fill = (int64_t *)malloc((size_t)(L + 1) * sizeof(int64_t));
    int64_t *edges_of = (int64_t *)malloc((size_t)(nnz > 0 ? nnz : 1) * sizeof(int64_t));
    if (!q || !k || !v || !mixed || !first || !fill || !edges_of) { status = ORACLE_ERR_NOMEM; goto done; }

    oracle_linear(B * L, E, E, query, wq, bq, q);
    oracle_linear(B * S, E, E, key, wk, bk, k);
    oracle_linear(B * S, E, E, value, wv, bv, v);

    for (int64_t t = 0; t <= L; ++t) first[t] = 0;
    for (int64_t e = 0; e < nnz; ++e) first[target_index[e] + 1] += 1;
    for (int64_t t = 0; t < L; ++t) first[t + 1] += first[t];
    for (int64_t t = 0; t <= L; ++t) fill[t] = first[t];
    for (int64_t e = 0; e < nnz; ++e) edges_of[fill[target_index[e]]++] = e;

    /* steps 2-4 for every (sample, target) */
#pragma omp parallel
    {
        int64_t max_deg = 0;
        for (int64_t t = 0; t < L; ++t)
            if (first[t + 1] - first[t] > max_deg) max_deg = first[t + 1] - first[t];
        double *kr = (double *)malloc((size_t)(max_deg > 0 ? max_deg : 1) * E * sizeof(double));
        double *vr = (double *)malloc((size_t)(max_deg > 0 ? max_deg : 1) * E * sizeof(double));
        double *wr = (double *)malloc((size_t)(max_deg > 0 ? max_deg : 1) * H * sizeof(double));
        unsigned char *mk = (unsigned char *)malloc((size_t)(max_deg > 0 ? max_deg : 1));
        int local_status = (kr && vr && wr && mk) ? ORACLE_OK : ORACLE_ERR_NOMEM;
#pragma omp for schedule(dynamic, 16)
        for (int64_t bt = 0; bt < B * L; ++bt) {
            if (local_status != ORACLE_OK) continue;
            const int64_t b = bt / L, t = bt % L;
            const int64_t deg = first[t + 1] - first[t];
            for (int64_t j = 0; j < deg; ++j) {
                const int64_t s = source_index[edges_of[first[t] + j]];
                memcpy(kr + j * E, k + (b * S + s) * E, (size_t)E * sizeof(double));
                memcpy(vr + j * E, v + (b * S + s) * E, (size_t)E * sizeof(double));
                mk[j] = key_padding_mask ? key_padding_mask[b * S + s] : 0;
            }
            oracle_attend_masked(E, H, q + (b * L + t) * E, deg, kr, vr, mk, mixed + (b * L + t) * E, wr);
            if (weight)
                for (int64_t j = 0; j < deg; ++j) {
                    const int64_t e = edges_of[first[t] + j];
                    for (int64_t h = 0; h < H; ++h) weight[(b * nnz + e) * H + h] = wr[j * H + h];
                }
        }
        if (local_status != ORACLE_OK) {
#pragma omp atomic write
            status = local_status;
        }
        free(kr); free(vr); free(wr); free(mk);
    }
    if (status != ORACLE_OK) goto done;

    /* step 5: join heads (already adjacent in mixed) and out_proj */
    oracle_linear(B * L, E, E, mixed, wo, bo, output);

done:
    free(q); free(k); free(v); free(mixed); free(first); free(fill); free(edges_of);
    return status;
}

int oracle_forward(int64_t batch, int64_t query_features, int64_t key_features,
                   int64_t embed_dim, int64_t num_heads,
                   const double *query, const double *key, const double *value,
                   const double *wq, const double *bq, const double *wk, const double *bk,
                   const double *wv, const double *bv, const double *wo, const double *bo,
                   int64_t nnz, const int64_t *source_index, const int64_t *target_index,
                   double *output, double *weight)
{
    return oracle_forward_masked(batch, query_features, key_features, embed_dim, num_heads, query, key, value,
                                 wq, bq, wk, bk, wv, bv, wo, bo, nnz, source_index, target_index, NULL,
                                 output, weight);
}

/* Mean over heads of per-head weights: kpnn2 forward(), average_attn_weights
 * (True averages the weights over the heads). w_head is (rows, H); w_avg (rows). */
/* ------------------------------------------------------------------------ */
/* Backward of one nn.Linear layer (the projections of Notes step 1 and      */
/* out_proj of step 5): for Y = X W^T + b and a gradient dY of Y,            */
/*   dX[r, i] = sum_o dY[r, o] * W[o, i]                                     */
/*   dW[o, i] = sum_r dY[r, o] * X[r, i]                                     */
/*   db[o]    = sum_r dY[r, o]                                               */
/* Any of dX, dW, db may be NULL. Sums run over r in increasing order.       */
/* ------------------------------------------------------------------------ */

void oracle_linear_backward(int64_t rows, int64_t in_dim, int64_t out_dim, const double *X,
                            const double *W, const double *dY, double *dX, double *dW, double *db)
{
    if (dX) {
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t i = 0; i < in_dim; ++i) {
                double acc = 0.0;
                for (int64_t o = 0; o < out_dim; ++o) acc += dY[r * out_dim + o] * W[o * in_dim + i];
                dX[r * in_dim + i] = acc;
            }
    }
    if (dW) {
#pragma omp parallel for schedule(static)
        for (int64_t o = 0; o < out_dim; ++o)
            for (int64_t i = 0; i < in_dim; ++i) {
                double acc = 0.0;
                for (int64_t r = 0; r < rows; ++r) acc += dY[r * out_dim + o] * X[r * in_dim + i];
                dW[o * in_dim + i] = acc;
            }
    }
    if (db) {
#pragma omp parallel for schedule(static)
        for (int64_t o = 0; o < out_dim; ++o) {
            double acc = 0.0;
            for (int64_t r = 0; r < rows; ++r) acc += dY[r * out_dim + o];
            db[o] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Backward of one full forward pass: the chain rule of Notes steps 1-5.     */
/* (The page's training path recomputes the attention in the backward pass  */
/* instead of keeping the packed per-edge tensors; so does this function:    */
/* it recomputes the forward from the inputs.)                               */
/* Given dout = dLoss/d output (B, L, E):                                    */
/*   step 5:  dmixed = dout Wo, dWo = dout^T mixed, dbo = sum dout           */
/*   steps 2-4, per (sample b, target t, head h), over the live edges e into */
/*   t, with weights w_e and scores s_e of the forward:                      */
/*     dw_e  = dot(dmixed[t, h], v[s_e, h])                                  */
/*     ds_e  = w_e * (dw_e - sum_e' w_e' dw_e')      (softmax backward)      */
/*     dq[t, h]   += ds_e * k[s_e, h] / sqrt(d)                              */
/*     dk[s_e, h] += ds_e * q[t, h] / sqrt(d)                                */
/*     dv[s_e, h] += w_e * dmixed[t, h]                                      */
/*   dropped keys (key_padding_mask) have no weight and get nothing;         */
/*   step 1:  each projection through oracle_linear_backward.                */
/* Outputs: dquery (B, L, E), dkey and dvalue (B, S, E) - one per input even */
/* when the caller passes one tensor for several inputs (the caller adds     */
/* them) - and dwq.. dwo (E, E), dbq.. dbo (E) (bias gradients may be NULL). */
/* ------------------------------------------------------------------------ */

int oracle_backward(int64_t batch, int64_t query_features, int64_t key_features, int64_t embed_dim,
                    int64_t num_heads, const double *query, const double *key, const double *value,
                    const double *wq, const double *bq, const double *wk, const double *bk, const double *wv,
                    const double *bv, const double *wo, const double *bo, int64_t nnz,
                    const int64_t *source_index, const int64_t *target_index,
                    const unsigned char *key_padding_mask, const double *dout, double *dquery, double *dkey,
                    double *dvalue, double *dwq, double *dbq, double *dwk, double *dbk, double *dwv, double *dbv,
                    double *dwo, double *dbo)
{
    (void)bo;
    const int64_t B = batch, L = query_features, S = key_features, E = embed_dim, H = num_heads;
    if (B < 1 || L < 1 || S < 1 || E < 1 || H < 1 || E % H != 0) return ORACLE_ERR_ARG;
    const int64_t d = E / H;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    int status = ORACLE_OK;
    double *q = (double *)malloc((size_t)(B * L * E) * sizeof(double));
    double *k = (double *)malloc((size_t)(B * S * E) * sizeof(double));
    double *v = (double *)malloc((size_t)(B * S * E) * sizeof(double));
    double *mixed = (double *)calloc((size_t)(B * L * E), sizeof(double));
    double *dmixed = (double *)malloc((size_t)(B * L * E) * sizeof(double));
    double *dq = (double *)calloc((size_t)(B * L * E), sizeof(double));
    double *dk = (double *)calloc((size_t)(B * S * E), sizeof(double));
    double *dv = (double *)calloc((size_t)(B * S * E), sizeof(double));
    int64_t *first = (int64_t *)malloc((size_t)(L + 1) * sizeof(int64_t));
    int64_t *fill = (int64_t *)malloc((size_t)(L + 1) * sizeof(int64_t));
    int64_t *edges_of = (int64_t *)malloc((size_t)(nnz > 0 ? nnz : 1) * sizeof(int64_t));
    if (!q || !k || !v || !mixed || !dmixed || !dq || !dk || !dv || !first || !fill || !edges_of) {
        status = ORACLE_ERR_NOMEM;
        goto done;
    }
    /* forward recompute: projections and, per target, its edges in index-array order */
    oracle_linear(B * L, E, E, query, wq, bq, q);
    oracle_linear(B * S, E, E, key, wk, bk, k);
    oracle_linear(B * S, E, E, value, wv, bv, v);
    for (int64_t t = 0; t <= L; ++t) first[t] = 0;
    for (int64_t e = 0; e < nnz; ++e) first[target_index[e] + 1] += 1;
    for (int64_t t = 0; t < L; ++t) first[t + 1] += first[t];
    for (int64_t t = 0; t <= L; ++t) fill[t] = first[t];
    for (int64_t e = 0; e < nnz; ++e) edges_of[fill[target_index[e]]++] = e;

    /* steps 2-4 forward (weights and mixed) and backward, one sample per thread:
       dk and dv of a sample only receive from that sample's targets */
#pragma omp parallel
    {
        int64_t max_deg = 0;
        for (int64_t t = 0; t < L; ++t)
            if (first[t + 1] - first[t] > max_deg) max_deg = first[t + 1] - first[t];
        const int64_t cap = max_deg > 0 ? max_deg : 1;
        double *w = (double *)malloc((size_t)cap * sizeof(double));
        double *dw = (double *)malloc((size_t)cap * sizeof(double));
        int local_status = (w && dw) ? ORACLE_OK : ORACLE_ERR_NOMEM;
#pragma omp for schedule(dynamic, 1)
        for (int64_t b = 0; b < B; ++b) {
            if (local_status != ORACLE_OK) continue;
            /* forward mixed of every target of this sample, then step 5's dmixed */
            for (int64_t t = 0; t < L; ++t) {
                const int64_t deg = first[t + 1] - first[t];
                for (int64_t h = 0; h < H; ++h) {
                    double m = -INFINITY;
                    int64_t live = 0;
                    for (int64_t j = 0; j < deg; ++j) {
                        const int64_t s = source_index[edges_of[first[t] + j]];
                        if (key_padding_mask && key_padding_mask[b * S + s]) continue;
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c) dot += q[(b * L + t) * E + h * d + c] * k[(b * S + s) * E + h * d + c];
                        w[j] = dot * inv_sqrt_d;
                        if (w[j] > m) m = w[j];
                        ++live;
                    }
                    if (live == 0) continue;
                    double denom = 0.0;
                    for (int64_t j = 0; j < deg; ++j) {
                        const int64_t s = source_index[edges_of[first[t] + j]];
                        if (key_padding_mask && key_padding_mask[b * S + s]) continue;
                        denom += exp(w[j] - m);
                    }
                    for (int64_t j = 0; j < deg; ++j) {
                        const int64_t s = source_index[edges_of[first[t] + j]];
                        if (key_padding_mask && key_padding_mask[b * S + s]) continue;
                        const double wj = exp(w[j] - m) / denom;
                        for (int64_t c = 0; c < d; ++c)
                            mixed[(b * L + t) * E + h * d + c] += wj * v[(b * S + s) * E + h * d + c];
                    }
                }
            }
        }
        free(w);
        free(dw);
        if (local_status != ORACLE_OK) {
#pragma omp atomic write
            status = local_status;
        }
    }
    if (status != ORACLE_OK) goto done;
    /* step 5 backward */
    oracle_linear_backward(B * L, E, E, mixed, wo, dout, dmixed, dwo, dbo);
#pragma omp parallel
    {
        int64_t max_deg = 0;
        for (int64_t t = 0; t < L; ++t)
            if (first[t + 1] - first[t] > max_deg) max_deg = first[t + 1] - first[t];
        const int64_t cap = max_deg > 0 ? max_deg : 1;
        double *w = (double *)malloc((size_t)cap * sizeof(double));
        double *dw = (double *)malloc((size_t)cap * sizeof(double));
        int local_status = (w && dw) ? ORACLE_OK : ORACLE_ERR_NOMEM;
#pragma omp for schedule(dynamic, 1)
        for (int64_t b = 0; b < B; ++b) {
            if (local_status != ORACLE_OK) continue;
            for (int64_t t = 0; t < L; ++t) {
                const int64_t deg = first[t + 1] - first[t];
                const double *qt = q + (b * L + t) * E;
                const double *gt = dmixed + (b * L + t) * E;
                for (int64_t h = 0; h < H; ++h) {
                    /* the forward weights of this (target, head) */
                    double m = -INFINITY;
                    int64_t live = 0;
                    for (int64_t j = 0; j < deg; ++j) {
                        const int64_t s = source_index[edges_of[first[t] + j]];
                        if (key_padding_mask && key_padding_mask[b * S + s]) continue;
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c) dot += qt[h * d + c] * k[(b * S + s) * E + h * d + c];
                        w[j] = dot * inv_sqrt_d;
                        if (w[j] > m) m = w[j];
                        ++live;
                    }
                    if (live == 0) continue;
                    double denom = 0.0;
                    for (int64_t j = 0; j < deg; ++j) {
                        const int64_t s = source_index[edges_of[first[t] + j]];
                        if (key_padding_mask && key_padding_mask[b * S + s]) continue;
                        denom += exp(w[j] - m);
                    }
                    /* dw_e and their weighted sum */
                    double wdw = 0.0;
                    for (int64_t j = 0; j < deg; ++j) {
                        const int64_t s = source_index[edges_of[first[t] + j]];
                        if (key_padding_mask && key_padding_mask[b * S + s]) continue;
                        w[j] = exp(w[j] - m) / denom;
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c) dot += gt[h * d + c] * v[(b * S + s) * E + h * d + c];
                        dw[j] = dot;
                        wdw += w[j] * dot;
                    }
                    for (int64_t j = 0; j < deg; ++j) {
                        const int64_t s = source_index[edges_of[first[t] + j]];
                        if (key_padding_mask && key_padding_mask[b * S + s]) continue;
                        const double ds = w[j] * (dw[j] - wdw);
                        for (int64_t c = 0; c < d; ++c) {
                            dq[(b * L + t) * E + h * d + c] += ds * k[(b * S + s) * E + h * d + c] * inv_sqrt_d;
                            dk[(b * S + s) * E + h * d + c] += ds * qt[h * d + c] * inv_sqrt_d;
                            dv[(b * S + s) * E + h * d + c] += w[j] * gt[h * d + c];
                        }
                    }
                }
            }
        }
        free(w);
        free(dw);
        if (local_status != ORACLE_OK) {
#pragma omp atomic write
            status = local_status;
        }
    }
    if (status != ORACLE_OK) goto done;
    /* step 1 backward */
    oracle_linear_backward(B * L, E, E, query, wq, dq, dquery, dwq, dbq);
    oracle_linear_backward(B * S, E, E, key, wk, dk, dkey, dwk, dbk);
    oracle_linear_backward(B * S, E, E, value, wv, dv, dvalue, dwv, dbv);

done:
    free(q); free(k); free(v); free(mixed); free(dmixed); free(dq); free(dk); free(dv);
    free(first); free(fill); free(edges_of);
    return status;
}

void oracle_average_heads(int64_t rows, int64_t num_heads, const double *w_head, double *w_avg)
{
    for (int64_t r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int64_t h = 0; h < num_heads; ++h) acc += w_head[r * num_heads + h];
        w_avg[r] = acc / (double)num_heads;
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
