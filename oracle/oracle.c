/*
 * CPU oracle for the sequence-parallel linear layer on packed THD activations.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct statement of
 * what the GPU path computes. Only the test suite, the smoke check and the timed
 * CPU baseline of the benchmark load it; the library under test never does, and the
 * two share no code, headers or constants.
 *
 * Sources (three web pages on tensor-parallel communication/GEMM overlap):
 *  - "Do tp overlap support thd, whose sequence length is flexible?" (Megatron-LM
 *    discussion #1240), answer, QKV and MLP diagrams: the column-parallel layer
 *    consumes the all-gathered input [S, H]; the row-parallel layer produces [S, H]
 *    that is summed over ranks and split by rows.
 *  - "Support dynamic token counts in TP communication/GEMM overlap" (TransformerEngine
 *    issue #3564), sections "Implementation approach in the prototype" and
 *    "Constrain the initial behavior": the active data is a contiguous prefix of the
 *    capacity buffer; chunk views and offsets are rebuilt from the active first
 *    dimension T; T must be nonzero, within capacity and divisible by the TP size.
 *
 * Conventions.
 *  - bf16 values travel as their 16-bit patterns (uint16_t). Widening bf16 -> double
 *    is exact (shift into the top half of a float).
 *  - Every product is formed and summed in double, in the index order the definition
 *    states (h = 0..H-1; j = 0..tp-1 outer, k = 0..K-1 inner).
 *  - Linear weights are stored the way PyTorch stores nn.Linear weights: out x in,
 *    row-major. So the column-parallel weight is Wt[N][H] and Y = X * Wt^T; the
 *    row-parallel shard weights are Bt_j[H][K] and S = sum_j A_j * Bt_j^T.
 *  - Chunk r of an active shape (T, H) split over tp ranks is rows [r*c, (r+1)*c)
 *    with c = T / tp, computed from T and never from the capacity.
 *
 * Parity status: every function here is pinned by CPU tests against closed forms,
 * brute-force integer arithmetic, a library matmul special case (tp = 1), the
 * shard-concatenation identity and a hand-worked example.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern to double. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Round a double to the nearest bf16, ties to even, in one step (no intermediate
 * float rounding): keep 8 significant bits (7 stored plus the implicit one); below
 * the smallest normal the spacing stays 2^-133 (bf16 subnormals). A result past
 * the largest finite bf16 becomes infinity; NaN becomes the canonical quiet NaN. */
uint16_t oracle_round_bf16(double v)
{
    if (isnan(v)) return (uint16_t)0x7fc0u;
    double r = v;
    if (v != 0.0 && !isinf(v)) {
        int e;
        frexp(fabs(v), &e);            /* |v| = m * 2^e with m in [0.5, 1) */
        int lsb = (e - 1) - 7;         /* weight of the last kept bit */
        if (lsb < -133) lsb = -133;
        double unit = ldexp(1.0, lsb);
        r = nearbyint(v / unit) * unit; /* default rounding mode: to nearest even */
    }
    float f = (float)r;                /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Chunk layout from the active shape: offset of chunk r in rows, and its row count.
 * The offset is r * (T / tp): the active first dimension, not the capacity. */
int64_t oracle_chunk_rows(int64_t T, int tp) { return T / tp; }
int64_t oracle_chunk_offset(int64_t T, int tp, int r) { return (int64_t)r * (T / tp); }

/* All-gather into the capacity buffer G[capacity][H]:
 * G[r*c + i][h] = X_r[i][h] for r < tp, i < c. Rows >= T are not touched. */
void oracle_allgather(int tp, int64_t T, int64_t H,
                      const uint16_t *const *shards, uint16_t *G)
{
    int64_t c = oracle_chunk_rows(T, tp);
    for (int r = 0; r < tp; ++r) {
        int64_t row0 = oracle_chunk_offset(T, tp, r);
        for (int64_t i = 0; i < c; ++i)
            for (int64_t h = 0; h < H; ++h)
                G[(row0 + i) * H + h] = shards[r][i * H + h];
    }
}

/* Plain product of selected rows: Y[q][n] = sum_{h<K} X[rows[q]][h] * Wt[n][h].
 * X has leading dimension ldx (elements); Y is nrows x N, row-major, double. */
void oracle_gemm_xwt_rows(const uint16_t *X, int64_t ldx, const uint16_t *Wt,
                          int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                          double *Y)
{
    int64_t q;
#pragma omp parallel for schedule(dynamic, 1)
    for (q = 0; q < nrows; ++q) {
        const uint16_t *x = X + rows[q] * ldx;
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t *w = Wt + n * K;
            double acc = 0.0;
            for (int64_t h = 0; h < K; ++h)
                acc += bf16_to_double(x[h]) * bf16_to_double(w[h]);
            Y[q * N + n] = acc;
        }
    }
}

/* AG-GEMM: gather the tp token shards into G (capacity buffer, prefix of T rows),
 * then Y[t][n] = sum_h G[t][h] * Wt[n][h] for t < T. Y is T x N, double. */
void oracle_ag_gemm(int tp, int64_t T, int64_t H, int64_t N,
                    const uint16_t *const *shards, const uint16_t *Wt,
                    uint16_t *G, double *Y)
{
    oracle_allgather(tp, T, H, shards, G);
    int64_t t;
#pragma omp parallel for schedule(dynamic, 1)
    for (t = 0; t < T; ++t) {
        const uint16_t *g = G + t * H;
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t *w = Wt + n * H;
            double acc = 0.0;
            for (int64_t h = 0; h < H; ++h)
                acc += bf16_to_double(g[h]) * bf16_to_double(w[h]);
            Y[t * N + n] = acc;
        }
    }
}

/* One output element of the cross-shard sum:
 * S[t][n] = sum_{j<tp} sum_{k<K} A_j[t][k] * Bt_j[n][k]. */
static double rs_element(int tp, int64_t K, const uint16_t *const *A,
                         const uint16_t *const *Bt, int64_t t, int64_t n)
{
    double s = 0.0;
    for (int j = 0; j < tp; ++j) {
        const uint16_t *a = A[j] + t * K;
        const uint16_t *b = Bt[j] + n * K;
        double partial = 0.0;
        for (int64_t k = 0; k < K; ++k)
            partial += bf16_to_double(a[k]) * bf16_to_double(b[k]);
        s += partial;
    }
    return s;
}

/* GEMM-RS: S = sum_j A_j * Bt_j^T over all T active rows (S is T x H, double), then
 * the row scatter Yr[i][n] = S[r*c + i][n] into each rank's block (c x H, double).
 * S may be NULL when only the scattered blocks are wanted. */
void oracle_gemm_rs(int tp, int64_t T, int64_t K, int64_t H,
                    const uint16_t *const *A, const uint16_t *const *Bt,
                    double *S, double *const *Yr)
{
    int64_t c = oracle_chunk_rows(T, tp);
    int64_t t;
#pragma omp parallel for schedule(dynamic, 1)
    for (t = 0; t < T; ++t) {
        int r = (int)(t / c);                      /* owner of row t */
        int64_t i = t - oracle_chunk_offset(T, tp, r); /* row inside the owner's block */
        for (int64_t n = 0; n < H; ++n) {
            double v = rs_element(tp, K, A, Bt, t, n);
            if (S) S[t * H + n] = v;
            Yr[r][i * H + n] = v;
        }
    }
}

/* GEMM-RS on selected rows of the active prefix (for full-size spot checks). The
 * caller passes, per shard j, only the selected rows: A_rows[j][q][k] = A_j[rows[q]][k].
 * out[q][n] = S[rows[q]][n]; owner[q] = rows[q] / c; local[q] = rows[q] - owner[q]*c. */
void oracle_gemm_rs_rows(int tp, int64_t T, int64_t K, int64_t H,
                         const uint16_t *const *A_rows, const uint16_t *const *Bt,
                         const int64_t *rows, int64_t nrows,
                         double *out, int32_t *owner, int64_t *local)
{
    int64_t c = oracle_chunk_rows(T, tp);
    int64_t q;
#pragma omp parallel for schedule(dynamic, 1)
    for (q = 0; q < nrows; ++q) {
        int64_t t = rows[q];
        int r = (int)(t / c);
        owner[q] = r;
        local[q] = t - oracle_chunk_offset(T, tp, r);
        for (int64_t n = 0; n < H; ++n)
            out[q * H + n] = rs_element(tp, K, A_rows, Bt, q, n);
    }
}

/* The weight operand in its mathematical layout, K x N row-major (the layout the
 * workloads write W[hidden, N] and B_j[K, hidden] in): Y[q][n] = sum_k X[rows[q]][k] *
 * W[k][n]. With W stored this way the same products serve the backward pass: the
 * column-parallel layer's input gradient is sum_j dY_j * Wt_j (Wt_j stored [N_j, H],
 * i.e. K x N with K = N_j), the row-parallel layer's is dS * Bt_j. */
void oracle_gemm_xw_rows(const uint16_t *X, int64_t ldx, const uint16_t *W, int64_t N, int64_t K,
                         const int64_t *rows, int64_t nrows, double *Y)
{
    int64_t q;
#pragma omp parallel for schedule(dynamic, 1)
    for (q = 0; q < nrows; ++q) {
        const uint16_t *x = X + rows[q] * ldx;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += bf16_to_double(x[k]) * bf16_to_double(W[k * N + n]);
            Y[q * N + n] = acc;
        }
    }
}

/* Weight gradient: the contraction over the T active tokens of two [T, .] activations,
 * out[m][n] = sum_{t<T} D[t][m] * G[t][n] (D [T, M], G [T, N], out [M, N], double).
 * For the column-parallel layer D = dY and G = the gathered input (dWt = dY^T G); for
 * the row-parallel layer D = the gathered dS and G = A_j (dBt_j = dS^T A_j). */
void oracle_gemm_tn(const uint16_t *D, int64_t M, const uint16_t *G, int64_t N, int64_t T, double *out)
{
    int64_t m;
#pragma omp parallel for schedule(dynamic, 1)
    for (m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t t = 0; t < T; ++t)
                acc += bf16_to_double(D[t * M + m]) * bf16_to_double(G[t * N + n]);
            out[m * N + n] = acc;
        }
    }
}

/* Reduce-scatter of tp partial results (the "bulk" method's independent reduce-scatter
 * in "How to setup TP Overlap configs"): every rank holds a full partial P_j [T, H];
 * rank r keeps rows [r*c, (r+1)*c) of their sum, Y_r[i][n] = sum_{j<tp} P_j[r*c + i][n],
 * summed in the order j = 0..tp-1 in double. */
void oracle_reduce_scatter(int tp, int64_t T, int64_t H, const uint16_t *const *P, double *const *Yr)
{
    int64_t c = oracle_chunk_rows(T, tp);
    int64_t t;
#pragma omp parallel for schedule(dynamic, 1)
    for (t = 0; t < T; ++t) {
        int r = (int)(t / c);
        int64_t i = t - oracle_chunk_offset(T, tp, r);
        for (int64_t n = 0; n < H; ++n) {
            double s = 0.0;
            for (int j = 0; j < tp; ++j) s += bf16_to_double(P[j][t * H + n]);
            Yr[r][i * H + n] = s;
        }
    }
}

/* SwiGLU between the column-parallel fc1 and the row-parallel fc2 (the GELU/SwiGLU box
 * of the MLP diagram in "Do tp overlap support thd..."): fc1's output row holds the
 * gate half first and the up half second, Y[t] = [g_0..g_{F-1}, u_0..u_{F-1}], and
 * Z[t][f] = silu(g_f) * u_f with silu(x) = x / (1 + e^{-x}), all in double. */
double oracle_silu(double x)
{
    return x / (1.0 + exp(-x));
}

void oracle_swiglu(const double *Y, int64_t rows, int64_t F, double *Z)
{
    for (int64_t t = 0; t < rows; ++t)
        for (int64_t f = 0; f < F; ++f)
            Z[t * F + f] = oracle_silu(Y[t * 2 * F + f]) * Y[t * 2 * F + F + f];
}

/* Active-shape constraints, in the order the page lists them: two-dimensional,
 * nonzero, within capacity, hidden unchanged, first dimension divisible by tp.
 * Returns 0 when accepted, else the 1-based index of the first violated rule. */
int oracle_check_active_shape(int ndim, int64_t T, int64_t hidden,
                              int64_t cap_tokens, int64_t cap_hidden, int tp)
{
    if (ndim != 2) return 1;
    if (T <= 0 || hidden <= 0) return 2;
    if (T > cap_tokens) return 3;
    if (hidden != cap_hidden) return 4;
    if (T % tp != 0) return 5;
    return 0;
}
