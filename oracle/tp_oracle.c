/*
 * tp_oracle.c - plain, slow fp64 CPU oracle for the tensor-parallel MLP.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference leg load this library.  It shares no code with the
 * CUDA path and the CUDA path never calls it.
 *
 * What it computes, and where the pages state it:
 *   - Column-parallel first layer: W1 split along its output (column)
 *     dimension, Y_i = act(X W1_i), X replicated, no exchange afterwards
 *     ("Tensor Parallelism in Action: Megatron-LM Matrix Splitting",
 *     section 1, "Column Parallel (W1)"; "Tensor parallelism" guide, section
 *     "Concept").
 *   - The activation is applied per shard because it is elementwise:
 *     GeLU([y1 | y2]) = [GeLU(y1) | GeLU(y2)] ("Tensor Parallelism in
 *     Action", section 2, interview question 2).
 *   - Row-parallel second layer: W2 split along its input (row) dimension,
 *     Z_i = Y_i W2_i are partial products ("Tensor Parallelism in Action",
 *     section 1, "Row Parallel (W2)"; "Slice the matrix itself", section
 *     "Column-Parallel & Row-Parallel GEMMs").
 *   - All-reduce-sum of the partials, Z = sum_i Z_i ("Slice the matrix
 *     itself", section "Mathematical formulation - row-parallel matrix
 *     multiplication summation"; "Tensor Parallelism in Action", section 1,
 *     "Output Combination").
 *   - Attention: heads are sharded across ranks ("Tensor parallelism" guide,
 *     section "Walking through a transformer block"), so the QKV projection
 *     is column-parallel by head and the output projection row-parallel; the
 *     attention core of each head is local (orc_attention), and one whole
 *     block adds the two all-reduces and residuals (orc_block_forward).
 *   - The collectives around the all-reduce: reduce-scatter, all-gather and
 *     the sum rounded once to bfloat16 ("Tensor Parallelism in Action",
 *     section 2, question 3 names AllReduce, AllGather and ReduceScatter).
 *   - The backward pass of the MLP: the input gradient is again a sum over
 *     shards (the all-reduce of the backward pass), the weight gradients are
 *     per shard ("Slice the matrix itself", section "Strict NVLink Domain
 *     Constraint": all-reduces in every layer's forward and backward pass).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - GeLU is the exact form 0.5 y (1 + erf(y / sqrt 2)).
 *   - SwiGLU ("Gate/Up" in "Slice the matrix itself") is SiLU(g) * u with
 *     SiLU(g) = g / (1 + exp(-g)); W1 is given as [Wg | Wu] ([H x 2F], gate
 *     first) and shard i takes the SAME columns of Wg and of Wu.
 *   - QKV weights are [Wq | Wk | Wv], each [H x H], head h in columns
 *     [h*hd, (h+1)*hd); shard i takes heads [i*nh/T, (i+1)*nh/T) of all three.
 *   - Shards are equal: F % T == 0 and n_heads % T == 0, else an error.
 *   - The all-reduce sum runs over shards in ascending order, left to right.
 *
 * Everything is fp64 on the exact input values: float32 and bfloat16 inputs
 * are widened exactly.  Loops are the plain definitions; OpenMP only splits
 * independent output rows between threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F64 2 /* test inputs for finite differences */

#define ORC_GELU 0
#define ORC_SWIGLU 1
#define ORC_IDENTITY 2

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_INDIVISIBLE 2
#define ORC_ERR_OOM 5

/* ---- element access ---------------------------------------------------- */

size_t orc_elem_bytes(int dt) { return dt == ORC_BF16 ? 2u : dt == ORC_F64 ? 8u : 4u; }

/* Exact value of element idx of an array of float32 or bfloat16 (the upper
 * 16 bits of a float32). */
double orc_value(const void *base, int64_t idx, int dt)
{
    float f;
    if (dt == ORC_F64)
        return ((const double *)base)[idx];
    if (dt == ORC_F32) {
        f = ((const float *)base)[idx];
    } else {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        memcpy(&f, &bits, sizeof f);
    }
    return (double)f;
}

uint16_t orc_f32_to_bf16(float f);

/* Value of a bfloat16 bit pattern. */
static double bf16_bits_value(uint16_t b) { return orc_value(&b, 0, ORC_BF16); }

/* ---- activations ------------------------------------------------------- */

/* GeLU(y) = y * Phi(y), Phi the standard normal CDF, via erf. */
double orc_gelu(double y) { return 0.5 * y * (1.0 + erf(y / sqrt(2.0))); }

/* SiLU(g) = g * sigmoid(g). */
double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/* ---- shard partition (bit copies) -------------------------------------- */

/* Column block i of W1 (which = 0), or, for SwiGLU, of the gate half
 * (which = 0) or the up half (which = 1), as a row-major [H x F/T] array.
 * W1 is [H x F] (GeLU, identity) or [H x 2F] = [Wg | Wu] (SwiGLU). */
int orc_shard_w1(const void *W1, int dt, int64_t H, int64_t F, int T, int act,
                 int i, int which, void *out)
{
    if (!W1 || !out || H <= 0 || F <= 0 || T <= 0 || i < 0 || i >= T)
        return ORC_ERR_ARG;
    if (F % T != 0)
        return ORC_ERR_INDIVISIBLE;
    if (which != 0 && !(act == ORC_SWIGLU && which == 1))
        return ORC_ERR_ARG;
    const size_t eb = orc_elem_bytes(dt);
    const int64_t Fs = F / T;
    const int64_t ld = (act == ORC_SWIGLU) ? 2 * F : F;
    const int64_t col0 = (int64_t)which * F + (int64_t)i * Fs;
    for (int64_t k = 0; k < H; ++k)
        for (int64_t c = 0; c < Fs; ++c)
            memcpy((char *)out + (size_t)(k * Fs + c) * eb,
                   (const char *)W1 + (size_t)(k * ld + col0 + c) * eb, eb);
    return ORC_OK;
}

/* Row block i of W2 ([F x H]) as a row-major [F/T x H] array. */
int orc_shard_w2(const void *W2, int dt, int64_t F, int64_t H, int T, int i, void *out)
{
    if (!W2 || !out || H <= 0 || F <= 0 || T <= 0 || i < 0 || i >= T)
        return ORC_ERR_ARG;
    if (F % T != 0)
        return ORC_ERR_INDIVISIBLE;
    const size_t eb = orc_elem_bytes(dt);
    const int64_t Fs = F / T;
    for (int64_t r = 0; r < Fs; ++r)
        for (int64_t c = 0; c < H; ++c)
            memcpy((char *)out + (size_t)(r * H + c) * eb,
                   (const char *)W2 + (size_t)((i * Fs + r) * H + c) * eb, eb);
    return ORC_OK;
}

/* Heads of shard i from each of Wq, Wk, Wv: Wqkv is [H x 3H] = [Wq|Wk|Wv];
 * out is [H x 3*W] with W = (n_heads/T)*head_dim, holding the Wq columns,
 * then the Wk columns, then the Wv columns of those heads. */
int orc_shard_wqkv(const void *Wqkv, int dt, int64_t H, int n_heads, int head_dim,
                   int T, int i, void *out)
{
    if (!Wqkv || !out || H <= 0 || n_heads <= 0 || head_dim <= 0 || T <= 0 ||
        i < 0 || i >= T || (int64_t)n_heads * head_dim != H)
        return ORC_ERR_ARG;
    if (n_heads % T != 0)
        return ORC_ERR_INDIVISIBLE;
    const size_t eb = orc_elem_bytes(dt);
    const int64_t W = (int64_t)(n_heads / T) * head_dim;
    for (int64_t k = 0; k < H; ++k)
        for (int p = 0; p < 3; ++p)
            for (int64_t c = 0; c < W; ++c)
                memcpy((char *)out + (size_t)(k * 3 * W + p * W + c) * eb,
                       (const char *)Wqkv + (size_t)(k * 3 * H + p * H + i * W + c) * eb, eb);
    return ORC_OK;
}

/* Rows of Wo ([H x H], input dim = heads side by side) that belong to the
 * heads of shard i: out is [W x H], W = (n_heads/T)*head_dim. */
int orc_shard_wo(const void *Wo, int dt, int64_t H, int n_heads, int head_dim,
                 int T, int i, void *out)
{
    if (!Wo || !out || H <= 0 || n_heads <= 0 || head_dim <= 0 || T <= 0 ||
        i < 0 || i >= T || (int64_t)n_heads * head_dim != H)
        return ORC_ERR_ARG;
    if (n_heads % T != 0)
        return ORC_ERR_INDIVISIBLE;
    const size_t eb = orc_elem_bytes(dt);
    const int64_t W = (int64_t)(n_heads / T) * head_dim;
    memcpy(out, (const char *)Wo + (size_t)(i * W * H) * eb, (size_t)(W * H) * eb);
    return ORC_OK;
}

/* ---- dense building blocks --------------------------------------------- */

/* One output row of a plain linear layer: out[c] = sum_k a[k] * W[k][c],
 * W row-major [K x N] with leading dimension ldw, starting at column col0.
 * a is a row of A (element offset a0, element type dt). */
static void row_times_matrix(const void *A, int64_t a0, int dt, int64_t K,
                             const void *W, int64_t ldw, int64_t col0, int64_t N,
                             double *out)
{
    for (int64_t c = 0; c < N; ++c)
        out[c] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double a = orc_value(A, a0 + k, dt);
        for (int64_t c = 0; c < N; ++c)
            out[c] += a * orc_value(W, k * ldw + col0 + c, dt);
    }
}

/* Same, with the row given as fp64 values. */
static void drow_times_matrix(const double *a, int64_t K, const void *W, int dt,
                              int64_t N, double *out)
{
    for (int64_t c = 0; c < N; ++c)
        out[c] = 0.0;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t c = 0; c < N; ++c)
            out[c] += a[k] * orc_value(W, k * N + c, dt);
}

static int check_rows(const int64_t *rows, int64_t n_rows, int64_t M)
{
    if (n_rows < 0 || (n_rows > 0 && !rows))
        return ORC_ERR_ARG;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= M)
            return ORC_ERR_ARG;
    return ORC_OK;
}

/* Activation of one row of first-layer products y (F values, or 2F = [g|u]
 * for SwiGLU) into h (F values). */
static void activate_row(const double *y, int64_t F, int act, double *h)
{
    for (int64_t c = 0; c < F; ++c) {
        if (act == ORC_GELU)
            h[c] = orc_gelu(y[c]);
        else if (act == ORC_SWIGLU)
            h[c] = orc_silu(y[c]) * y[F + c];
        else
            h[c] = y[c];
    }
}

/* Plain linear layer on selected rows: out[r][c] = sum_k A[rows[r]][k] W[k][c],
 * A [M x K], W [K x N]. */
int orc_linear(const void *A, const void *W, int dt, int64_t M, int64_t K, int64_t N,
               const int64_t *rows, int64_t n_rows, double *out)
{
    if (!A || !W || !out || M <= 0 || K <= 0 || N <= 0)
        return ORC_ERR_ARG;
    if (check_rows(rows, n_rows, M))
        return ORC_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r)
        row_times_matrix(A, rows[r] * K, dt, K, W, N, 0, N, out + r * N);
    return ORC_OK;
}

/* ---- the MLP ----------------------------------------------------------- */

/* Unsharded first layer on selected rows: Y[r] = act(X[rows[r]] W1), F values
 * per row (for SwiGLU, SiLU(X Wg) * (X Wu)). */
int orc_colpar_full(const void *X, const void *W1, int dt, int64_t M, int64_t H,
                    int64_t F, int act, const int64_t *rows, int64_t n_rows, double *Y)
{
    if (!X || !W1 || !Y || M <= 0 || H <= 0 || F <= 0 || act < 0 || act > 2)
        return ORC_ERR_ARG;
    if (check_rows(rows, n_rows, M))
        return ORC_ERR_ARG;
    const int64_t ncols = (act == ORC_SWIGLU) ? 2 * F : F;
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        double *y = (double *)malloc((size_t)ncols * sizeof(double));
        if (!y) {
#pragma omp atomic write
            err = ORC_ERR_OOM;
            continue;
        }
        row_times_matrix(X, rows[r] * H, dt, H, W1, ncols, 0, ncols, y);
        activate_row(y, F, act, Y + r * F);
        free(y);
    }
    return err;
}

/* First layer of shard i alone, from the oracle's own copy of the shard:
 * Y_i[r] = act(X[rows[r]] W1_i), F/T values per row. */
int orc_colpar_shard(const void *X, const void *W1, int dt, int64_t M, int64_t H,
                     int64_t F, int T, int act, int i, const int64_t *rows,
                     int64_t n_rows, double *Yi)
{
    if (!X || !W1 || !Yi || M <= 0 || H <= 0 || F <= 0 || T <= 0 || i < 0 || i >= T ||
        act < 0 || act > 2)
        return ORC_ERR_ARG;
    if (F % T != 0)
        return ORC_ERR_INDIVISIBLE;
    if (check_rows(rows, n_rows, M))
        return ORC_ERR_ARG;
    const size_t eb = orc_elem_bytes(dt);
    const int64_t Fs = F / T;
    const int nparts = (act == ORC_SWIGLU) ? 2 : 1;
    /* shard copy: [H x Fs] per part, parts side by side -> [H x nparts*Fs]
       so that the SwiGLU shard reads as [Wg_i | Wu_i]. */
    void *part = malloc((size_t)(H * Fs) * eb);
    void *w1i = malloc((size_t)(H * Fs * nparts) * eb);
    if (!part || !w1i) {
        free(part);
        free(w1i);
        return ORC_ERR_OOM;
    }
    for (int p = 0; p < nparts; ++p) {
        int e = orc_shard_w1(W1, dt, H, F, T, act, i, p, part);
        if (e) {
            free(part);
            free(w1i);
            return e;
        }
        for (int64_t k = 0; k < H; ++k)
            memcpy((char *)w1i + (size_t)(k * nparts * Fs + p * Fs) * eb,
                   (char *)part + (size_t)(k * Fs) * eb, (size_t)Fs * eb);
    }
    free(part);
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        double *y = (double *)malloc((size_t)(nparts * Fs) * sizeof(double));
        if (!y) {
#pragma omp atomic write
            err = ORC_ERR_OOM;
            continue;
        }
        row_times_matrix(X, rows[r] * H, dt, H, w1i, nparts * Fs, 0, nparts * Fs, y);
        activate_row(y, Fs, act, Yi + r * Fs);
        free(y);
    }
    free(w1i);
    return err;
}

/* Unsharded MLP on selected rows (orc_mlp_unsharded, orc_mlp_unsharded_hbf16):
 * h = act(X W1) per row, optionally rounded to bfloat16 (round_h), then h W2. */
static int mlp_unsharded(const void *X, const void *W1, const void *W2, int dt, int64_t M,
                         int64_t H, int64_t F, int act, int round_h, const int64_t *rows,
                         int64_t n_rows, double *Z)
{
    if (!W2 || !Z)
        return ORC_ERR_ARG;
    if (n_rows == 0)
        return check_rows(rows, n_rows, M);
    double *Y = (double *)malloc((size_t)(n_rows * F) * sizeof(double));
    if (!Y)
        return ORC_ERR_OOM;
    int e = orc_colpar_full(X, W1, dt, M, H, F, act, rows, n_rows, Y);
    if (e) {
        free(Y);
        return e;
    }
    if (round_h)
        for (int64_t k = 0; k < n_rows * F; ++k)
            Y[k] = bf16_bits_value(orc_f32_to_bf16((float)Y[k]));
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r)
        drow_times_matrix(Y + r * F, F, W2, dt, H, Z + r * H);
    free(Y);
    return ORC_OK;
}

/* Unsharded MLP on selected rows: Z[r] = act(X[rows[r]] W1) W2, H values per
 * row.  This is the dense result that the sharded computation must equal. */
int orc_mlp_unsharded(const void *X, const void *W1, const void *W2, int dt, int64_t M,
                      int64_t H, int64_t F, int act, const int64_t *rows, int64_t n_rows,
                      double *Z)
{
    return mlp_unsharded(X, W1, W2, dt, M, H, F, act, 0, rows, n_rows, Z);
}

/* The same MLP with the first layer's output rounded to bfloat16 before the
 * second layer reads it, as the workloads store it: the column-parallel
 * output Y_i = act(X W1_i) is the row-parallel layer's input ("Tensor
 * Parallelism in Action", section 1, "Row Parallel (W2)"), a bfloat16 tensor
 * here.  Each fp64 h is rounded to float32 and then to bfloat16, both to
 * nearest even; the second layer is fp64 on those values.  A diagnostic
 * beside orc_mlp_unsharded, which keeps h in fp64: it leaves out the one
 * rounding the method's dtype prescribes, so what remains of a kernel's error
 * is its own arithmetic. */
int orc_mlp_unsharded_hbf16(const void *X, const void *W1, const void *W2, int dt, int64_t M,
                            int64_t H, int64_t F, int act, const int64_t *rows, int64_t n_rows,
                            double *Z)
{
    return mlp_unsharded(X, W1, W2, dt, M, H, F, act, 1, rows, n_rows, Z);
}

/* Sharded MLP: for each shard i (ascending), Y_i = act(X W1_i) and the
 * partial product Z_i = Y_i W2_i from the oracle's own shard copies; then
 * Z = sum_i Z_i (the all-reduce-sum).  Same rows and layout as above. */
int orc_mlp_sharded(const void *X, const void *W1, const void *W2, int dt, int64_t M,
                    int64_t H, int64_t F, int T, int act, const int64_t *rows,
                    int64_t n_rows, double *Z)
{
    if (!X || !W1 || !W2 || !Z || M <= 0 || H <= 0 || F <= 0 || T <= 0)
        return ORC_ERR_ARG;
    if (F % T != 0)
        return ORC_ERR_INDIVISIBLE;
    if (check_rows(rows, n_rows, M))
        return ORC_ERR_ARG;
    const size_t eb = orc_elem_bytes(dt);
    const int64_t Fs = F / T;
    double *Yi = (double *)malloc((size_t)(n_rows * Fs + 1) * sizeof(double));
    double *Zi = (double *)malloc((size_t)(n_rows * H + 1) * sizeof(double));
    void *w2i = malloc((size_t)(Fs * H) * eb);
    if (!Yi || !Zi || !w2i) {
        free(Yi);
        free(Zi);
        free(w2i);
        return ORC_ERR_OOM;
    }
    for (int64_t e = 0; e < n_rows * H; ++e)
        Z[e] = 0.0;
    int err = ORC_OK;
    for (int i = 0; i < T && !err; ++i) {
        err = orc_colpar_shard(X, W1, dt, M, H, F, T, act, i, rows, n_rows, Yi);
        if (!err)
            err = orc_shard_w2(W2, dt, F, H, T, i, w2i);
        if (err)
            break;
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r)
            drow_times_matrix(Yi + r * Fs, Fs, w2i, dt, H, Zi + r * H);
        for (int64_t e = 0; e < n_rows * H; ++e)
            Z[e] += Zi[e];
    }
    free(Yi);
    free(Zi);
    free(w2i);
    return err;
}

/* ---- attention projections --------------------------------------------- */

/* QKV projection of shard i: out[r] = X[rows[r]] Wqkv_i, 3*W values per row
 * ([Q_i | K_i | V_i]), from the oracle's own copy of the shard. */
int orc_qkv_shard(const void *X, const void *Wqkv, int dt, int64_t M, int64_t H,
                  int n_heads, int head_dim, int T, int i, const int64_t *rows,
                  int64_t n_rows, double *out)
{
    if (!X || !Wqkv || !out || M <= 0 || T <= 0 || n_heads <= 0 ||
        (int64_t)n_heads * head_dim != H)
        return ORC_ERR_ARG;
    if (n_heads % T != 0)
        return ORC_ERR_INDIVISIBLE;
    if (check_rows(rows, n_rows, M))
        return ORC_ERR_ARG;
    const size_t eb = orc_elem_bytes(dt);
    const int64_t W = (int64_t)(n_heads / T) * head_dim;
    void *wi = malloc((size_t)(H * 3 * W) * eb);
    if (!wi)
        return ORC_ERR_OOM;
    int e = orc_shard_wqkv(Wqkv, dt, H, n_heads, head_dim, T, i, wi);
    if (!e)
        e = orc_linear(X, wi, dt, M, H, 3 * W, rows, n_rows, out);
    free(wi);
    return e;
}

/* Row-parallel output projection: Z = sum_i A_i Wo_i over shards in
 * ascending order, A [M x H] with the heads side by side (A_i = the columns
 * of shard i's heads), Wo_i the matching rows of Wo. */
int orc_oproj_sharded(const void *A, const void *Wo, int dt, int64_t M, int64_t H,
                      int n_heads, int head_dim, int T, const int64_t *rows,
                      int64_t n_rows, double *Z)
{
    if (!A || !Wo || !Z || M <= 0 || T <= 0 || n_heads <= 0 ||
        (int64_t)n_heads * head_dim != H)
        return ORC_ERR_ARG;
    if (n_heads % T != 0)
        return ORC_ERR_INDIVISIBLE;
    if (check_rows(rows, n_rows, M))
        return ORC_ERR_ARG;
    const size_t eb = orc_elem_bytes(dt);
    const int64_t W = (int64_t)(n_heads / T) * head_dim;
    void *woi = malloc((size_t)(W * H) * eb);
    double *zi = (double *)malloc((size_t)(n_rows * H + 1) * sizeof(double));
    if (!woi || !zi) {
        free(woi);
        free(zi);
        return ORC_ERR_OOM;
    }
    for (int64_t e = 0; e < n_rows * H; ++e)
        Z[e] = 0.0;
    for (int i = 0; i < T; ++i) {
        orc_shard_wo(Wo, dt, H, n_heads, head_dim, T, i, woi);
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r)
            row_times_matrix(A, rows[r] * H + i * W, dt, W, woi, H, 0, H, zi + r * H);
        for (int64_t e = 0; e < n_rows * H; ++e)
            Z[e] += zi[e];
    }
    free(woi);
    free(zi);
    return ORC_OK;
}

/* ---- the all-reduce-sum arithmetic ------------------------------------- */

/* Z[k] = ((P[0][k] + P[1][k]) + ...) + P[T-1][k] in float32, shards in
 * ascending order; P is [T x n].  This fixes the bits the device shard-sum
 * must reproduce. */
void orc_partial_sum_f32(const float *P, int T, int64_t n, float *Z)
{
    for (int64_t k = 0; k < n; ++k) {
        float s = P[k];
        for (int i = 1; i < T; ++i)
            s = s + P[(int64_t)i * n + k];
        Z[k] = s;
    }
}

/* Threads the OpenMP runtime would use. */
int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- the other collectives named for tensor parallelism ------------------
 * "Tensor Parallelism in Action", section 2, question 3 names AllReduce,
 * AllGather and ReduceScatter; the "Tensor parallelism" guide's ring byte
 * count 2 (T - 1) / T * H * B is a reduce-scatter half followed by an
 * all-gather half.  With all T ranks on one device: */

/* Reduce-scatter: rank i receives block i (n/T values) of the sum over ranks,
 * out[i][k] = ((P[0][i nb + k] + P[1][i nb + k]) + ...) in float32. */
int orc_reduce_scatter_f32(const float *P, int T, int64_t n, float *out)
{
    if (!P || !out || T <= 0 || n < 0)
        return ORC_ERR_ARG;
    if (n % T != 0)
        return ORC_ERR_INDIVISIBLE;
    const int64_t nb = n / T;
    for (int i = 0; i < T; ++i)
        for (int64_t k = 0; k < nb; ++k) {
            float s = P[i * nb + k];
            for (int j = 1; j < T; ++j)
                s = s + P[(int64_t)j * n + i * nb + k];
            out[(int64_t)i * nb + k] = s;
        }
    return ORC_OK;
}

/* All-gather: the T blocks of nb elements each, concatenated in rank order. */
int orc_all_gather(const void *parts, int T, int64_t nb, int elem_bytes, void *out)
{
    if (!parts || !out || T <= 0 || nb < 0 || elem_bytes <= 0)
        return ORC_ERR_ARG;
    memcpy(out, parts, (size_t)(T * nb) * (size_t)elem_bytes);
    return ORC_OK;
}

/* float32 -> bfloat16 bits, round to nearest, ties to even (finite inputs). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    const uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

/* All-reduce-sum with a bfloat16 result: the float32 ascending-order sum,
 * rounded once to bfloat16. */
void orc_partial_sum_bf16(const float *P, int T, int64_t n, uint16_t *Z)
{
    for (int64_t k = 0; k < n; ++k) {
        float s = P[k];
        for (int i = 1; i < T; ++i)
            s = s + P[(int64_t)i * n + k];
        Z[k] = orc_f32_to_bf16(s);
    }
}

/* ---- backward of the tensor-parallel MLP -------------------------------
 * "Slice the matrix itself", section "Strict NVLink Domain Constraint": the
 * all-reduces run on every layer's forward AND backward pass; the duoan.github.io
 * teaser: a layer contract says "which gradient path communicates".  For
 * Z = act(X W1) W2 and an upstream gradient dZ, with P = X W1 the
 * pre-activation and Hh = act(P):
 *   dH = dZ W2^T            (per shard: dH_i = dZ W2_i^T, no exchange)
 *   dP = dH * act'(P)        (elementwise; SwiGLU: dG = dH u SiLU'(g), dU = dH SiLU(g))
 *   dW2 = Hh^T dZ            (row block i = Hh_i^T dZ, local)
 *   dW1 = X^T dP             (column block i = X^T dP_i, local)
 *   dX = dP W1^T = sum_i dP_i W1_i^T   (the backward all-reduce-sum)
 * GeLU'(y) = Phi(y) + y phi(y); SiLU'(g) = s (1 + g (1 - s)), s = 1/(1+e^-g). */

double orc_gelu_grad(double y)
{
    const double pi = 3.14159265358979323846;
    return 0.5 * (1.0 + erf(y / sqrt(2.0))) + y * exp(-0.5 * y * y) / sqrt(2.0 * pi);
}

double orc_silu_grad(double g)
{
    const double s = 1.0 / (1.0 + exp(-g));
    return s * (1.0 + g * (1.0 - s));
}

/* For one token row r: P (ncols = F or 2F values), dH (F values), and
 * dP (ncols values: for SwiGLU [dG | dU]) and Hh (F values). */
static void token_backward(const void *X, const void *W1, const void *W2, const void *dZ, int dt,
                           int64_t H, int64_t F, int act, int64_t r, double *P, double *dH,
                           double *dP, double *Hh)
{
    const int64_t ncols = (act == ORC_SWIGLU) ? 2 * F : F;
    row_times_matrix(X, r * H, dt, H, W1, ncols, 0, ncols, P);
    /* dH[f] = sum_h dZ[r][h] W2[f][h] */
    for (int64_t f = 0; f < F; ++f) {
        double acc = 0.0;
        for (int64_t h = 0; h < H; ++h)
            acc += orc_value(dZ, r * H + h, dt) * orc_value(W2, f * H + h, dt);
        dH[f] = acc;
    }
    for (int64_t f = 0; f < F; ++f) {
        if (act == ORC_GELU) {
            dP[f] = dH[f] * orc_gelu_grad(P[f]);
            Hh[f] = orc_gelu(P[f]);
        } else if (act == ORC_SWIGLU) {
            const double g = P[f], u = P[F + f];
            dP[f] = dH[f] * u * orc_silu_grad(g);
            dP[F + f] = dH[f] * orc_silu(g);
            Hh[f] = orc_silu(g) * u;
        } else {
            dP[f] = dH[f];
            Hh[f] = P[f];
        }
    }
}

/* dX on selected token rows: dX[r][h] = sum_c dP[r][c] W1[h][c]. */
int orc_mlp_backward_dx(const void *X, const void *W1, const void *W2, const void *dZ, int dt,
                        int64_t M, int64_t H, int64_t F, int act, const int64_t *rows,
                        int64_t n_rows, double *dX)
{
    if (!X || !W1 || !W2 || !dZ || !dX || M <= 0 || H <= 0 || F <= 0 || act < 0 || act > 2)
        return ORC_ERR_ARG;
    if (check_rows(rows, n_rows, M))
        return ORC_ERR_ARG;
    const int64_t ncols = (act == ORC_SWIGLU) ? 2 * F : F;
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_rows; ++i) {
        double *buf = (double *)malloc((size_t)(ncols * 2 + F * 2) * sizeof(double));
        if (!buf) {
#pragma omp atomic write
            err = ORC_ERR_OOM;
            continue;
        }
        double *P = buf, *dP = buf + ncols, *dH = buf + 2 * ncols, *Hh = dH + F;
        token_backward(X, W1, W2, dZ, dt, H, F, act, rows[i], P, dH, dP, Hh);
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t c = 0; c < ncols; ++c)
                acc += dP[c] * orc_value(W1, h * ncols + c, dt);
            dX[i * H + h] = acc;
        }
        free(buf);
    }
    return err;
}

/* Weight gradients on selected FFN columns f (for SwiGLU, f names the pair
 * gate column f / up column F + f):
 *   dW1c[k][j] = sum_m X[m][k] dP[m][f_j]    (and dW1c_up for the up column),
 *   dW2r[j][h] = sum_m Hh[m][f_j] dZ[m][h].
 * dW1c is [H x n] (SwiGLU: [H x 2n], gate columns then up columns),
 * dW2r is [n x H].  Every token contributes. */
int orc_mlp_backward_dw(const void *X, const void *W1, const void *W2, const void *dZ, int dt,
                        int64_t M, int64_t H, int64_t F, int act, const int64_t *fcols,
                        int64_t n, double *dW1c, double *dW2r)
{
    if (!X || !W1 || !W2 || !dZ || !dW1c || !dW2r || M <= 0 || H <= 0 || F <= 0 || act < 0 ||
        act > 2 || n < 0 || (n > 0 && !fcols))
        return ORC_ERR_ARG;
    for (int64_t j = 0; j < n; ++j)
        if (fcols[j] < 0 || fcols[j] >= F)
            return ORC_ERR_ARG;
    const int64_t ncols = (act == ORC_SWIGLU) ? 2 * F : F;
    const int nparts = (act == ORC_SWIGLU) ? 2 : 1;
    /* per token, the values of dP and Hh at the selected columns */
    double *dPs = (double *)calloc((size_t)(M * n * nparts + 1), sizeof(double));
    double *Hs = (double *)calloc((size_t)(M * n + 1), sizeof(double));
    if (!dPs || !Hs) {
        free(dPs);
        free(Hs);
        return ORC_ERR_OOM;
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t j = 0; j < n; ++j) {
            const int64_t f = fcols[j];
            double p[2] = {0.0, 0.0}, dh = 0.0;
            for (int part = 0; part < nparts; ++part)
                for (int64_t k = 0; k < H; ++k)
                    p[part] += orc_value(X, m * H + k, dt) * orc_value(W1, k * ncols + part * F + f, dt);
            for (int64_t h = 0; h < H; ++h)
                dh += orc_value(dZ, m * H + h, dt) * orc_value(W2, f * H + h, dt);
            if (act == ORC_GELU) {
                dPs[(m * n + j) * nparts] = dh * orc_gelu_grad(p[0]);
                Hs[m * n + j] = orc_gelu(p[0]);
            } else if (act == ORC_SWIGLU) {
                dPs[(m * n + j) * 2] = dh * p[1] * orc_silu_grad(p[0]);
                dPs[(m * n + j) * 2 + 1] = dh * orc_silu(p[0]);
                Hs[m * n + j] = orc_silu(p[0]) * p[1];
            } else {
                dPs[m * n + j] = dh;
                Hs[m * n + j] = p[0];
            }
        }
    }
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t k = 0; k < H; ++k)
        for (int part = 0; part < nparts; ++part)
            for (int64_t j = 0; j < n; ++j) {
                double acc = 0.0;
                for (int64_t m = 0; m < M; ++m)
                    acc += orc_value(X, m * H + k, dt) * dPs[(m * n + j) * nparts + part];
                dW1c[k * n * nparts + part * n + j] = acc;
            }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < n; ++j)
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m)
                acc += Hs[m * n + j] * orc_value(dZ, m * H + h, dt);
            dW2r[j * H + h] = acc;
        }
    free(dPs);
    free(Hs);
    return ORC_OK;
}

/* ---- one tensor-parallel transformer block ---------------------------------
 * "Slice the matrix itself", section "All-Reduce Synchronization": a block
 * needs two all-reduces, one after the attention's row-parallel projection
 * and one after the MLP's; the "Tensor parallelism" guide, section "Walking
 * through a transformer block": heads are sharded across ranks, and the two
 * all-reduces sit on the attention and MLP residual paths.  Readings: causal
 * scaled-dot-product attention per head, softmax(q k^T / sqrt(hd)) v; a
 * residual add after each all-reduce; no normalisation layers (the pages
 * name none).  For token r:
 *   q, k_j, v_j = x_r Wq, x_j Wk, x_j Wv   (per head h: columns [h hd, (h+1) hd))
 *   o_h = sum_{j <= r} softmax_j(q_h . k_jh / sqrt(hd)) v_jh
 *   a = sum over shards i of (o of shard i's heads) Wo_i   (all-reduce 1)
 *   h_r = x_r + a
 *   out_r = h_r + sum_i act(h_r W1_i) W2_i                  (all-reduce 2)
 * When `sharded`, each shard's heads and MLP columns are computed from the
 * oracle's own shard copies and the partial products summed in shard order;
 * otherwise the dense matrices are used.  hout (may be NULL) receives h. */
int orc_block_forward(const void *X, const void *Wqkv, const void *Wo, const void *W1,
                      const void *W2, int dt, int64_t M, int64_t H, int n_heads, int head_dim,
                      int64_t F, int act, int causal, int T, int sharded, const int64_t *rows,
                      int64_t n_rows, double *out, double *hout)
{
    if (!X || !Wqkv || !Wo || !W1 || !W2 || !out || M <= 0 || H <= 0 || F <= 0 || T <= 0 ||
        n_heads <= 0 || head_dim <= 0 || (int64_t)n_heads * head_dim != H)
        return ORC_ERR_ARG;
    if (n_heads % T != 0 || F % T != 0)
        return ORC_ERR_INDIVISIBLE;
    if (check_rows(rows, n_rows, M))
        return ORC_ERR_ARG;
    int64_t kmax = 0; /* keys needed: rows [0, kmax) */
    for (int64_t i = 0; i < n_rows; ++i)
        if (rows[i] + 1 > kmax)
            kmax = rows[i] + 1;
    if (!causal)
        kmax = M;
    /* K and V of every needed key token, [kmax x H] each, fp64 */
    double *K = (double *)malloc((size_t)(kmax * H + 1) * sizeof(double));
    double *V = (double *)malloc((size_t)(kmax * H + 1) * sizeof(double));
    if (!K || !V) {
        free(K);
        free(V);
        return ORC_ERR_OOM;
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t j = 0; j < kmax; ++j) {
        row_times_matrix(X, j * H, dt, H, Wqkv, 3 * H, H, H, K + j * H);
        row_times_matrix(X, j * H, dt, H, Wqkv, 3 * H, 2 * H, H, V + j * H);
    }
    const int hps = n_heads / T;
    const int64_t W = (int64_t)hps * head_dim, Fs = F / T;
    const int64_t ncols = (act == ORC_SWIGLU) ? 2 * F : F;
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t r = rows[i];
        const int64_t nk = causal ? r + 1 : M;
        double *buf = (double *)malloc((size_t)(3 * H + nk + ncols + F) * sizeof(double));
        if (!buf) {
#pragma omp atomic write
            err = ORC_ERR_OOM;
            continue;
        }
        double *q = buf, *o = buf + H, *h = buf + 2 * H, *p = buf + 3 * H, *y = p + nk, *hh = y + ncols;
        row_times_matrix(X, r * H, dt, H, Wqkv, 3 * H, 0, H, q);
        for (int hd_i = 0; hd_i < n_heads; ++hd_i) {
            const int64_t c0 = (int64_t)hd_i * head_dim;
            double mx = -INFINITY;
            for (int64_t j = 0; j < nk; ++j) {
                double sdot = 0.0;
                for (int d = 0; d < head_dim; ++d)
                    sdot += q[c0 + d] * K[j * H + c0 + d];
                p[j] = sdot / sqrt((double)head_dim);
                if (p[j] > mx)
                    mx = p[j];
            }
            double sum = 0.0;
            for (int64_t j = 0; j < nk; ++j) {
                p[j] = exp(p[j] - mx);
                sum += p[j];
            }
            for (int d = 0; d < head_dim; ++d) {
                double acc = 0.0;
                for (int64_t j = 0; j < nk; ++j)
                    acc += p[j] * V[j * H + c0 + d];
                o[c0 + d] = acc / sum;
            }
        }
        /* all-reduce 1: a = sum over shards of o_i Wo_i (or the dense o Wo) */
        for (int64_t c = 0; c < H; ++c)
            h[c] = 0.0;
        const int nsh = sharded ? T : 1;
        const int64_t Wsh = sharded ? W : H;
        for (int sidx = 0; sidx < nsh; ++sidx) {
            for (int64_t c = 0; c < H; ++c) {
                double acc = 0.0;
                for (int64_t k = 0; k < Wsh; ++k)
                    acc += o[sidx * Wsh + k] * orc_value(Wo, (sidx * Wsh + k) * H + c, dt);
                h[c] += acc;
            }
        }
        for (int64_t c = 0; c < H; ++c)
            h[c] += orc_value(X, r * H + c, dt);
        if (hout)
            for (int64_t c = 0; c < H; ++c)
                hout[i * H + c] = h[c];
        /* all-reduce 2: the MLP on h */
        const int64_t Fb = sharded ? Fs : F;
        for (int64_t c = 0; c < H; ++c)
            out[i * H + c] = 0.0;
        for (int sidx = 0; sidx < (sharded ? T : 1); ++sidx) {
            const int nparts = (act == ORC_SWIGLU) ? 2 : 1;
            for (int part = 0; part < nparts; ++part)
                for (int64_t f = 0; f < Fb; ++f) {
                    double acc = 0.0;
                    for (int64_t k = 0; k < H; ++k)
                        acc += h[k] * orc_value(W1, k * ncols + part * F + sidx * Fb + f, dt);
                    y[part * Fb + f] = acc;
                }
            activate_row(y, Fb, act, hh);
            for (int64_t c = 0; c < H; ++c) {
                double acc = 0.0;
                for (int64_t f = 0; f < Fb; ++f)
                    acc += hh[f] * orc_value(W2, (sidx * Fb + f) * H + c, dt);
                out[i * H + c] += acc;
            }
        }
        for (int64_t c = 0; c < H; ++c)
            out[i * H + c] += h[c];
        free(buf);
    }
    free(K);
    free(V);
    return err;
}

/* ---- attention core per head -----------------------------------------------
 * "Tensor parallelism" guide, section "Walking through a transformer block":
 * heads are sharded across ranks, so each head's attention is computed on the
 * shard that owns it.  Reading (as for the block): scaled dot-product
 * attention, causal or over all keys.  For head h and token r:
 *   s_j = q_r . k_j / sqrt(hd),  w_j = exp(s_j - max_j s_j),
 *   o_r = sum_j w_j v_j / sum_j w_j
 * over keys j <= r (causal) or j < M.  Q, K and V are head-major
 * [n_heads][M][hd]; out is [n_rows][n_heads hd], heads side by side. */
int orc_attention(const void *Q, const void *K, const void *V, int dt, int64_t M, int n_heads,
                  int head_dim, int causal, const int64_t *rows, int64_t n_rows, double *out)
{
    if (!Q || !K || !V || !out || M <= 0 || n_heads <= 0 || head_dim <= 0)
        return ORC_ERR_ARG;
    if (check_rows(rows, n_rows, M))
        return ORC_ERR_ARG;
    const int64_t width = (int64_t)n_heads * head_dim;
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t r = rows[i];
        const int64_t nk = causal ? r + 1 : M;
        double *s = (double *)malloc((size_t)nk * sizeof(double));
        if (!s) {
#pragma omp atomic write
            err = ORC_ERR_OOM;
            continue;
        }
        for (int h = 0; h < n_heads; ++h) {
            const int64_t base = (int64_t)h * M * head_dim;
            double mx = -INFINITY;
            for (int64_t j = 0; j < nk; ++j) {
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d)
                    dot += orc_value(Q, base + r * head_dim + d, dt) *
                           orc_value(K, base + j * head_dim + d, dt);
                s[j] = dot / sqrt((double)head_dim);
                if (s[j] > mx)
                    mx = s[j];
            }
            double den = 0.0;
            for (int64_t j = 0; j < nk; ++j) {
                s[j] = exp(s[j] - mx);
                den += s[j];
            }
            for (int d = 0; d < head_dim; ++d) {
                double num = 0.0;
                for (int64_t j = 0; j < nk; ++j)
                    num += s[j] * orc_value(V, base + j * head_dim + d, dt);
                out[i * width + (int64_t)h * head_dim + d] = num / den;
            }
        }
        free(s);
    }
    return err;
}
