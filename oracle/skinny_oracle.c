/*
 * skinny_oracle.c -- the CPU oracle for the skinny BF16 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline / reference leg may load this code.  The product path
 * (the CUDA library under latency_skinny_bf16_gb300/) never calls it, links it
 * or shares code with it; there is no CPU fallback.
 *
 * What it computes.  The pages describe the low-latency router GEMM
 * ("[Perf][Feat] Add generic cuteDSL LL BF16 router (GEMM)", vllm PR #42562
 * report, section "Implementation breakdown" items 1-2 and the
 * _ll_bf16_dotprod.py / _ll_bf16_splitk.py snippets) and the decode-time
 * bf16_skinny_gemm projections ("GLM-5.2 Blackwell decode optimizations",
 * vllm PR #48597, section "Implementation breakdown" item 3): for token m and
 * output column (expert / projection row) n,
 *
 *     Y[m][n] = sum_k  float(X[m][k]) * float(W[n][k])
 *
 * with X [M,K] and W [N,K] in bf16, the products and the accumulator in a
 * wider type (the pages: fp32 acc_dtype, fp32 out_dtype).  That is exactly a
 * matrix product Y = X . W^T.  The oracle writes the definition out with no
 * blocking, fusion or reordering: decode each bf16 input exactly, multiply in
 * fp64 (exact: two 8-bit significands give at most 16 bits), and add the
 * products in ascending k in fp64.
 *
 * Companion output A[m][n] = sum_k |x*w| feeds the elementwise tolerance
 * |y - y_ref| <= 1e-5 * A + 1e-6 that the parity tests apply.
 *
 * Plain C99, host compiler only, no CUDA header.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

/* bfloat16 is the upper half of an IEEE-754 binary32: sign, 8 exponent bits
 * (bias 127), 7 stored significand bits.  Decoding is exact: place the 16 bits
 * in the high half of a binary32 word and reinterpret; the binary32 value
 * widens to binary64 exactly. */
double skinny_oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t word = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* Y[m*ldy + n] = sum_{k<K} x(m,k) * w(n,k) in fp64, ascending k.
 * A (may be NULL) receives sum_{k<K} |x(m,k) * w(n,k)| at A[m*lda + n].
 * X is [M rows, ldx stride], W is [N rows, ldw stride]; both bf16 bit
 * patterns.  K == 0 gives Y = 0 (the empty sum).  Entries of Y outside
 * m<M, n<N are never touched. */
void skinny_oracle_gemm(const uint16_t *X, int64_t ldx,
                        const uint16_t *W, int64_t ldw,
                        double *Y, int64_t ldy,
                        double *A, int64_t lda,
                        int M, int N, int K)
{
    for (int m = 0; m < M; ++m) {
        const uint16_t *xrow = X + (int64_t)m * ldx;
        for (int n = 0; n < N; ++n) {
            const uint16_t *wrow = W + (int64_t)n * ldw;
            double sum = 0.0;
            double abs_sum = 0.0;
            for (int k = 0; k < K; ++k) {
                double prod = skinny_oracle_bf16_to_f64(xrow[k]) *
                              skinny_oracle_bf16_to_f64(wrow[k]);
                sum += prod;
                abs_sum += fabs(prod);
            }
            Y[(int64_t)m * ldy + n] = sum;
            if (A) A[(int64_t)m * lda + n] = abs_sum;
        }
    }
}

/* The same definition evaluated only at `count` sampled output positions
 * (rows[i], cols[i]); used to check full-size launches without computing all
 * of Y.  y[i] and a[i] receive the value and the absolute-product sum. */
void skinny_oracle_gemm_points(const uint16_t *X, int64_t ldx,
                               const uint16_t *W, int64_t ldw,
                               int K, const int32_t *rows, const int32_t *cols,
                               int count, double *y, double *a)
{
    for (int i = 0; i < count; ++i) {
        const uint16_t *xrow = X + (int64_t)rows[i] * ldx;
        const uint16_t *wrow = W + (int64_t)cols[i] * ldw;
        double sum = 0.0;
        double abs_sum = 0.0;
        for (int k = 0; k < K; ++k) {
            double prod = skinny_oracle_bf16_to_f64(xrow[k]) *
                          skinny_oracle_bf16_to_f64(wrow[k]);
            sum += prod;
            abs_sum += fabs(prod);
        }
        y[i] = sum;
        if (a) a[i] = abs_sum;
    }
}

/* Router epilogue (the consumer of the router logits: "[Perf][Feat] Add
 * generic cuteDSL LL BF16 router (GEMM)", section "Implementation breakdown"
 * item 4, the MoE gate's forward; the pages print no epilogue, so this is the
 * plainest one): for each token m, the softmax of its N logits and the k
 * experts of largest probability.
 *
 *   p_n = exp(l_n - l_max) / sum_j exp(l_j - l_max)          (fp64)
 *   ids  = the k indices of the largest logits, in descending order of the
 *          logit as given (float32), equal logits by ascending index; a NaN
 *          logit ranks below every other value (-inf included), and NaNs
 *          among themselves by ascending index
 *   weights[i] = p_{ids[i]}, or with renormalize != 0
 *   weights[i] = p_{ids[i]} / sum_{i'<k} p_{ids[i']}
 *
 * l_max is the largest logit that is not NaN (-inf when there is none).  The
 * arithmetic is IEEE: a NaN or +inf logit makes the sum NaN, so every weight
 * of that token is NaN, while its ids stay well defined (the pages say nothing
 * on non-finite logits; this is the plain IEEE reading).  Selection is made on
 * the float32 logits exactly as given (the same values the GPU kernel
 * compares), by k passes of "highest-ranked not yet chosen" over the row;
 * 1 <= k <= N. */
static int topk_ranks_above(float v, int n, float b, int nb)
{
    const int vnan = isnan(v), bnan = isnan(b);
    if (vnan != bnan) return bnan;
    if (!vnan && v != b) return v > b;
    return n < nb;
}

void skinny_oracle_router_topk(const float *L, int64_t ldl, int M, int N, int k, int renormalize,
                               double *weights, int64_t ldwt, int32_t *ids, int64_t ldid,
                               unsigned char *taken /* N bytes of scratch */)
{
    for (int m = 0; m < M; ++m) {
        const float *row = L + (int64_t)m * ldl;
        float lmax = -INFINITY;
        for (int n = 0; n < N; ++n)
            if (!isnan(row[n]) && row[n] > lmax) lmax = row[n];
        double denom = 0.0;
        for (int n = 0; n < N; ++n) denom += exp((double)row[n] - (double)lmax);
        memset(taken, 0, (size_t)N);
        double chosen = 0.0;
        for (int i = 0; i < k; ++i) {
            int best = -1;
            for (int n = 0; n < N; ++n)
                if (!taken[n] && (best < 0 || topk_ranks_above(row[n], n, row[best], best))) best = n;
            taken[best] = 1;
            ids[(int64_t)m * ldid + i] = best;
            const double pv = exp((double)row[best] - (double)lmax) / denom;
            weights[(int64_t)m * ldwt + i] = pv;
            chosen += pv;
        }
        if (renormalize)
            for (int i = 0; i < k; ++i) weights[(int64_t)m * ldwt + i] /= chosen;
    }
}

/* fp32 router weights ("GLM-5.2 Blackwell decode optimizations": the router
 * GEMM keeps fp32 weights for the model family that needs them, FP32 router
 * GEMM shape support): the same definition with W in fp32,
 *
 *     Y[m][n] = sum_k  float(X[m][k]) * W[n][k]        X bf16, W fp32
 *
 * Each product of an 8-bit and a 24-bit significand is exact in fp64; the
 * products are added in ascending k in fp64.  A (may be NULL) receives
 * sum_k |x * w|. */
void skinny_oracle_gemm_f32w(const uint16_t *X, int64_t ldx,
                             const float *W, int64_t ldw,
                             double *Y, int64_t ldy,
                             double *A, int64_t lda,
                             int M, int N, int K)
{
    for (int i = 0; i < M; ++i) {
        const uint16_t *xr = X + (int64_t)i * ldx;
        for (int j = 0; j < N; ++j) {
            const float *wr = W + (int64_t)j * ldw;
            double acc = 0.0, acc_abs = 0.0;
            for (int kk = 0; kk < K; ++kk) {
                const double t = skinny_oracle_bf16_to_f64(xr[kk]) * (double)wr[kk];
                acc += t;
                acc_abs += fabs(t);
            }
            Y[(int64_t)i * ldy + j] = acc;
            if (A) A[(int64_t)i * lda + j] = acc_abs;
        }
    }
}

/* RMS norm of the query latent before the q_b projection ("GLM-5.2 Blackwell
 * decode optimizations", section "Implementation breakdown" item 2 and the
 * fused_norm_rope snippet's pid == 2 branch: q_c = _rms_norm(q_c,
 * q_rms_norm_w, eps, Q_DIM), stored to q_c_out): for each token m,
 *
 *     r_m   = 1 / sqrt( (1/K) sum_k x(m,k)^2 + eps )
 *     xn(m,k) = x(m,k) * r_m * g(k)
 *
 * all in fp64 (x and g decoded exactly from bf16).  The value is returned
 * unrounded in XN (the bf16 rounding of the stored q_c_out is left to the
 * caller, which also needs to know how close each value is to a rounding
 * boundary). */
void skinny_oracle_rmsnorm(const uint16_t *X, int64_t ldx, const uint16_t *G, double eps,
                           int M, int K, double *XN, int64_t ldxn)
{
    for (int m = 0; m < M; ++m) {
        const uint16_t *xm = X + (int64_t)m * ldx;
        double ss = 0.0;
        for (int k = 0; k < K; ++k) {
            const double v = skinny_oracle_bf16_to_f64(xm[k]);
            ss += v * v;
        }
        const double r = 1.0 / sqrt(ss / (double)K + eps);
        for (int k = 0; k < K; ++k)
            XN[(int64_t)m * ldxn + k] = skinny_oracle_bf16_to_f64(xm[k]) * r * skinny_oracle_bf16_to_f64(G[k]);
    }
}
