/*
 * CPU oracle for the quantized tensor-core GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library or its Python
 * binding may load, link or call this file.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg use it.  It shares no code,
 * header, table or constant with the CUDA path.
 *
 * Every function is the plain definition of what the path computes, written
 * as straight loops: integer results accumulate in int64, floating-point
 * results in double.  No blocking, no reordering beyond the definition.
 * Callers may split work over output rows (each row is independent).
 *
 * Sources (web pages on the subject):
 *  [L4]   "Hand-Written PTX Tensor-Core GEMM Kernels: A Multi-Precision Study
 *          on NVIDIA L4" (arXiv 2608.10103), abstract: FP16, INT8 and INT4
 *          GEMM, square N = 512..8192.
 *  [SM75] "fused-int4-gemm-sm75" README: INT4 weight-only linear, packed INT4
 *          weights, sign extension, register dequantization, per-group scales
 *          with group_size = 128 ("AWQ-Compatible Scales").
 *  [W4A4] "Warp-Specialized Kernel Implementation for W4A4 MatMul on Latest
 *          GPU Architectures", section 1 (Problem Definition):
 *          Y = (Q(X) . Q(W)^T) (.) scale + L(X) + b.
 *
 * Data layouts (fixed by the workload definitions):
 *  A, X    : M x K, row-major (K contiguous), leading dimension in elements
 *            (in bytes for packed 4-bit data).
 *  B, W    : N x K, row-major (= K-major), same convention.
 *  C, Y    : M x N, row-major.
 *  s4p     : two signed 4-bit values per byte along K; the LOW nibble holds
 *            the even k, the HIGH nibble the odd k; two's complement nibble.
 *  fp16    : IEEE binary16, passed as raw uint16_t bit patterns.
 *
 * Return values: 0 on success, nonzero on a detected error (argument out of
 * range, int32 overflow of an integer result).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- IEEE binary16 conversions through the compiler's _Float16 type ---- */

double orc_half_to_double(uint16_t h)
{
    _Float16 f;
    memcpy(&f, &h, sizeof f);
    return (double)f;
}

/* Round-to-nearest-even conversion of a binary32 value to binary16. */
uint16_t orc_float_to_half(float x)
{
    _Float16 f = (_Float16)x;
    uint16_t h;
    memcpy(&h, &f, sizeof h);
    return h;
}

/* Round-to-nearest-even conversion of a binary64 value to binary16 (one
 * rounding, not via binary32). */
uint16_t orc_double_to_half(double x)
{
    _Float16 f = (_Float16)x;
    uint16_t h;
    memcpy(&h, &f, sizeof h);
    return h;
}

/* ---- 4-bit packing [L4] INT4 GEMM operands, [SM75] INT4 packing ---- */

/* Value of one two's-complement nibble n (0..15): n < 8 -> n, else n - 16. */
static int nibble_value(unsigned n)
{
    n &= 0xFu;
    return n < 8u ? (int)n : (int)n - 16;
}

/* V[r][k] = signed value of nibble k of row r of P.  k even -> low nibble of
 * byte k/2, k odd -> high nibble. */
int orc_s4_unpack(int64_t rows, int64_t K, const uint8_t *P, int64_t ldp,
                  int8_t *V, int64_t ldv)
{
    if (rows < 0 || K < 0 || (K & 1) || ldp < K / 2 || ldv < K)
        return 1;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = P[r * ldp + k / 2];
            unsigned n = (k % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
            V[r * ldv + k] = (int8_t)nibble_value(n);
        }
    return 0;
}

/* Inverse of orc_s4_unpack.  Every value must lie in [-8, 7]. */
int orc_s4_pack(int64_t rows, int64_t K, const int8_t *V, int64_t ldv,
                uint8_t *P, int64_t ldp)
{
    if (rows < 0 || K < 0 || (K & 1) || ldp < K / 2 || ldv < K)
        return 1;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; k += 2) {
            int lo = V[r * ldv + k], hi = V[r * ldv + k + 1];
            if (lo < -8 || lo > 7 || hi < -8 || hi > 7)
                return 2;
            P[r * ldp + k / 2] =
                (uint8_t)(((unsigned)lo & 0xFu) | (((unsigned)hi & 0xFu) << 4));
        }
    return 0;
}

/* ---- [L4] exact INT8 GEMM: C[i][j] = sum_k A[i][k] * B[j][k] ---- */

int orc_gemm_s8(int64_t M, int64_t N, int64_t K,
                const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                int32_t *C, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || ldc < N)
        return 1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            int64_t acc = 0;
            for (int64_t k = 0; k < K; ++k)
                acc += (int64_t)A[i * lda + k] * (int64_t)B[j * ldb + k];
            if (acc < INT32_MIN || acc > INT32_MAX)
                return 3;
            C[i * ldc + j] = (int32_t)acc;
        }
    return 0;
}

/* ---- [L4] exact INT4 GEMM: unpack both operands, then the INT8 definition ---- */

int orc_gemm_s4(int64_t M, int64_t N, int64_t K,
                const uint8_t *A, int64_t lda_bytes,
                const uint8_t *B, int64_t ldb_bytes,
                int32_t *C, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0 || (K & 1) || lda_bytes < K / 2 ||
        ldb_bytes < K / 2 || ldc < N)
        return 1;
    int8_t *Au = (int8_t *)malloc((size_t)(M * K + 1));
    int8_t *Bu = (int8_t *)malloc((size_t)(N * K + 1));
    int rc = 4;
    if (Au && Bu) {
        rc = orc_s4_unpack(M, K, A, lda_bytes, Au, K);
        if (!rc)
            rc = orc_s4_unpack(N, K, B, ldb_bytes, Bu, K);
        if (!rc)
            rc = orc_gemm_s8(M, N, K, Au, K, Bu, K, C, ldc);
    }
    free(Au);
    free(Bu);
    return rc;
}

/* ---- [L4] FP16 GEMM with wide accumulation: C = A . B^T in double ---- */

int orc_gemm_f16(int64_t M, int64_t N, int64_t K,
                 const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                 double *C, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || ldc < N)
        return 1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += orc_half_to_double(A[i * lda + k]) *
                       orc_half_to_double(B[j * ldb + k]);
            C[i * ldc + j] = acc;
        }
    return 0;
}

/* ---- [SM75] W4A16 weight-only linear ----
 * Y[m][n] = sum_k X[m][k] * (q[n][k] * s[n][k / group]).
 * q: s4p, N x K (K-major).  s: fp16, N x (K / group), leading dim lds.
 * The weight is dequantized in exact arithmetic (double) and the product is
 * summed in double: dequantize-then-GEMM. */
int orc_w4a16(int64_t M, int64_t N, int64_t K,
              const uint16_t *X, int64_t ldx,
              const uint8_t *Wq, int64_t ldw_bytes,
              const uint16_t *S, int64_t lds, int64_t group,
              double *Y, int64_t ldy)
{
    if (M < 0 || N < 0 || K < 0 || (K & 1) || group <= 0 || K % group ||
        ldx < K || ldw_bytes < K / 2 || lds < K / group || ldy < N)
        return 1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                uint8_t byte = Wq[n * ldw_bytes + k / 2];
                int q = nibble_value((k % 2 == 0) ? byte : (unsigned)byte >> 4);
                double w = (double)q * orc_half_to_double(S[n * lds + k / group]);
                acc += orc_half_to_double(X[m * ldx + k]) * w;
            }
            Y[m * ldy + n] = acc;
        }
    return 0;
}

/* ---- [W4A4] Q(.): per-row, per-K-block symmetric absmax 4-bit quantizer ----
 * For row m and block j (k in [j*block, (j+1)*block)):
 *   a = max |x| over the block, in binary32;
 *   s = binary16(a / 7), a / 7 an IEEE binary32 division, rounded to nearest
 *       even into binary16;
 *   q = 0 if s == 0, else clamp(rint(x / s), -8, 7) with x / s an IEEE
 *       binary32 division by the rounded scale and rint round-half-even.
 * The page names Q(.) only as "4-bit quantization"; this symmetric absmax
 * reading with divisor 7 is the plainest one consistent with per-block scale
 * factors.  Output: q packed s4p (M x K/2 bytes), s as fp16 (M x K/block). */
int orc_w4a4_quantize(int64_t M, int64_t K, const float *X, int64_t ldx,
                      int64_t block, uint8_t *Q, int64_t ldq_bytes,
                      uint16_t *S, int64_t lds)
{
    if (M < 0 || K < 0 || block <= 0 || (block & 1) || K % block ||
        ldx < K || ldq_bytes < K / 2 || lds < K / block)
        return 1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < K / block; ++j) {
            const float *x = X + m * ldx + j * block;
            float a = 0.0f;
            for (int64_t t = 0; t < block; ++t) {
                float v = fabsf(x[t]);
                if (v > a)
                    a = v;
            }
            uint16_t sh = orc_float_to_half(a / 7.0f);
            S[m * lds + j] = sh;
            float s = (float)orc_half_to_double(sh);
            for (int64_t t = 0; t < block; t += 2) {
                int q[2];
                for (int u = 0; u < 2; ++u) {
                    if (s == 0.0f) {
                        q[u] = 0;
                    } else {
                        float r = rintf(x[t + u] / s);
                        if (r < -8.0f) r = -8.0f;
                        if (r > 7.0f) r = 7.0f;
                        q[u] = (int)r;
                    }
                }
                int64_t k = j * block + t;
                Q[m * ldq_bytes + k / 2] =
                    (uint8_t)(((unsigned)q[0] & 0xFu) | (((unsigned)q[1] & 0xFu) << 4));
            }
        }
    return 0;
}

/* ---- [W4A4] low-rank down-projection: XU = X . U in double ----
 * X: M x K binary32, U: K x R fp16 (row-major, ldu >= R), XU: M x R double. */
int orc_lowrank_xu(int64_t M, int64_t K, int64_t R, const float *X, int64_t ldx,
                   const uint16_t *U, int64_t ldu, double *XU, int64_t ldxu)
{
    if (M < 0 || K < 0 || R < 0 || ldx < K || ldu < R || ldxu < R)
        return 1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t r = 0; r < R; ++r) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)X[m * ldx + k] * orc_half_to_double(U[k * ldu + r]);
            XU[m * ldxu + r] = acc;
        }
    return 0;
}

/* ---- [W4A4] the GEMM: Y = (Q(X) . Q(W)^T) (.) scale + L(X) + b ----
 * "(.) scale" is read as the block-wise scales applied per K-block inside the
 * sum: for block j,  sX[m][j] * sW[n][j] * sum_{k in block j} qX[m][k]*qW[n][k].
 * L(X)[m][n] = sum_r XU[m][r] * V[r][n]  (XU = X.U, given here in double).
 * b is added per output column.  XU/V (R = 0) and bias may be absent (NULL):
 * the term is then omitted.
 * The column-wise affine calibration ([W4A4] sections 1 and 5.2: the drain
 * warps apply the scaling factors and a column-wise affine correction before
 * writing) is read as the map t -> alpha[n] * t + b[n] on each output column,
 * t being the scaled product plus L(X).  alpha (fp16, N entries) may be NULL,
 * which means alpha = 1: the formula as printed. */
int orc_w4a4_gemm(int64_t M, int64_t N, int64_t K,
                  const uint8_t *QX, int64_t ldqx_bytes,
                  const uint16_t *SX, int64_t ldsx,
                  const uint8_t *QW, int64_t ldqw_bytes,
                  const uint16_t *SW, int64_t ldsw, int64_t block,
                  const double *XU, int64_t ldxu,
                  const uint16_t *V, int64_t ldv, int64_t R,
                  const uint16_t *alpha, const uint16_t *bias, double *Y, int64_t ldy)
{
    if (M < 0 || N < 0 || K < 0 || block <= 0 || (block & 1) || K % block ||
        ldqx_bytes < K / 2 || ldqw_bytes < K / 2 || ldsx < K / block ||
        ldsw < K / block || ldy < N || R < 0)
        return 1;
    if (R > 0 && (!XU || !V || ldxu < R || ldv < N))
        return 1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t j = 0; j < K / block; ++j) {
                int64_t dot = 0;
                for (int64_t k = j * block; k < (j + 1) * block; ++k) {
                    uint8_t bx = QX[m * ldqx_bytes + k / 2];
                    uint8_t bw = QW[n * ldqw_bytes + k / 2];
                    int qx = nibble_value((k % 2 == 0) ? bx : (unsigned)bx >> 4);
                    int qw = nibble_value((k % 2 == 0) ? bw : (unsigned)bw >> 4);
                    dot += (int64_t)qx * (int64_t)qw;
                }
                acc += orc_half_to_double(SX[m * ldsx + j]) *
                       orc_half_to_double(SW[n * ldsw + j]) * (double)dot;
            }
            for (int64_t r = 0; r < R; ++r)
                acc += XU[m * ldxu + r] * orc_half_to_double(V[r * ldv + n]);
            if (alpha)
                acc *= orc_half_to_double(alpha[n]);
            if (bias)
                acc += orc_half_to_double(bias[n]);
            Y[m * ldy + n] = acc;
        }
    return 0;
}
