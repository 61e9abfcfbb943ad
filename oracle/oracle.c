/*
 * oracle.c -- plain, slow fp64 CPU reference for the GEMM computation fixed by
 * the TVM TIRX tile-op pages.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the bench's CPU-baseline leg call it; the product path never does,
 * and nothing here is shared with the CUDA code.
 *
 * What it computes, for every output element (i, j):
 *
 *     ref[i][j] = alpha * sum_k A[i][k] * B[j][k]  +  beta * C[i][j]
 *     abs[i][j] =         sum_k |A[i][k]| * |B[j][k]|
 *
 *  - A is row-major M x K and B is stored N x K, so the product is A times B
 *    transposed ("mma.sync" page, section "Operand coordinates and
 *    ownership": the B atom axes are (N, K/2) although the product uses B
 *    transposed; its worked example checks against a @ b.T).
 *  - A and B hold f16 or bf16 values; C and the result are float32 on the
 *    GPU (same section, operand table).  Here every value is widened exactly
 *    to double and the k sum runs sequentially in double.
 *  - alpha and beta are applied at the call site, after the product
 *    ("mma.sync" page, section "Accumulation, transpose and alpha/beta").
 *    C == NULL or beta == 0 means the C term is absent and C is not read.
 *  - Row-gathered form: row i of A is row idx[i] of a table with table_rows
 *    rows ("cp.async.bulk.tensor" page, section "Gather4 and scatter4": the
 *    row coordinates are runtime operands chosen by the caller).  An index
 *    outside [0, table_rows) makes that A row zero and the call returns 1.
 *
 * The result is left in double: the tests round it to float32 (and then to
 * bf16/f16) themselves, which for exactly representable results is the
 * single rounding that one fma.rn.f32 performs ("fma" page, section
 * "Operand specification").
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16_bits(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* zero or subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25); /* (1024 + f) * 2^(e - 15 - 10) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static double decode_bf16_bits(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);             /* zero or subnormal: f * 2^(1-127-7) */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x80), e - 134); /* (128 + f) * 2^(e - 127 - 7) */
    return sign ? -v : v;
}

/* Decoded value of every 16-bit pattern, filled once by oracle_init(). */
static double g_value[2][65536];
static int g_ready = 0;

void oracle_init(void)
{
    if (g_ready)
        return;
    for (uint32_t bits = 0; bits < 65536u; ++bits) {
        g_value[ORACLE_F16][bits] = decode_f16_bits((uint16_t)bits);
        g_value[ORACLE_BF16][bits] = decode_bf16_bits((uint16_t)bits);
    }
    g_ready = 1;
}

double oracle_decode(int dtype, uint16_t bits)
{
    return dtype == ORACLE_BF16 ? decode_bf16_bits(bits) : decode_f16_bits(bits);
}

/* Row i of the logical A operand, or NULL when the gathered index is invalid. */
static const uint16_t *a_row(int64_t i, const uint16_t *A, int64_t lda,
                             const int32_t *idx, int64_t table_rows)
{
    if (!idx)
        return A + i * lda;
    int64_t r = idx[i];
    if (r < 0 || r >= table_rows)
        return NULL;
    return A + r * lda;
}

/* One output element.  Returns 1 when A's row came from an invalid index. */
static int one_entry(int64_t i, int64_t j, int64_t K, int dtype,
                     const uint16_t *A, int64_t lda, const int32_t *idx,
                     int64_t table_rows, const uint16_t *B, int64_t ldb,
                     const float *C, int64_t ldc, double alpha, double beta,
                     double *ref, double *abs_out)
{
    const double *val = g_value[dtype == ORACLE_BF16 ? ORACLE_BF16 : ORACLE_F16];
    const uint16_t *arow = a_row(i, A, lda, idx, table_rows);
    const uint16_t *brow = B + j * ldb;
    double sum = 0.0, sum_abs = 0.0;
    if (arow) {
        for (int64_t k = 0; k < K; ++k) {
            double a = val[arow[k]];
            double b = val[brow[k]];
            sum += a * b;
            sum_abs += fabs(a) * fabs(b);
        }
    }
    double r = alpha * sum;
    if (C && beta != 0.0)
        r += beta * (double)C[i * ldc + j];
    *ref = r;
    if (abs_out)
        *abs_out = sum_abs;
    return arow ? 0 : 1;
}

/*
 * Rows [i0, i1) of the full result, all N columns.  ref and abs_out (may be
 * NULL) are indexed [(i - i0) * ldr + j].  Returns 1 if any gathered index in
 * the range was invalid, 0 otherwise.
 */
int oracle_gemm_rows(int64_t i0, int64_t i1, int64_t N, int64_t K, int dtype,
                     const uint16_t *A, int64_t lda, const int32_t *idx,
                     int64_t table_rows, const uint16_t *B, int64_t ldb,
                     const float *C, int64_t ldc, double alpha, double beta,
                     double *ref, double *abs_out, int64_t ldr)
{
    int bad = 0;
    oracle_init();
    for (int64_t i = i0; i < i1; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            int64_t o = (i - i0) * ldr + j;
            bad |= one_entry(i, j, K, dtype, A, lda, idx, table_rows, B, ldb, C,
                             ldc, alpha, beta, &ref[o], abs_out ? &abs_out[o] : NULL);
        }
    }
    return bad;
}

/* Selected entries (ii[e], jj[e]) for e in [0, n). */
int oracle_gemm_entries(int64_t n, const int64_t *ii, const int64_t *jj,
                        int64_t K, int dtype, const uint16_t *A, int64_t lda,
                        const int32_t *idx, int64_t table_rows,
                        const uint16_t *B, int64_t ldb, const float *C,
                        int64_t ldc, double alpha, double beta, double *ref,
                        double *abs_out)
{
    int bad = 0;
    oracle_init();
    for (int64_t e = 0; e < n; ++e)
        bad |= one_entry(ii[e], jj[e], K, dtype, A, lda, idx, table_rows, B, ldb,
                         C, ldc, alpha, beta, &ref[e], abs_out ? &abs_out[e] : NULL);
    return bad;
}

/*
 * Row-scattered form ("cp.async.bulk.tensor" page, section "Gather4 and
 * scatter4": scatter4 is the store-side dual of gather4 and writes four
 * caller-chosen rows of the destination).  Row i of the product A * B^T goes
 * to row d = idx[i] of D, and the C term comes from that same destination
 * row, so C and D are indexed alike as in every other form:
 *
 *     D[d][j] = alpha * sum_k A[i][k] * B[j][k]  +  beta * C[d][j],  d = idx[i]
 *
 * For i in [i0, i1) this fills row (i - i0) of ref / abs_out (ldr apart) with
 * the values that row i sends; where they land is the caller's business.  An
 * index outside [0, d_rows) sends nothing: its row is set to NaN and the call
 * returns 1.
 */
int oracle_scatter_rows(int64_t i0, int64_t i1, int64_t N, int64_t K, int dtype,
                        const uint16_t *A, int64_t lda, const int32_t *idx,
                        int64_t d_rows, const uint16_t *B, int64_t ldb,
                        const float *C, int64_t ldc, double alpha, double beta,
                        double *ref, double *abs_out, int64_t ldr)
{
    const double *val;
    int bad = 0;
    oracle_init();
    val = g_value[dtype == ORACLE_BF16 ? ORACLE_BF16 : ORACLE_F16];
    for (int64_t i = i0; i < i1; ++i) {
        const int64_t d = idx[i];
        const uint16_t *arow = A + i * lda;
        double *out = ref + (i - i0) * ldr;
        double *out_abs = abs_out ? abs_out + (i - i0) * ldr : NULL;
        if (d < 0 || d >= d_rows) {
            for (int64_t j = 0; j < N; ++j) {
                out[j] = NAN;
                if (out_abs)
                    out_abs[j] = NAN;
            }
            bad = 1;
            continue;
        }
        for (int64_t j = 0; j < N; ++j) {
            const uint16_t *brow = B + j * ldb;
            double sum = 0.0, sum_abs = 0.0;
            for (int64_t kk = 0; kk < K; ++kk) {
                double a = val[arow[kk]];
                double b = val[brow[kk]];
                sum += a * b;
                sum_abs += fabs(a) * fabs(b);
            }
            double r = alpha * sum;
            if (C && beta != 0.0)
                r += beta * (double)C[d * ldc + j];
            out[j] = r;
            if (out_abs)
                out_abs[j] = sum_abs;
        }
    }
    return bad;
}

/*
 * FP4 weights with block scales.  The "cp.async.bulk.tensor" page (section
 * "Interleave and packed FP4") gives the float4_e2m1fn operand format; it does
 * not give the numbers the codes stand for or how blocks are scaled.  Those
 * come from the OCP Microscaling (MX) formats definition that the e2m1 name
 * refers to: an E2M1 element has 1 sign bit, 2 exponent bits with bias 1 and
 * 1 mantissa bit, exponent 0 being subnormal (mantissa * 0.5), no infinity or
 * NaN; a UE8M0 block scale s stands for 2^(s - 127), s = 255 being NaN; one
 * scale covers 32 consecutive elements along K.
 */
double oracle_decode_e2m1(int code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

double oracle_decode_ue8m0(int s)
{
    return s == 255 ? NAN : ldexp(1.0, s - 127);
}

/*
 * Rows [i0, i1) of D = alpha * A * W^T + beta * C with
 *   W[j][k] = e2m1(code of element k in row j of Wq) * ue8m0(Ws[k / 32][j]).
 * Row j of Wq holds K / 2 bytes; element k is the low nibble of byte k / 2 when
 * k is even and the high nibble when k is odd.  Ws holds K / 32 rows of N
 * scale bytes, lds bytes apart.  A is f16 or bf16 (dtype), as in
 * oracle_gemm_rows; ref and abs_out likewise.
 */
void oracle_w4_rows(int64_t i0, int64_t i1, int64_t N, int64_t K, int dtype,
                    const uint16_t *A, int64_t lda, const uint8_t *Wq, int64_t ldq,
                    const uint8_t *Ws, int64_t lds, const float *C, int64_t ldc,
                    double alpha, double beta, double *ref, double *abs_out, int64_t ldr)
{
    const double *val;
    oracle_init();
    val = g_value[dtype == ORACLE_BF16 ? ORACLE_BF16 : ORACLE_F16];
    for (int64_t i = i0; i < i1; ++i) {
        const uint16_t *arow = A + i * lda;
        for (int64_t j = 0; j < N; ++j) {
            const uint8_t *wrow = Wq + j * ldq;
            double sum = 0.0, sum_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int byte = wrow[k / 2];
                int code = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
                double w = oracle_decode_e2m1(code) * oracle_decode_ue8m0(Ws[(k / 32) * lds + j]);
                double a = val[arow[k]];
                sum += a * w;
                sum_abs += fabs(a) * fabs(w);
            }
            double r = alpha * sum;
            if (C && beta != 0.0)
                r += beta * (double)C[i * ldc + j];
            ref[(i - i0) * ldr + j] = r;
            if (abs_out)
                abs_out[(i - i0) * ldr + j] = sum_abs;
        }
    }
}

/*
 * Both operands FP4 with block scales (the block-scaled tensor-core product):
 * rows [i0, i1) of D = alpha * A * B^T + beta * C with
 *   A[i][k] = e2m1(code of element k in row i of Aq) * ue8m0(As[k / 32][i]),
 *   B[j][k] = e2m1(code of element k in row j of Bq) * ue8m0(Bs[k / 32][j]).
 * Rows of Aq and Bq hold K / 2 bytes, element k in the low nibble of byte
 * k / 2 when k is even and in the high nibble when k is odd (ldaq, ldbq bytes
 * apart); As holds K / 32 rows of M scale bytes (ldas apart) and Bs K / 32 rows
 * of N (ldbs apart), one scale per 32 consecutive elements along K, as the OCP
 * Microscaling definition the float4_e2m1fn name refers to groups them ("cp.async.bulk.tensor"
 * page, section "Interleave and packed FP4", gives the operand format).
 * ref and abs_out as in oracle_gemm_rows.
 */
static double fp4_element(const uint8_t *codes, const uint8_t *scales, int64_t lds,
                          int64_t row, int64_t k)
{
    int byte = codes[k / 2];
    int code = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
    return oracle_decode_e2m1(code) * oracle_decode_ue8m0(scales[(k / 32) * lds + row]);
}

void oracle_e2m1_rows(int64_t i0, int64_t i1, int64_t N, int64_t K,
                      const uint8_t *Aq, int64_t ldaq, const uint8_t *As, int64_t ldas,
                      const uint8_t *Bq, int64_t ldbq, const uint8_t *Bs, int64_t ldbs,
                      const float *C, int64_t ldc, double alpha, double beta,
                      double *ref, double *abs_out, int64_t ldr)
{
    for (int64_t i = i0; i < i1; ++i) {
        const uint8_t *arow = Aq + i * ldaq;
        for (int64_t j = 0; j < N; ++j) {
            const uint8_t *brow = Bq + j * ldbq;
            double dot = 0.0, dot_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = fp4_element(arow, As, ldas, i, k);
                double b = fp4_element(brow, Bs, ldbs, j, k);
                dot += a * b;
                dot_abs += fabs(a) * fabs(b);
            }
            double d = alpha * dot;
            if (C && beta != 0.0)
                d += beta * (double)C[i * ldc + j];
            ref[(i - i0) * ldr + j] = d;
            if (abs_out)
                abs_out[(i - i0) * ldr + j] = dot_abs;
        }
    }
}
