/*
 * CPU oracle for the tiled fp16 GEMM with optional fused bias + GELU epilogue.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes (plain definition, no blocking, no fusion, no reordering):
 *
 *   S[i,j] = sum_{k=0}^{K-1} A[i,k] * B[k,j]            in fp64
 *   x      = S[i,j] + bias[j]      (bias treated as 0 when absent)
 *   y      = GELU(x) = 0.5 * x * (1 + erf(x / sqrt(2)))  if the GELU epilogue is on,
 *            else y = x
 *   C[i,j] = y rounded once, to nearest-even, to IEEE binary16
 *
 * Sources:
 *   - "TileLang: writing LLM GPU kernels by thinking in tiles" (dev.to),
 *     section 2 "The basic idea: a GPU should reuse data": C[i,j] = sum_k A[i,k]*B[k,j],
 *     with A M x K, B K x N, C M x N; the triple loop is the definition.
 *   - same page, section 3 "What TileLang code actually looks like": A is (M,K),
 *     B is (K,N), C is (M,N), all row-major, fp16 inputs and output, fp32
 *     accumulation on the GPU. The oracle accumulates in fp64, which is exact
 *     for every product of two binary16 numbers and much tighter than fp32.
 *   - "Designing high-performance GPU kernels with TileLang ..." (scrapefeed),
 *     section 3 "Epilogue Fusion and Memory Efficiency": the epilogue is
 *     GELU(MatMul + Bias), bias first, then the activation, applied to the
 *     unrounded product. The pages do not say which GELU; the exact erf form is
 *     the reading taken here. Bias has length N and is added to column j.
 *
 * Parity pins (checked by the CPU test suite against things other than this
 * file): exhaustive binary16 decode and targeted encode against numpy's
 * float16 conversion; identity, permutation and rank-1 closed forms; brute
 * force with exact rational arithmetic on tiny shapes; fp64 matrix product
 * from numpy on random shapes; GELU against textbook values of the normal CDF
 * and the odd-part identity GELU(x) - GELU(-x) = x.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- IEEE 754 binary16 <-> binary64, written from the format definition ---- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal (or zero): f * 2^-24 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even, in one step.
 * Overflow (|x| >= 65520, the midpoint between 65504 and 2^16) gives inf. */
uint16_t oracle_double_to_half(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    double a = fabs(x);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: quantum 2^-24; scaling by a power of two is exact */
        double q = nearbyint(ldexp(a, 24)); /* default mode: to nearest, ties even */
        return (uint16_t)(sign | (uint16_t)q);  /* q == 1024 encodes 2^-14 correctly */
    }
    int E;
    (void)frexp(a, &E);          /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1;               /* a in [2^e, 2^(e+1)), e in [-14, 15] */
    double q = nearbyint(ldexp(a, 10 - e)); /* significand in [1024, 2048] */
    if (q >= 2048.0) { q = 1024.0; e += 1; }
    if (e > 15) return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* GELU with the exact Gaussian CDF: x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)). */
double oracle_gelu(double x) {
    return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
}

static double epilogue(double s, const uint16_t* bias, int64_t j, int gelu) {
    double x = s + (bias ? oracle_half_to_double(bias[j]) : 0.0);
    return gelu ? oracle_gelu(x) : x;
}

static double* decode_table(void) {
    double* t = (double*)malloc(65536 * sizeof(double));
    if (!t) return NULL;
    for (int h = 0; h < 65536; ++h) t[h] = oracle_half_to_double((uint16_t)h);
    return t;
}

/*
 * Rows [row0, row0 + nrows) of C = epi(A @ B + bias).
 * A: M x K binary16 bits, row-major. B: K x N binary16 bits, row-major.
 * bias: N binary16 bits or NULL. gelu: 0 or 1.
 * C: nrows x N binary16 bits (row r of the output is row row0 + r of C), or NULL.
 * C64: nrows x N doubles holding the value before the final rounding, or NULL.
 * threads <= 0 uses the OpenMP default. Returns 0, or -1 on bad arguments /
 * out of memory.
 */
int oracle_gemm_rows(const uint16_t* A, const uint16_t* B, const uint16_t* bias,
                     uint16_t* C, double* C64, int64_t M, int64_t N, int64_t K,
                     int gelu, int64_t row0, int64_t nrows, int threads) {
    if (M < 0 || N < 0 || K < 0 || row0 < 0 || nrows < 0 || row0 + nrows > M) return -1;
    if (gelu != 0 && gelu != 1) return -1;
    if (nrows == 0 || N == 0) return 0;
    double* lut = decode_table();
    if (!lut) return -1;
    int failed = 0;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
#pragma omp parallel
    {
        double* acc = (double*)malloc((size_t)N * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!acc) continue;
            int64_t i = row0 + r;
            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
            /* i-k-j order: the k-th term A[i,k] * B[k,:] added to the row sum */
            for (int64_t k = 0; k < K; ++k) {
                double a = lut[A[i * K + k]];
                const uint16_t* brow = B + k * N;
                for (int64_t j = 0; j < N; ++j) acc[j] += a * lut[brow[j]];
            }
            for (int64_t j = 0; j < N; ++j) {
                double y = epilogue(acc[j], bias, j, gelu);
                if (C) C[r * N + j] = oracle_double_to_half(y);
                if (C64) C64[r * N + j] = y;
            }
        }
        free(acc);
    }
    free(lut);
    return failed ? -1 : 0;
}

/* The whole of C (M x N). Same conventions as oracle_gemm_rows. */
int oracle_gemm(const uint16_t* A, const uint16_t* B, const uint16_t* bias,
                uint16_t* C, double* C64, int64_t M, int64_t N, int64_t K,
                int gelu, int threads) {
    return oracle_gemm_rows(A, B, bias, C, C64, M, N, K, gelu, 0, M, threads);
}

/*
 * Individual elements C[rows[t], cols[t]] for t in [0, count): each one is the
 * same definition evaluated alone, so full-size problems can be checked at
 * sampled positions. out / out64 as in oracle_gemm_rows (either may be NULL).
 */
int oracle_gemm_sampled(const uint16_t* A, const uint16_t* B, const uint16_t* bias,
                        int64_t M, int64_t N, int64_t K, int gelu,
                        const int64_t* rows, const int64_t* cols, int64_t count,
                        uint16_t* out, double* out64, int threads) {
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    if (gelu != 0 && gelu != 1) return -1;
    for (int64_t t = 0; t < count; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < count; ++t) {
        int64_t i = rows[t], j = cols[t];
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += oracle_half_to_double(A[i * K + k]) * oracle_half_to_double(B[k * N + j]);
        double y = epilogue(s, bias, j, gelu);
        if (out) out[t] = oracle_double_to_half(y);
        if (out64) out64[t] = y;
    }
    return 0;
}

/* ---- weight-only 4-bit GEMM ----
 *
 * "TileLang: writing LLM GPU kernels by thinking in tiles", section 5
 * ("Quantized LLM inference"): weights are stored as 4-bit integers,
 * dequantized into a tile, and the tile is multiplied like an fp16 weight
 * matrix. The pages fix no format; the reading taken here:
 *   - Bq: N rows of K/2 bytes, one row per output column n (the weight of
 *     a linear layer, out x in); byte j of row n holds q[2j][n] in its low 4
 *     bits and q[2j+1][n] in its high 4 bits, each a two's-complement integer
 *     in [-8, 7];
 *   - scales: ceil(K/group) rows of N binary16 values; q[k][n] belongs to
 *     group k / group;
 *   - the dequantized weight is W[k][n] = q[k][n] * scale[k/group][n] rounded
 *     once to binary16 (the fp16 tile the conversion produces);
 *   - C = epi(A @ W + bias) exactly as oracle_gemm_rows.
 */

/* Two's-complement value of the 4-bit field at bit `shift` of `byte`. */
int oracle_int4_value(uint8_t byte, int shift) {
    int v = (byte >> shift) & 0xF;
    return v >= 8 ? v - 16 : v;
}

/*
 * FP4 weights. The same section names 4-bit floating point (FP4) beside INT4
 * as a weight format. Reading taken: FP4 is the E2M1 element of the OCP
 * microscaling formats, each 4-bit field being
 *   bit 3      sign s
 *   bits 2..1  exponent e, bias 1
 *   bit 0      mantissa m
 * with value (-1)^s * 2^(e-1) * (1 + m/2) for e > 0 and (-1)^s * m/2 for e = 0
 * (zero and the one subnormal, 0.5); there are no infinities or NaN. Storage,
 * scales and rounding are those of the INT4 format above: the dequantized
 * weight is W[k][n] = v * scale[k/group][n] rounded once to binary16.
 */
double oracle_e2m1_value(uint8_t byte, int shift) {
    const int v = (byte >> shift) & 0xF;
    const int s = (v >> 3) & 1, e = (v >> 1) & 3, m = v & 1;
    const double x = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -x : x;
}

/* Value of the 4-bit field at bit `shift` of `byte` in weight format `format`
 * (0: two's-complement INT4, 1: FP4 E2M1). */
static double field_value(uint8_t byte, int shift, int format) {
    return format == 1 ? oracle_e2m1_value(byte, shift) : (double)oracle_int4_value(byte, shift);
}

/* W (K x N binary16 bits) from the packed weights and scales. */
int oracle_dequant_w4f(const uint8_t* Bq, const uint16_t* scales, uint16_t* W, int64_t N, int64_t K, int64_t group,
                       int format) {
    if (N < 0 || K < 0 || group <= 0 || (K % 2) != 0 || format < 0 || format > 1) return -1;
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t* row = Bq + n * (K / 2);
        for (int64_t k = 0; k < K; ++k) {
            const uint16_t* srow = scales + (k / group) * N;
            const double q = field_value(row[k / 2], (k % 2) ? 4 : 0, format);
            W[k * N + n] = oracle_double_to_half(q * oracle_half_to_double(srow[n]));
        }
    }
    return 0;
}

int oracle_dequant_w4(const uint8_t* Bq, const uint16_t* scales, uint16_t* W, int64_t N, int64_t K, int64_t group) {
    return oracle_dequant_w4f(Bq, scales, W, N, K, group, 0);
}

/* Rows [row0, row0 + nrows) of C = epi(A @ W + bias), W from oracle_dequant_w4f. */
int oracle_gemm_w4f_rows(const uint16_t* A, const uint8_t* Bq, const uint16_t* scales, const uint16_t* bias,
                         uint16_t* C, double* C64, int64_t M, int64_t N, int64_t K, int64_t group, int format,
                         int gelu, int64_t row0, int64_t nrows, int threads) {
    if (N < 0 || K < 0 || (K % 2) != 0 || group <= 0) return -1;
    uint16_t* W = (uint16_t*)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(uint16_t));
    if (!W) return -1;
    int rc = oracle_dequant_w4f(Bq, scales, W, N, K, group, format);
    if (rc == 0) rc = oracle_gemm_rows(A, W, bias, C, C64, M, N, K, gelu, row0, nrows, threads);
    free(W);
    return rc;
}

int oracle_gemm_w4_rows(const uint16_t* A, const uint8_t* Bq, const uint16_t* scales, const uint16_t* bias,
                        uint16_t* C, double* C64, int64_t M, int64_t N, int64_t K, int64_t group, int gelu,
                        int64_t row0, int64_t nrows, int threads) {
    return oracle_gemm_w4f_rows(A, Bq, scales, bias, C, C64, M, N, K, group, 0, gelu, row0, nrows, threads);
}

/* ---- Attention forward ----
 *
 * "TileLang: writing LLM GPU kernels by thinking in tiles", section 5 ("Why
 * this matters specifically for LLMs", FlashAttention): S = Q K^T / sqrt(d),
 * P = softmax(S) along each row, O = P V. "Designing high-performance GPU
 * kernels with TileLang ..." (section 5, FlashAttention) adds the causal mask.
 * Readings taken here: tensors are (batch, sequence, head, dim) row-major, the
 * layout of the bshd example the pages walk through; with the causal mask,
 * query position i sees key positions 0..i; softmax over the visible keys.
 *
 * The definition, one query row at a time, in fp64: every visible score, the
 * row maximum subtracted before exp (softmax is unchanged by a shift of its
 * inputs; the shift only keeps exp finite), exp, their sum, the weighted sum of
 * V rows divided by that sum, rounded once to binary16. No tiling and no
 * online rescaling: those are the kernel's business.
 *
 * rows[t] is a flat query row index (b * S + s) * H + h; output row t of O
 * (nrows x D binary16, and O64 in fp64 if not NULL) is that query's result.
 */
int oracle_attention_rows(const uint16_t* Q, const uint16_t* K, const uint16_t* V, uint16_t* O, double* O64,
                          int64_t B, int64_t S, int64_t H, int64_t D, int causal, double scale,
                          const int64_t* rows, int64_t nrows, int threads) {
    if (B < 0 || S < 0 || H < 0 || D < 0 || nrows < 0) return -1;
    for (int64_t t = 0; t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= B * S * H) return -1;
    double* lut = decode_table();
    if (!lut) return -1;
    int rc = 0;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel
#endif
    {
        double* sc = (double*)malloc((size_t)(S > 0 ? S : 1) * sizeof(double));
        double* acc = (double*)malloc((size_t)(D > 0 ? D : 1) * sizeof(double));
        double* q = (double*)malloc((size_t)(D > 0 ? D : 1) * sizeof(double));
        const int have = sc && acc && q;
        if (!have) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            rc = -1;
        }
        /* every thread reaches the work-sharing loop; one without buffers skips its rows */
        {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (int64_t t = 0; t < nrows; ++t) {
                if (!have) continue;
                const int64_t r = rows[t];
                const int64_t h = r % H, bs = r / H, si = bs % S, b = bs / S;
                for (int64_t d = 0; d < D; ++d) q[d] = lut[Q[r * D + d]];
                const int64_t visible = causal ? si + 1 : S;
                double m = -INFINITY;
                for (int64_t j = 0; j < visible; ++j) {
                    const uint16_t* kr = K + ((b * S + j) * H + h) * D;
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d) dot += q[d] * lut[kr[d]];
                    sc[j] = dot * scale;
                    if (sc[j] > m) m = sc[j];
                }
                double l = 0.0;
                for (int64_t d = 0; d < D; ++d) acc[d] = 0.0;
                for (int64_t j = 0; j < visible; ++j) {
                    const double pj = exp(sc[j] - m);
                    l += pj;
                    const uint16_t* vr = V + ((b * S + j) * H + h) * D;
                    for (int64_t d = 0; d < D; ++d) acc[d] += pj * lut[vr[d]];
                }
                for (int64_t d = 0; d < D; ++d) {
                    const double y = acc[d] / l;
                    if (O64) O64[t * D + d] = y;
                    if (O) O[t * D + d] = oracle_double_to_half(y);
                }
            }
        }
        free(sc);
        free(acc);
        free(q);
    }
    free(lut);
    return rc;
}

/* ---- Row softmax ----
 *
 * "Designing high-performance GPU kernels with TileLang ..." (scrapefeed),
 * section 4 "Advanced Reductions and Softmax": row-wise softmax, a maximum
 * over the row for numerical stability, then the sum of exponentials.
 * Y[i,j] = exp(X[i,j] - max_j X[i,:]) / sum_j exp(X[i,j] - max_j X[i,:]) in
 * fp64, rounded once to binary16. X and Y are M x N binary16, row-major.
 * Rows [row0, row0 + nrows) are computed; Y holds those rows (Y64 in fp64 if
 * not NULL). A row whose maximum is -inf (every entry -inf) has no defined
 * softmax; the arithmetic gives NaN, which is what is stored.
 */
int oracle_softmax_rows(const uint16_t* X, uint16_t* Y, double* Y64, int64_t M, int64_t N, int64_t row0,
                        int64_t nrows, int threads) {
    if (M < 0 || N < 0 || row0 < 0 || nrows < 0 || row0 + nrows > M) return -1;
    double* lut = decode_table();
    if (!lut) return -1;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        const uint16_t* x = X + (row0 + r) * N;
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j)
            if (lut[x[j]] > m) m = lut[x[j]];
        double l = 0.0;
        for (int64_t j = 0; j < N; ++j) l += exp(lut[x[j]] - m);
        for (int64_t j = 0; j < N; ++j) {
            const double y = exp(lut[x[j]] - m) / l;
            if (Y64) Y64[r * N + j] = y;
            if (Y) Y[r * N + j] = oracle_double_to_half(y);
        }
    }
    free(lut);
    return 0;
}

/* Number of threads an OpenMP parallel region of this library uses. */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
