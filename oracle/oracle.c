/*
 * oracle.c -- plain, slow, obviously correct CPU reference for the decode-step
 * weight-streaming matrix-vector product y = W.x and its skinny-batched form
 * Y = X.W^T, in fp64.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg may load this library. It shares no code,
 * header, table or helper with the CUDA path (memory_bound_weight_gb300/csrc).
 *
 * What it computes, and where the pages define it:
 *   - y = W.x with W stored (rows, K) row-major: "W (d,n) @ x (n,) -> xout (d,)",
 *     one output per row, each row a dot product with x
 *     (yalm, "Fast LLM inference from scratch", sec. 2 CPU matmul and
 *     sec. 3.1 GPU matmul; llm-rs vs vLLM, sec. 2 "Decode with one request is
 *     a memory problem": every weight used for one multiply and one add).
 *   - INT4 group-64 weights: 4-bit codes plus one fp16 scale per 64 weights
 *     (tinyinfer, "How I Built an LLM Inference Engine From Scratch in CUDA",
 *     TL;DR). The pages give no dequant formula; this oracle takes the
 *     symmetric reading w = (q - 8) * s.
 *   - AWQ-style INT4 weights: 4-bit codes with an fp16 scale and a zero point
 *     per 128 weights (llm-rs vs vLLM, sec. 6, format table); w = (q - z) * s
 *     with z a 4-bit code. The same codes reordered once at load time (sec. 6
 *     and sec. 7: Marlin-style reordered weights) give the same product; the
 *     reorder is a fixed permutation of the 8 nibbles of each 4-byte word.
 *   - Batched decode: the same weights used for M activation rows
 *     (llm-rs vs vLLM, sec. 3 "Batching moves decode from memory toward math").
 *   - Fusions around a GEMV: RMSNorm of x folded into the projection
 *     (llm-rs vs vLLM, "Decode: from ~35% to ~70% of the ceiling": norms folded
 *     into the projections), the residual add and the gated SiLU product
 *     silu(W1.x) * (W3.x) fused into the matmul that produces them (yalm,
 *     sec. 3.3 "Fusion and a better matmul"; TileInfer: SwiGLU in the GEMV
 *     epilogue).
 *   - Symmetric INT8 weights with one Float32 scale per output channel
 *     (TileInfer, "Pushing further with cheating: INT8 quantization"): codes
 *     q in [-127, 127], w_ik = s_i * q_ik, and the load-time quantizer that
 *     makes them, s_i = max_k |w_ik| / 127 and q_ik = w_ik / s_i rounded to the
 *     nearest integer.
 *
 * Readings where the pages are silent (all recorded in the design notes):
 *   - nibble order: the low nibble of byte b holds code k = 2b (even k), the
 *     high nibble code k = 2b + 1;
 *   - a group is 64 (or 128) consecutive k within one row;
 *   - AWQ zero points are packed two per byte, low nibble = even group, with
 *     ceil(G/2) bytes per row (G = K/128 groups);
 *   - accumulation order: k = 0 .. K-1 sequentially in fp64 per output;
 *   - RMSNorm: xn_k = x_k * g_k / sqrt(mean_k(x_k^2) + eps), computed in fp64 and
 *     rounded to bf16 (round to nearest even), since the normalised vector is
 *     the bf16 activation the projection consumes;
 *   - SiLU(a) = a / (1 + exp(-a)); the fused output is silu(gate) * up, and the
 *     residual add is y + r, both on the fp64 GEMV results;
 *   - INT8 quantizer: the scale is computed in fp32 (the stored precision),
 *     the quotient w / s in fp32 (IEEE division), rounded to the nearest
 *     integer with ties to even; an all-zero row gets s = 0 and q = 0.
 *
 * Every product w*x is exact in fp64 (INT4: w has at most 15 significant
 * bits; INT8: s * q has at most 32; x at most 8), so the only rounding is in
 * the fp64 summation.
 *
 * Each GEMV also returns yabs[i] = sum_k |w_ik * x_k| in fp64, the quantity
 * the parity tolerance is stated against.
 *
 * Parallelism: OpenMP over output rows (the row-parallel shape of yalm's
 * OpenMP CPU matmul). Each output is summed by one thread in k order, so the
 * result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Number formats, written from their definitions.                           */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0 -> subnormal 0.f * 2^-14; exponent 31 -> inf / NaN. */
double oracle_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* f/1024 * 2^-14 */
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp(1024.0 + (double)f, e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE 754 binary32. 1 sign bit, 8 exponent
 * bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* f/128 * 2^-126 */
    else if (e == 255)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp(128.0 + (double)f, e - 134);     /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

/* Round a double to the nearest bfloat16, ties to even (finite inputs).
 * Written on the value, not on bit patterns: find the bf16 spacing at |v|,
 * round |v| / spacing to the nearest integer with ties to even. */
uint16_t oracle_double_to_bf16_rne(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex);                                  /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 1;                                 /* a in [2^e, 2^(e+1)) */
    if (e < -126)
        e = -126;                                   /* subnormal range: fixed spacing */
    double ulp = ldexp(1.0, e - 7);
    double n = a / ulp;                             /* exact: power-of-two division */
    double fl = floor(n);
    double rem = n - fl;
    double r = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0))
        r = fl + 1.0;
    double q = r * ulp;                             /* exact */
    if (q >= ldexp(1.0, 128))                       /* rounded past the bf16 maximum */
        return sign | 0x7F80;
    /* encode q (a bf16 value) */
    if (q < ldexp(1.0, -126))
        return sign | (uint16_t)(q / ldexp(1.0, -133));
    frexp(q, &ex);
    int be = ex - 1 + 127;
    int frac = (int)(q / ldexp(1.0, ex - 1 - 7)) - 128;
    return sign | (uint16_t)(be << 7) | (uint16_t)frac;
}

/* ------------------------------------------------------------------------ */
/* INT4 unpack and dequant, one weight at a time.                            */
/* ------------------------------------------------------------------------ */

/* 4-bit code of weight (i, k): byte i*K/2 + k/2, low nibble if k is even. */
static int code_at(const uint8_t *codes, int64_t K, int64_t i, int64_t k)
{
    uint8_t b = codes[i * (K / 2) + k / 2];
    return (k % 2 == 0) ? (b & 0x0F) : (b >> 4);
}

/* Group-64 symmetric: w = (q - 8) * s, s = fp16 scale of group k/64 of row i. */
static double dequant_g64(const uint8_t *codes, const uint16_t *scales,
                          int64_t K, int64_t i, int64_t k)
{
    int q = code_at(codes, K, i, k);
    double s = oracle_f16_to_double(scales[i * (K / 64) + k / 64]);
    return (double)(q - 8) * s;
}

/* Load-time repacked layout of the same codes (llm-rs vs vLLM, sec. 6
 * "Quantization helps memory-bound work, and can hurt compute-bound work" and
 * sec. 7 "Reading the scoreboard": 4-bit weights reordered once at load time,
 * so that the kernel's unpack hands the multiply its operands in order). A
 * row keeps its K/2 bytes; within each 4-byte word (weights k = 8w .. 8w+7,
 * nibble slot t = bits 4t .. 4t+3 of the little-endian word) weight 8w + j
 * sits in slot j/2 + 4*(j%2): the even k in slots 0-3, the odd k in 4-7. */
static int repacked_slot(int j) { return j / 2 + 4 * (j % 2); }

/* 4-bit code of weight (i, k) in the repacked layout. */
static int repacked_code_at(const uint8_t *codes, int64_t K, int64_t i, int64_t k)
{
    int t = repacked_slot((int)(k % 8));
    uint8_t b = codes[i * (K / 2) + (k / 8) * 4 + t / 2];
    return (t % 2 == 0) ? (b & 0x0F) : (b >> 4);
}

/* out = the repacked layout of canonical codes [N][K/2] (K a multiple of 8). */
void oracle_repack_int4(const uint8_t *codes, int64_t N, int64_t K, uint8_t *out)
{
    for (int64_t i = 0; i < N; i++) {
        for (int64_t b = 0; b < K / 2; b++) out[i * (K / 2) + b] = 0;
        for (int64_t k = 0; k < K; ++k) {
            int q = code_at(codes, K, i, k);
            int t = repacked_slot((int)(k % 8));
            int64_t at = i * (K / 2) + (k / 8) * 4 + t / 2;
            out[at] = (uint8_t)(out[at] | (t % 2 == 0 ? q : q << 4));
        }
    }
}

/* AWQ-style group-128: w = (q - z) * s with scale and zero point of group
 * g = k/128 of row i; zero points packed two per byte, low nibble = even g.
 * `repacked`: the codes are in the repacked layout above. */
static double dequant_awq_any(const uint8_t *codes, const uint16_t *scales,
                              const uint8_t *zeros, int64_t K, int64_t i, int64_t k,
                              int repacked)
{
    int64_t G = K / 128;
    int64_t zstride = (G + 1) / 2;
    int64_t g = k / 128;
    int q = repacked ? repacked_code_at(codes, K, i, k) : code_at(codes, K, i, k);
    uint8_t zb = zeros[i * zstride + g / 2];
    int z = (g % 2 == 0) ? (zb & 0x0F) : (zb >> 4);
    double s = oracle_f16_to_double(scales[i * G + g]);
    return (double)(q - z) * s;
}

static double dequant_awq(const uint8_t *codes, const uint16_t *scales,
                          const uint8_t *zeros, int64_t K, int64_t i, int64_t k)
{
    return dequant_awq_any(codes, scales, zeros, K, i, k, 0);
}

void oracle_dequant_int4_g64(const uint8_t *codes, const uint16_t *scales,
                             int64_t N, int64_t K, double *out)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < N; i++)
        for (int64_t k = 0; k < K; k++)
            out[i * K + k] = dequant_g64(codes, scales, K, i, k);
}

void oracle_dequant_int4_awq_g128(const uint8_t *codes, const uint16_t *scales,
                                  const uint8_t *zeros, int64_t N, int64_t K,
                                  double *out)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < N; i++)
        for (int64_t k = 0; k < K; k++)
            out[i * K + k] = dequant_awq(codes, scales, zeros, K, i, k);
}

/* ------------------------------------------------------------------------ */
/* Matrix-vector and skinny matrix products.                                 */
/* Y[m][i] = sum_k X[m][k] * w(i, k); yabs[m][i] = sum_k |X[m][k] * w(i, k)|. */
/* Output layout: Y is (M, N) row-major. M = 1 is the plain GEMV.            */
/* ------------------------------------------------------------------------ */

void oracle_gemm_bf16(const uint16_t *W, const uint16_t *X, int64_t M,
                      int64_t N, int64_t K, double *Y, double *Yabs)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < N; i++) {
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, aabs = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double w = oracle_bf16_to_double(W[i * K + k]);
                double x = oracle_bf16_to_double(X[m * K + k]);
                acc += w * x;
                aabs += fabs(w * x);
            }
            Y[m * N + i] = acc;
            Yabs[m * N + i] = aabs;
        }
    }
}

void oracle_gemm_int4_g64(const uint8_t *codes, const uint16_t *scales,
                          const uint16_t *X, int64_t M, int64_t N, int64_t K,
                          double *Y, double *Yabs)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < N; i++) {
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, aabs = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double w = dequant_g64(codes, scales, K, i, k);
                double x = oracle_bf16_to_double(X[m * K + k]);
                acc += w * x;
                aabs += fabs(w * x);
            }
            Y[m * N + i] = acc;
            Yabs[m * N + i] = aabs;
        }
    }
}

static void gemm_awq_any(const uint8_t *codes, const uint16_t *scales,
                         const uint8_t *zeros, const uint16_t *X, int64_t M,
                         int64_t N, int64_t K, double *Y, double *Yabs,
                         int repacked)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < N; i++) {
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, aabs = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double w = dequant_awq_any(codes, scales, zeros, K, i, k, repacked);
                double x = oracle_bf16_to_double(X[m * K + k]);
                acc += w * x;
                aabs += fabs(w * x);
            }
            Y[m * N + i] = acc;
            Yabs[m * N + i] = aabs;
        }
    }
}

void oracle_gemm_int4_awq_g128(const uint8_t *codes, const uint16_t *scales,
                               const uint8_t *zeros, const uint16_t *X,
                               int64_t M, int64_t N, int64_t K, double *Y,
                               double *Yabs)
{
    gemm_awq_any(codes, scales, zeros, X, M, N, K, Y, Yabs, 0);
}

/* The same product with the codes in the repacked layout. */
void oracle_gemm_int4_awq_g128_repacked(const uint8_t *codes, const uint16_t *scales,
                                        const uint8_t *zeros, const uint16_t *X,
                                        int64_t M, int64_t N, int64_t K, double *Y,
                                        double *Yabs)
{
    gemm_awq_any(codes, scales, zeros, X, M, N, K, Y, Yabs, 1);
}

/* ------------------------------------------------------------------------ */
/* Symmetric INT8, one fp32 scale per output channel.                        */
/* ------------------------------------------------------------------------ */

/* Y[m][i] = sum_k w_ik * X[m][k] with w_ik = S[i] * Q[i][k] (TileInfer,
 * "Pushing further with cheating: INT8 quantization": one scale per output
 * channel). The plain definition: dequantize each weight, multiply, add. The
 * pages' kernel sums q * x and applies S[i] once at the end, which is the same
 * value up to rounding order. Q int8 [N][K], S fp32 [N], X bf16 [M][K]. */
void oracle_gemm_int8_pc(const int8_t *Q, const float *S, const uint16_t *X,
                         int64_t M, int64_t N, int64_t K, double *Y,
                         double *Yabs)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < N; i++) {
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, aabs = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double w = (double)S[i] * (double)Q[i * K + k];
                double x = oracle_bf16_to_double(X[m * K + k]);
                acc += w * x;
                aabs += fabs(w * x);
            }
            Y[m * N + i] = acc;
            Yabs[m * N + i] = aabs;
        }
    }
}

/* Load-time quantizer of one weight matrix (same section): for each row i,
 * s_i = max_k |w_ik| / 127 in fp32, and q_ik = w_ik / s_i rounded to the
 * nearest integer (fp32 quotient, ties to even), so the largest entry lands
 * on +-127 and every entry is off by at most s_i / 2. W bf16 [N][K]. */
void oracle_quantize_int8_pc(const uint16_t *W, int64_t N, int64_t K,
                             int8_t *Q, float *S)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < N; i++) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; k++) {
            float a = (float)fabs(oracle_bf16_to_double(W[i * K + k]));
            if (a > amax)
                amax = a;
        }
        float s = amax / 127.0f;                    /* fp32 division */
        S[i] = s;
        for (int64_t k = 0; k < K; k++) {
            if (s == 0.0f) {
                Q[i * K + k] = 0;
                continue;
            }
            float w = (float)oracle_bf16_to_double(W[i * K + k]);
            float t = w / s;                          /* fp32 division */
            float r = rintf(t);                       /* nearest, ties to even */
            if (r > 127.0f)
                r = 127.0f;
            if (r < -127.0f)
                r = -127.0f;
            Q[i * K + k] = (int8_t)r;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Fusions around the GEMV.                                                  */
/* ------------------------------------------------------------------------ */

/* RMSNorm of each row of X with weight G (the prologue folded into a
 * projection), before the activation is rounded to bf16:
 * V[m][k] = X[m][k] * G[k] / sqrt(mean_k X[m][k]^2 + eps), in fp64.
 * X bf16 [M][K], G bf16 [K], V double [M][K]. */
void oracle_rmsnorm_f64(const uint16_t *X, const uint16_t *G, int64_t M,
                        int64_t K, double eps, double *V)
{
    for (int64_t m = 0; m < M; m++) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double x = oracle_bf16_to_double(X[m * K + k]);
            ss += x * x;
        }
        double inv = 1.0 / sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; k++) {
            double x = oracle_bf16_to_double(X[m * K + k]);
            double g = oracle_bf16_to_double(G[k]);
            V[m * K + k] = x * inv * g;
        }
    }
}

/* The normalised activation the projection consumes:
 * Xn[m][k] = bf16(V[m][k]) (round to nearest even) with V as above.
 * Xn bf16 [M][K]. */
void oracle_rmsnorm_bf16(const uint16_t *X, const uint16_t *G, int64_t M,
                         int64_t K, double eps, uint16_t *Xn)
{
    double *row = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
    for (int64_t m = 0; m < M; m++) {
        oracle_rmsnorm_f64(X + m * K, G, 1, K, eps, row);
        for (int64_t k = 0; k < K; k++)
            Xn[m * K + k] = oracle_double_to_bf16_rne(row[k]);
    }
    free(row);
}

/* Gated SiLU of two GEMV results of the same shape: out = silu(A) * B with
 * silu(a) = a / (1 + exp(-a)) (yalm: F.silu(w1(x)) * w3(x)). */
void oracle_swiglu(const double *A, const double *B, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = A[i] / (1.0 + exp(-A[i])) * B[i];
}

/* Residual add: out = Y + R (R bf16), the result written back into the
 * residual stream (yalm: fused matmul + add_residuals). */
void oracle_add_residual(const double *Y, const uint16_t *R, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = Y[i] + oracle_bf16_to_double(R[i]);
}

/* Threads the OpenMP loops above will use (for reporting the CPU baseline). */
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
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
