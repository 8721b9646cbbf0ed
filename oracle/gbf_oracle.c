/*
 * gbf_oracle.c -- plain, slow fp64 CPU oracle for the fused
 * GEMM + epilogue path.  TEST INFRASTRUCTURE ONLY: it is used by tests/,
 * by the smoke check and by the CPU-baseline leg of the benchmark.  No
 * product code path links or calls it, and it shares no code, header or
 * constant with the CUDA library.
 *
 * What it computes (each function cites the passage it follows):
 *
 *   gemm_epilogue   out = bf16( act(alpha*A*B + beta*C + bias) + residual )
 *       "Fusion and Epilogues" (metalworking.vercel.app), bullet
 *       "Epilogue fusion, the mechanical form": the GEMM ending alpha*AB +
 *       beta*C, bias, activation, applied on the way to the one write.
 *       "Kernel fusion" (guide.dupenodi.dev), section "Concept": bias,
 *       activation, scaling, residual add.  Order: bias inside the
 *       activation, residual outside it.
 *   swiglu          h = bf16( act(alpha*g) * (alpha*u) + beta*C ),
 *                   g = x*W_gate^T, u = x*W_up^T
 *       "Fusion Thinking", Pattern 2 (Fused SwiGLU): gate and up products of
 *       the same x, silu(gate)*up, level 2 = both products in one GEMM with
 *       SwiGLU in its epilogue.
 *   w4a16           w[k][n] = bf16((q[k][n] - 8) * s[k/G][n]), then the
 *                   gemm_epilogue formula with B = w.
 *       "Fusion Thinking", Pattern 3 (Dequant + GEMM): packed 2 x int4 per
 *       byte along N, high nibble first (interleave(w_hi, w_lo)), zero point
 *       8, per-group bf16 scales, result fed to the matrix product.
 *   wq_gemm         the gemm_epilogue formula with B = a dequantised
 *                   weight of one of three weight-only formats:
 *                   int4:  bf16((q - 8) * s[k/G][n])       (as w4a16)
 *                   fp8:   bf16(e4m3(q[k][n]) * s[k/G][n]) (bf16 group scales)
 *                   nvfp4: bf16(e2m1(q[k][n]) * e4m3(S[k/16][n]))
 *       "Fusion Thinking", Pattern 3 names INT4 / INT8 / NVFP4 weights with
 *       BF16 activations; "Fusion and Epilogues" lists INT4 / FP8 / FP4
 *       paths.  The element formats are the public OCP 8-bit (E4M3: bias 7,
 *       subnormals, no infinity, S.1111.111 = NaN) and 4-bit (E2M1: bias 1,
 *       values 0, 0.5, 1, 1.5, 2, 3, 4, 6) floating-point encodings; NVFP4
 *       scales each run of 16 elements along K by an E4M3 factor, and its
 *       per-tensor factor is the product's alpha.
 *   add_rmsnorm     r = a + x;  resid = bf16(r);
 *                   n = bf16( r / sqrt(mean_j(r_j^2) + eps) * w )   (per row)
 *       "Fusion Thinking", Pattern 1 (Fused RMSNorm + residual): one pass
 *       computes the residual sum, writes it for the next residual add, and
 *       normalises the (unrounded) sum with the row's root mean square.
 *   unfused modes   the same results with the intermediate written as bf16
 *       between the product and the pointwise pass ("kernel fusion",
 *       infraphysics.net: "the activation-after-matmul case"; "Fusion
 *       Thinking", Pattern 2 un-fused and Pattern 3 un-fused).
 *
 * Arithmetic: every product and sum in fp64 (double), rounded once to bf16
 * at the end with round-to-nearest-even; in the unfused modes the bf16
 * intermediates are rounded the same way.  Activations use the host libm:
 *   relu(v)      = max(v, 0)
 *   silu(v)      = v * sigmoid(v) = v / (1 + exp(-v))
 *   gelu_tanh(v) = 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))
 * (the tanh form of GELU; the pages name SiLU but define no GELU).
 *
 * Threads: the same file is also built with OpenMP (a second library, for
 * the all-cores timing and for the full-output checks of the large
 * workloads).  Then the loop over output elements (or rows) is shared out
 * among threads; each element is still computed by one thread with the same
 * sequential fp64 sum in the same order, so both builds give identical bits.
 *
 * Parity pins live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

/* Independent iterations of an output loop (ignored without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
#define ORACLE_PARALLEL_FOR _Pragma("omp parallel for schedule(dynamic, 16)")
#else
#define ORACLE_PARALLEL_FOR
#endif

/* Threads of the OpenMP build (1 without OpenMP). */
int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

enum { ACT_IDENTITY = 0, ACT_RELU = 1, ACT_SILU = 2, ACT_GELU_TANH = 3 };
enum { LAYOUT_KN = 0, LAYOUT_NK = 1 };

/* ---- bf16 <-> double ---------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16, ties to even, in one step (no detour
 * through binary32, which would round twice).  bf16 keeps 8 significant bits
 * for normal numbers (exponent >= -126); below that the spacing is fixed at
 * 2^-133.  Values at or beyond 2^128 after rounding become infinity. */
uint16_t oracle_bf16_from_f64(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);           /* a in [2^(e-1), 2^e) */
    int top = e - 1;
    int ulp_exp = (top < -126 ? -126 : top) - 7;
    double q = ldexp(a, -ulp_exp); /* exact power-of-two scaling */
    double r = nearbyint(q);       /* default rounding mode: ties to even */
    double rounded = ldexp(r, ulp_exp);
    if (rounded >= 0x1p128)
        return sign | 0x7F80;
    float f = (float)rounded;      /* exact: at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* ---- activations -------------------------------------------------------- */

double oracle_act(int act, double v)
{
    switch (act) {
    case ACT_IDENTITY:
        return v;
    case ACT_RELU:
        return v > 0.0 ? v : 0.0;
    case ACT_SILU:
        return v / (1.0 + exp(-v));
    case ACT_GELU_TANH: {
        const double c = sqrt(2.0 / M_PI);
        return 0.5 * v * (1.0 + tanh(c * (v + 0.044715 * v * v * v)));
    }
    default:
        return NAN;
    }
}

/* ---- element kernels ---------------------------------------------------- */

/* B~[k][n]: B[k][n] for the K x N layout, W[n][k] for the N x K layout. */
static double b_at(const uint16_t *B, int layout, int64_t N, int64_t K,
                   int64_t k, int64_t n)
{
    if (layout == LAYOUT_KN)
        return oracle_bf16_to_f64(B[k * N + n]);
    return oracle_bf16_to_f64(B[n * K + k]);
}

/* sum_k A[m][k] * B~[k][n] in fp64, k ascending. */
static double dot_ab(const uint16_t *A, const uint16_t *B, int layout,
                     int64_t N, int64_t K, int64_t m, int64_t n)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k)
        acc += oracle_bf16_to_f64(A[m * K + k]) * b_at(B, layout, N, K, k, n);
    return acc;
}

/* act(alpha*acc + beta*C + bias) + residual, fp64. Null operands are zero;
 * C is ignored when null (so beta does not matter then). */
static double epilogue(double acc, const uint16_t *C, const uint16_t *bias,
                       const uint16_t *residual, int64_t N, int64_t m,
                       int64_t n, double alpha, double beta, int act)
{
    double v = alpha * acc;
    if (C)
        v += beta * oracle_bf16_to_f64(C[m * N + n]);
    if (bias)
        v += oracle_bf16_to_f64(bias[n]);
    v = oracle_act(act, v);
    if (residual)
        v += oracle_bf16_to_f64(residual[m * N + n]);
    return v;
}

/* Dequantised weight w[k][n] = bf16((q - 8) * s[k/G][n]) as a double.
 * Wq is K x N/2 bytes; byte j of row k holds column 2j in its high nibble
 * and column 2j+1 in its low nibble. */
static double w4_at(const uint8_t *Wq, const uint16_t *scales, int64_t G,
                    int64_t N, int64_t k, int64_t n)
{
    uint8_t byte = Wq[k * (N / 2) + n / 2];
    int q = (n % 2 == 0) ? (byte >> 4) & 0xF : byte & 0xF;
    double s = oracle_bf16_to_f64(scales[(k / G) * N + n]);
    return oracle_bf16_to_f64(oracle_bf16_from_f64(((double)q - 8.0) * s));
}

/* OCP FP8 E4M3 (bias 7, 3 mantissa bits, subnormals, no infinities; the
 * two codes S.1111.111 are NaN), decoded from its definition. */
double oracle_fp8_e4m3_to_f64(uint8_t b)
{
    int sign = (b >> 7) & 1, e = (b >> 3) & 0xF, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* OCP FP4 E2M1 (bias 1, 1 mantissa bit, subnormal 0.5), low 4 bits of b. */
double oracle_fp4_e2m1_to_f64(uint8_t b)
{
    int sign = (b >> 3) & 1, e = (b >> 1) & 3, m = b & 1;
    double v = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
    return sign ? -v : v;
}

enum { WQ_INT4 = 0, WQ_FP8 = 1, WQ_NVFP4 = 2 };

/* Dequantised weight w[k][n] of format `kind` as a double (already rounded
 * to bf16, the precision the product consumes).  int4 and nvfp4 codes are
 * packed two per byte along N (column 2j in the high nibble of byte j, as
 * the int4 weights); fp8 codes are one byte each.  Scales: int4 and fp8 take
 * bf16 `scales` [K/G][N]; nvfp4 takes E4M3 bytes [K/16][N]. */
static double wq_at(int kind, const uint8_t *Wq, const void *scales, int64_t G,
                    int64_t N, int64_t k, int64_t n)
{
    double q, s;
    if (kind == WQ_FP8) {
        q = oracle_fp8_e4m3_to_f64(Wq[k * N + n]);
        s = oracle_bf16_to_f64(((const uint16_t *)scales)[(k / G) * N + n]);
    } else {
        uint8_t byte = Wq[k * (N / 2) + n / 2];
        int code = (n % 2 == 0) ? (byte >> 4) & 0xF : byte & 0xF;
        if (kind == WQ_INT4) {
            q = (double)code - 8.0;
            s = oracle_bf16_to_f64(((const uint16_t *)scales)[(k / G) * N + n]);
        } else {
            q = oracle_fp4_e2m1_to_f64((uint8_t)code);
            s = oracle_fp8_e4m3_to_f64(((const uint8_t *)scales)[(k / 16) * N + n]);
        }
    }
    return oracle_bf16_to_f64(oracle_bf16_from_f64(q * s));
}

static int wq_args_ok(int kind, int64_t G, int64_t N, int64_t K)
{
    if (K < 0 || N < 0 || kind < WQ_INT4 || kind > WQ_NVFP4)
        return 0;
    if (kind == WQ_NVFP4)
        return N % 2 == 0 && K % 16 == 0;
    if (G <= 0 || K % G != 0)
        return 0;
    return kind == WQ_FP8 || N % 2 == 0;
}

/* Element iteration helper: idx_m/idx_n == NULL means all M x N in row-major
 * order (count must then be M*N); otherwise count explicit (m, n) pairs. */
static void elem(const int64_t *idx_m, const int64_t *idx_n, int64_t N,
                 int64_t i, int64_t *m, int64_t *n)
{
    if (idx_m) {
        *m = idx_m[i];
        *n = idx_n[i];
    } else {
        *m = i / N;
        *n = i % N;
    }
}

/* 0 when every requested (m, n) lies inside the M x N output, -1 otherwise
 * (checked before any work, so the element loops below never stop early). */
static int elems_ok(const int64_t *idx_m, const int64_t *idx_n, int64_t M, int64_t N,
                    int64_t count)
{
    if (!idx_m)
        return count == M * N ? 0 : -1;
    for (int64_t i = 0; i < count; ++i)
        if (idx_m[i] < 0 || idx_m[i] >= M || idx_n[i] < 0 || idx_n[i] >= N)
            return -1;
    return 0;
}

static void emit(int64_t i, double v, uint16_t *out_bf16, double *out_f64)
{
    if (out_bf16)
        out_bf16[i] = oracle_bf16_from_f64(v);
    if (out_f64)
        out_f64[i] = v;
}

/* ---- public entry points ------------------------------------------------
 * Every function writes `count` results: out_bf16[i] (rounded once) and/or
 * out_f64[i] (the fp64 value before that rounding).  Returns 0, or -1 on a
 * bad argument. */

/* Fused GEMM + epilogue ("Fusion and Epilogues", epilogue fusion bullet;
 * "Kernel fusion" guide, Concept).  unfused != 0 rounds the plain product
 * D = A*B to bf16 before the pointwise pass, as a separate GEMM kernel that
 * writes D to memory would ("kernel fusion" wiki, activation after a matrix
 * product). */
int oracle_gemm_epilogue(const uint16_t *A, const uint16_t *B, int layout,
                         const uint16_t *C, const uint16_t *bias,
                         const uint16_t *residual, int64_t M, int64_t N,
                         int64_t K, double alpha, double beta, int act,
                         int unfused, const int64_t *idx_m,
                         const int64_t *idx_n, int64_t count,
                         uint16_t *out_bf16, double *out_f64)
{
    if (M < 0 || N < 0 || K < 0 || (layout != LAYOUT_KN && layout != LAYOUT_NK))
        return -1;
    if (elems_ok(idx_m, idx_n, M, N, count) != 0)
        return -1;
    ORACLE_PARALLEL_FOR
    for (int64_t i = 0; i < count; ++i) {
        int64_t m, n;
        elem(idx_m, idx_n, N, i, &m, &n);
        double acc = dot_ab(A, B, layout, N, K, m, n);
        if (unfused)
            acc = oracle_bf16_to_f64(oracle_bf16_from_f64(acc));
        emit(i, epilogue(acc, C, bias, residual, N, m, n, alpha, beta, act),
             out_bf16, out_f64);
    }
    return 0;
}

/* Gate/up dual GEMM with the GLU ending ("Fusion Thinking", Pattern 2):
 * g = x*W_gate~, u = x*W_up~ (same layout rule as gemm_epilogue),
 * h = act(alpha*g) * (alpha*u) + beta*C.  unfused != 0 rounds g and u to
 * bf16 first, as two separate GEMMs writing them to memory would. */
int oracle_swiglu(const uint16_t *x, const uint16_t *w_gate,
                  const uint16_t *w_up, int layout, const uint16_t *C,
                  int64_t M, int64_t N, int64_t K, double alpha, double beta,
                  int act, int unfused, const int64_t *idx_m,
                  const int64_t *idx_n, int64_t count, uint16_t *out_bf16,
                  double *out_f64)
{
    if (M < 0 || N < 0 || K < 0 || (layout != LAYOUT_KN && layout != LAYOUT_NK))
        return -1;
    if (elems_ok(idx_m, idx_n, M, N, count) != 0)
        return -1;
    ORACLE_PARALLEL_FOR
    for (int64_t i = 0; i < count; ++i) {
        int64_t m, n;
        elem(idx_m, idx_n, N, i, &m, &n);
        double g = dot_ab(x, w_gate, layout, N, K, m, n);
        double u = dot_ab(x, w_up, layout, N, K, m, n);
        if (unfused) {
            g = oracle_bf16_to_f64(oracle_bf16_from_f64(g));
            u = oracle_bf16_to_f64(oracle_bf16_from_f64(u));
        }
        double h = oracle_act(act, alpha * g) * (alpha * u);
        if (C)
            h += beta * oracle_bf16_to_f64(C[m * N + n]);
        emit(i, h, out_bf16, out_f64);
    }
    return 0;
}

/* Weight-only int4 GEMM ("Fusion Thinking", Pattern 3): the gemm_epilogue
 * formula with B~[k][n] = bf16((q[k][n] - 8) * s[k/G][n]).  The unfused
 * composition materialises the same bf16 weight, so it has the same
 * result; there is no separate unfused mode. */
int oracle_w4a16(const uint16_t *A, const uint8_t *Wq, const uint16_t *scales,
                 int64_t G, const uint16_t *C, const uint16_t *bias,
                 const uint16_t *residual, int64_t M, int64_t N, int64_t K,
                 double alpha, double beta, int act, const int64_t *idx_m,
                 const int64_t *idx_n, int64_t count, uint16_t *out_bf16,
                 double *out_f64)
{
    if (M < 0 || N < 0 || K < 0 || G <= 0 || N % 2 != 0 || K % G != 0)
        return -1;
    if (elems_ok(idx_m, idx_n, M, N, count) != 0)
        return -1;
    ORACLE_PARALLEL_FOR
    for (int64_t i = 0; i < count; ++i) {
        int64_t m, n;
        elem(idx_m, idx_n, N, i, &m, &n);
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += oracle_bf16_to_f64(A[m * K + k]) * w4_at(Wq, scales, G, N, k, n);
        emit(i, epilogue(acc, C, bias, residual, N, m, n, alpha, beta, act),
             out_bf16, out_f64);
    }
    return 0;
}

/* Weight-only GEMM of any of the three formats (wq_at): the gemm_epilogue
 * formula with B~ = the dequantised weight ("Fusion Thinking", Pattern 3).
 * G is ignored for nvfp4 (its blocks are 16 along K). */
int oracle_wq_gemm(int kind, const uint16_t *A, const uint8_t *Wq, const void *scales,
                   int64_t G, const uint16_t *C, const uint16_t *bias,
                   const uint16_t *residual, int64_t M, int64_t N, int64_t K,
                   double alpha, double beta, int act, const int64_t *idx_m,
                   const int64_t *idx_n, int64_t count, uint16_t *out_bf16,
                   double *out_f64)
{
    if (M < 0 || !wq_args_ok(kind, G, N, K))
        return -1;
    if (elems_ok(idx_m, idx_n, M, N, count) != 0)
        return -1;
    ORACLE_PARALLEL_FOR
    for (int64_t i = 0; i < count; ++i) {
        int64_t m, n;
        elem(idx_m, idx_n, N, i, &m, &n);
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += oracle_bf16_to_f64(A[m * K + k]) * wq_at(kind, Wq, scales, G, N, k, n);
        emit(i, epilogue(acc, C, bias, residual, N, m, n, alpha, beta, act),
             out_bf16, out_f64);
    }
    return 0;
}

/* The dequantised weight of any format on its own, K x N bf16. */
int oracle_wq_dequant(int kind, const uint8_t *Wq, const void *scales, int64_t G,
                      int64_t K, int64_t N, uint16_t *w_out)
{
    if (!wq_args_ok(kind, G, N, K))
        return -1;
    ORACLE_PARALLEL_FOR
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n)
            w_out[k * N + n] = oracle_bf16_from_f64(wq_at(kind, Wq, scales, G, N, k, n));
    return 0;
}

/* The dequantised weight on its own, K x N bf16 ("Fusion Thinking",
 * Pattern 3 un-fused: w_bf16 = dequantize(w_quant, scales)). */
int oracle_dequant_int4(const uint8_t *Wq, const uint16_t *scales, int64_t G,
                        int64_t K, int64_t N, uint16_t *w_out)
{
    if (K < 0 || N < 0 || G <= 0 || N % 2 != 0 || K % G != 0)
        return -1;
    ORACLE_PARALLEL_FOR
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n)
            w_out[k * N + n] = oracle_bf16_from_f64(w4_at(Wq, scales, G, N, k, n));
    return 0;
}

/* The pointwise pass alone, given an already-rounded bf16 product D
 * (used to check the unfused composition stage by stage). */
int oracle_pointwise_epilogue(const uint16_t *D, const uint16_t *C,
                              const uint16_t *bias, const uint16_t *residual,
                              int64_t M, int64_t N, double alpha, double beta,
                              int act, uint16_t *out_bf16)
{
    if (M < 0 || N < 0)
        return -1;
    ORACLE_PARALLEL_FOR
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            out_bf16[m * N + n] = oracle_bf16_from_f64(
                epilogue(oracle_bf16_to_f64(D[m * N + n]), C, bias, residual,
                         N, m, n, alpha, beta, act));
    return 0;
}

/* The GLU pointwise pass alone, given bf16 g and u. */
int oracle_swiglu_pointwise(const uint16_t *g, const uint16_t *u,
                            const uint16_t *C, int64_t M, int64_t N,
                            double alpha, double beta, int act,
                            uint16_t *out_bf16)
{
    if (M < 0 || N < 0)
        return -1;
    ORACLE_PARALLEL_FOR
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double h = oracle_act(act, alpha * oracle_bf16_to_f64(g[m * N + n])) *
                       (alpha * oracle_bf16_to_f64(u[m * N + n]));
            if (C)
                h += beta * oracle_bf16_to_f64(C[m * N + n]);
            out_bf16[m * N + n] = oracle_bf16_from_f64(h);
        }
    return 0;
}

/* Fused residual add + RMSNorm ("Fusion Thinking", Pattern 1): per row m,
 * r_j = a[m][j] + x[m][j] (exact in fp64), out_resid = bf16(r),
 * out_norm = bf16(r_j / sqrt(sum_j r_j^2 / N + eps) * w[j]).  unfused != 0
 * normalises the bf16-rounded residual instead, as a separate RMSNorm kernel
 * reading the stored residual would ("x = x + a; rmsnorm(x)"). */
int oracle_add_rmsnorm(const uint16_t *a, const uint16_t *x, const uint16_t *w, int64_t M,
                       int64_t N, double eps, int unfused, uint16_t *out_norm,
                       uint16_t *out_resid)
{
    if (M < 0 || N <= 0 || eps < 0.0)
        return -1;
    ORACLE_PARALLEL_FOR
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double r = oracle_bf16_to_f64(a[m * N + j]) + oracle_bf16_to_f64(x[m * N + j]);
            uint16_t rb = oracle_bf16_from_f64(r);
            if (out_resid)
                out_resid[m * N + j] = rb;
            if (unfused)
                r = oracle_bf16_to_f64(rb);
            ss += r * r;
        }
        double rrms = 1.0 / sqrt(ss / (double)N + eps);
        for (int64_t j = 0; j < N; ++j) {
            double r = oracle_bf16_to_f64(a[m * N + j]) + oracle_bf16_to_f64(x[m * N + j]);
            if (unfused)
                r = oracle_bf16_to_f64(oracle_bf16_from_f64(r));
            out_norm[m * N + j] = oracle_bf16_from_f64(r * rrms * oracle_bf16_to_f64(w[j]));
        }
    }
    return 0;
}
