/*
 * CPU oracle for the fused gated activations -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark may load this file's library.  The CUDA library never links,
 * includes or calls it, and it shares no code with the CUDA library.
 *
 * Everything here is plain fp64 C written straight from the definitions, one
 * loop per stage, with no blocking, fusion or reordering:
 *
 *  gelu_and_mul_sparse  -- vLLM PR "[Performance] Add Triton kernel for
 *      Gemma3n sparse GELU", section "Purpose": the activation fuses the row
 *      statistics, a threshold set from them, the tanh form of GELU and the
 *      product with the up half.  Reading of each stage (the page lists the
 *      stages but prints no formula):
 *        gate g = columns [0, d) of the row, up u = columns [d, 2d);
 *        mean   = sum_j g_j / d;
 *        var    = sum_j (g_j - mean)^2 / d       (population variance);
 *        cutoff = mean + sqrt(var) * z,  z = inverse normal CDF of the target
 *                 sparsity (passed in; 0.95 gives z = 1.6448536269514722);
 *        s_j    = max(g_j - cutoff, 0);
 *        out_j  = gelu_tanh(s_j) * u_j,
 *        gelu_tanh(x) = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
 *                 (the tanh form of GELU of Hendrycks and Gimpel, 2016).
 *
 *  silu_and_mul -- Megatron-LM PR "Size MoE activation kernel grid to the row
 *      count", section "What changed and why": the elementwise MoE activation
 *      out_j = silu(g_j) * u_j with silu(x) = x / (1 + exp(-x)), gate in the
 *      first d columns and up in the next d.  The bounded form of the same
 *      section (only the first n_rows live rows are computed) is this function
 *      called on those rows.
 *
 *  squared_relu -- same page, section "Scope and risks": the sibling MoE
 *      activation out_j = max(x_j, 0)^2 over [M, d] rows (not gated).
 *
 *  gelu_and_mul -- the dense form of the sparse-GELU page's activation (no
 *      threshold): out_j = gelu_tanh(g_j) * u_j.
 *
 * Inputs are bf16 bit patterns (uint16), decoded exactly to double; the
 * sparse GELU also takes fp16 and fp32 elements (the page validates all three
 * types).  The bf16 encoder below rounds a double to the nearest bf16, ties
 * to even, in one step (no detour through float, which would round twice).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_PI 3.14159265358979323846

/* Element types of the typed entry points (same numbering as the library's). */
enum { ORACLE_BF16 = 0, ORACLE_F16 = 1, ORACLE_F32 = 2 };

/*
 * Exact value of an IEEE binary16 bit pattern: sign, 5 exponent bits (bias
 * 15), 10 fraction bits; exponent 0 is subnormal (fraction * 2^-24), 31 is
 * infinity (fraction 0) or NaN.
 */
double oracle_f16_to_double(uint16_t bits)
{
    const int sign = bits >> 15, e = (bits >> 10) & 0x1F, f = bits & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);
    return sign ? -v : v;
}

/* Exact value of a bf16 bit pattern: the top 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest bf16 (8 significant bits, binary32 exponent
 * range), ties to even, with gradual underflow and overflow to infinity.
 * Method: pick the quantum 2^(e-7) of the binade of |v| (fixed at 2^-133
 * below the smallest normal 2^-126), divide by it (exact: a power of two),
 * round to the nearest integer with ties to even (rint in the default
 * rounding mode), scale back.
 */
uint16_t oracle_double_to_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    /* largest finite bf16 is (2 - 2^-7) 2^127; halfway to 2^128 rounds up */
    if (isinf(a) || a >= ldexp(2.0 - ldexp(1.0, -8), 127))
        return (uint16_t)(sign | 0x7F80u);
    int e2;
    frexp(a, &e2);            /* a = m 2^e2, m in [0.5, 1)  ->  binade 2^(e2-1) */
    int e = e2 - 1;
    if (e < -126)
        e = -126;
    double q = ldexp(1.0, e - 7);
    double r = rint(a / q) * q;   /* exactly representable in binary32 */
    float f = (float)r;
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    return (uint16_t)(sign | (uint16_t)(w >> 16));
}

/* Element j of a typed array, exactly, in double. */
static double load_elem(const void *base, int dtype, int64_t j)
{
    if (dtype == ORACLE_F32) {
        float f;
        memcpy(&f, (const char *)base + 4 * j, sizeof f);
        return (double)f;
    }
    uint16_t b;
    memcpy(&b, (const char *)base + 2 * j, sizeof b);
    return dtype == ORACLE_F16 ? oracle_f16_to_double(b) : oracle_bf16_to_double(b);
}

/*
 * tanh-approximate GELU, in double.  With y = sqrt(2/pi) (x + 0.044715 x^3),
 * gelu_tanh(x) = 0.5 x (1 + tanh(y)).  For y < 0 the sum 1 + tanh(y) cancels,
 * so that branch uses the exact identity 1 + tanh(y) = 2 e^{2y} / (1 + e^{2y}).
 */
double oracle_gelu_tanh(double x)
{
    const double k = sqrt(2.0 / ORACLE_PI);
    const double y = k * (x + 0.044715 * x * x * x);
    if (y < 0.0) {
        const double t = exp(2.0 * y);
        return x * t / (1.0 + t);
    }
    return 0.5 * x * (1.0 + tanh(y));
}

/* SiLU (swish), in double with libm exp. */
double oracle_silu(double x)
{
    return x / (1.0 + exp(-x));
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads an OpenMP region would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * gelu_and_mul_sparse, one row at a time, on elements of type `dtype`.
 *   in         : T rows of row_stride elements; gate = [0,d), up = [d,2d)
 *   ref        : T*d doubles, the unrounded result
 *   mask       : T*d bytes, 1 where g_j > cutoff (strictly), else 0
 *   row_mean, row_std, row_cutoff : T doubles each (any may be NULL)
 *   nthreads   : OpenMP threads over rows (<= 0: the runtime default)
 * Returns 0, or -1 on a bad size or type.
 */
int oracle_gelu_and_mul_sparse_typed(const void *in, int dtype, int64_t T, int64_t d,
                                     int64_t row_stride, double z, double *ref,
                                     uint8_t *mask, double *row_mean, double *row_std,
                                     double *row_cutoff, int nthreads)
{
    if (T < 0 || d <= 0 || row_stride < 2 * d || dtype < ORACLE_BF16 || dtype > ORACLE_F32)
        return -1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < T; ++r) {
        const int64_t g0 = r * row_stride, u0 = g0 + d;

        double sum = 0.0;
        for (int64_t j = 0; j < d; ++j)
            sum += load_elem(in, dtype, g0 + j);
        double mean = sum / (double)d;

        double ss = 0.0;
        for (int64_t j = 0; j < d; ++j) {
            double dev = load_elem(in, dtype, g0 + j) - mean;
            ss += dev * dev;
        }
        double var = ss / (double)d;
        double std = sqrt(var);

        double cutoff = mean + std * z;

        for (int64_t j = 0; j < d; ++j) {
            double g = load_elem(in, dtype, g0 + j);
            double u = load_elem(in, dtype, u0 + j);
            double s = g - cutoff;
            if (s < 0.0)
                s = 0.0;
            ref[r * d + j] = oracle_gelu_tanh(s) * u;
            if (mask)
                mask[r * d + j] = (uint8_t)(g > cutoff);
        }
        if (row_mean)
            row_mean[r] = mean;
        if (row_std)
            row_std[r] = std;
        if (row_cutoff)
            row_cutoff[r] = cutoff;
    }
    return 0;
}

/* gelu_and_mul_sparse on bf16 bit patterns (the library's default type). */
int oracle_gelu_and_mul_sparse(const uint16_t *in, int64_t T, int64_t d,
                               int64_t row_stride, double z, double *ref,
                               uint8_t *mask, double *row_mean,
                               double *row_std, double *row_cutoff,
                               int nthreads)
{
    return oracle_gelu_and_mul_sparse_typed(in, ORACLE_BF16, T, d, row_stride, z, ref, mask,
                                            row_mean, row_std, row_cutoff, nthreads);
}

/*
 * Round a double to the nearest IEEE binary16 value (ties to even, gradual
 * underflow, overflow to infinity) and return that value as a double.  Same
 * method as the bf16 encoder: the quantum of |v|'s binade is 2^(e-10), fixed
 * at 2^-24 below the smallest normal 2^-14.
 */
double oracle_round_f16(double v)
{
    if (isnan(v) || v == 0.0)
        return v;
    double a = fabs(v);
    if (isinf(a) || a >= 65520.0)      /* halfway between 65504 and 2^16 rounds up */
        return copysign(INFINITY, v);
    int e2;
    frexp(a, &e2);
    int e = e2 - 1;
    if (e < -14)
        e = -14;
    double q = ldexp(1.0, e - 10);
    return copysign(rint(a / q) * q, v);
}

/* Round a double to the nearest bf16 value, returned as a double. */
double oracle_round_bf16(double v)
{
    return oracle_bf16_to_double(oracle_double_to_bf16(v));
}

/*
 * gelu_and_mul_sparse in native-rounding mode: the op as a composition of
 * separate element-type ops, which the sparse-GELU page's kernel imitates
 * ("Cross-architecture warp and dtype validation": it rounds intermediates
 * back to the input type where PyTorch's separate ops would).  Each op of an element
 * type is computed in binary32 and its result rounded to the element type
 * (bf16 or fp16), so a boundary is R(x) = round_T(round_binary32(x)) with x
 * the op's exact value -- two roundings, which differ from one when the
 * binary32 result lands on a midpoint of the element type.  Boundaries:
 *   m = R(mean g),  sd = R(population std g)  (std from the exact mean),
 *   t = R(sd * zf)  with zf = z rounded to binary32 (a scalar operand),
 *   c = R(m + t),   s = max(R(g - c), 0),  a = R(gelu_tanh(s)),  out = R(a * u).
 * ref holds out (already rounded); mask is g > c; row_cutoff holds c.
 */
int oracle_gelu_and_mul_sparse_native(const void *in, int dtype, int64_t T, int64_t d,
                                      int64_t row_stride, double z, double *ref,
                                      uint8_t *mask, double *row_cutoff, int nthreads)
{
    if (T < 0 || d <= 0 || row_stride < 2 * d ||
        (dtype != ORACLE_BF16 && dtype != ORACLE_F16))
        return -1;
    double (*RT)(double) = dtype == ORACLE_F16 ? oracle_round_f16 : oracle_round_bf16;
#define R(x) RT((double)(float)(x))
    const double zf = (double)(float)z;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < T; ++r) {
        const int64_t g0 = r * row_stride, u0 = g0 + d;

        double sum = 0.0;
        for (int64_t j = 0; j < d; ++j)
            sum += load_elem(in, dtype, g0 + j);
        const double mean = sum / (double)d;
        double ss = 0.0;
        for (int64_t j = 0; j < d; ++j) {
            double dev = load_elem(in, dtype, g0 + j) - mean;
            ss += dev * dev;
        }
        const double m = R(mean);
        const double sd = R(sqrt(ss / (double)d));
        const double t = R(sd * zf);
        const double c = R(m + t);

        for (int64_t j = 0; j < d; ++j) {
            double g = load_elem(in, dtype, g0 + j);
            double u = load_elem(in, dtype, u0 + j);
            double s = R(g - c);
            if (s < 0.0)
                s = 0.0;
            double a = R(oracle_gelu_tanh(s));
            ref[r * d + j] = R(a * u);
            if (mask)
                mask[r * d + j] = (uint8_t)(g > c);
        }
        if (row_cutoff)
            row_cutoff[r] = c;
    }
#undef R
    return 0;
}

/* squared ReLU, in double. */
double oracle_squared_relu(double x)
{
    double r = x > 0.0 ? x : 0.0;
    if (isnan(x))
        r = x;
    return r * r;
}

/*
 * gelu_and_mul (dense): out = gelu_tanh(g) * u on [T, row_stride] rows.
 *   ref      : T*d doubles (may be NULL);  ref_bf16 : T*d bf16 patterns (may be NULL)
 */
int oracle_gelu_and_mul(const uint16_t *in, int64_t T, int64_t d, int64_t row_stride,
                        double *ref, uint16_t *ref_bf16, int nthreads)
{
    if (T < 0 || d <= 0 || row_stride < 2 * d)
        return -1;
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r) {
        const uint16_t *gate = in + r * row_stride;
        const uint16_t *up = gate + d;
        for (int64_t j = 0; j < d; ++j) {
            double y = oracle_gelu_tanh(oracle_bf16_to_double(gate[j])) *
                       oracle_bf16_to_double(up[j]);
            if (ref)
                ref[r * d + j] = y;
            if (ref_bf16)
                ref_bf16[r * d + j] = oracle_double_to_bf16(y);
        }
    }
    return 0;
}

/*
 * squared_relu over a contiguous [M, d] bf16 input.
 *   ref : M*d doubles (may be NULL);  ref_bf16 : M*d bf16 patterns (may be NULL)
 */
int oracle_squared_relu_rows(const uint16_t *in, int64_t M, int64_t d, double *ref,
                             uint16_t *ref_bf16, int nthreads)
{
    if (M < 0 || d <= 0)
        return -1;
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < M; ++r) {
        for (int64_t j = 0; j < d; ++j) {
            double y = oracle_squared_relu(oracle_bf16_to_double(in[r * d + j]));
            if (ref)
                ref[r * d + j] = y;
            if (ref_bf16)
                ref_bf16[r * d + j] = oracle_double_to_bf16(y);
        }
    }
    return 0;
}

/*
 * silu_and_mul over a contiguous [M, 2d] bf16 input.
 *   ref      : M*d doubles, silu(g) * u unrounded (may be NULL)
 *   ref_bf16 : M*d bf16 bit patterns, ref rounded to nearest-even (may be NULL)
 * Returns 0, or -1 on a bad size.
 */
int oracle_silu_and_mul(const uint16_t *in, int64_t M, int64_t d, double *ref,
                        uint16_t *ref_bf16, int nthreads)
{
    if (M < 0 || d <= 0)
        return -1;
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < M; ++r) {
        const uint16_t *gate = in + r * 2 * d;
        const uint16_t *up = gate + d;
        for (int64_t j = 0; j < d; ++j) {
            double y = oracle_silu(oracle_bf16_to_double(gate[j])) *
                       oracle_bf16_to_double(up[j]);
            if (ref)
                ref[r * d + j] = y;
            if (ref_bf16)
                ref_bf16[r * d + j] = oracle_double_to_bf16(y);
        }
    }
    return 0;
}
