/*
 * ck_oracle.c -- plain, slow, obviously correct CPU oracle for the INT8 quantized
 * linear layer.  TEST INFRASTRUCTURE ONLY: nothing in the product path may call it.
 * Only tests/, __graft_entry__.smoke() and the cpu_baseline / reference leg of
 * bench.py load this library.  It shares no code, header or table with the CUDA
 * library under int8_weight_quantized_gb300/csrc/.
 *
 * What it computes (sources are the comfy-kitchen issue and PR pages):
 *   y[m,n] = bf16( ((float(acc[m,n]) * x_scale[m]) * w_scale[n]) + bias[n] )
 *   acc[m,n] = sum_k q[m,k] * w[n,k]                       (exact integer)
 *   q[m,k]   = clamp(rint(v[m,k] / x_scale[m]), -127, 127),  x_scale[m] = amax_k|v[m,k]| / 127
 *   v        = x                  (per-row / tensorwise modes)
 *   v        = x @ H              (ConvRot mode, H = blockdiag of normalized Sylvester H_128)
 * and the 16-bit-activation path of the same layer (no activation quantize):
 *   y[m,n] = w_scale[n] * sum_k a[m,k] * w[n,k] + bias[n],  a = x or bf16(x @ H)
 * (ck_oracle_w8a16_linear, readings R12-R14 there).
 *
 *   - epilogue and its fp32 operation order: issue #280 "INT8 linears on sm_121 (GB10 /
 *     DGX Spark) run at ~37% of tensor-core peak ...", sections "Kernel used" and
 *     "Exactness" (acc * x_scale[m] * w_scale[n] (+ bias[n]), fp32, same order as the
 *     CUTLASS epilogue; int32 accumulation is exact);
 *   - per-row activation quantize: issue #278 "int8_linear silently falls back to a
 *     DP4A-emulated INT8 GEMM on Volta (sm_70) ...", section "2. quantize_int8_rowwise
 *     raises instead of falling back" (the op quantize_int8_rowwise);
 *   - tensorwise scales: issue #280, sections "Summary" (INT8 tensorwise linears) and
 *     "Exactness" (tensor-wide scales);
 *   - ConvRot: issue #278, section "Suggested fix" (stored weight W_rot = W @ H^T,
 *     activation rotated online x_rot = x @ H, GEMM entirely in the rotated basis);
 *   - int64 addressing: issue #136 "INT8 GEMM kernels index the output in int32:
 *     illegal memory access once m*n >= 2**31", sections "Summary" and "Suggested fix".
 *
 * Readings where the pages are silent:
 *   R1 rint is round-half-to-even (nearbyintf in the default FE_TONEAREST mode).
 *   R2 v / x_scale is one IEEE fp32 division (not a multiply by a reciprocal).
 *   R3 a row whose x_scale is 0 (all zeros, or amax so small that amax/127 underflows)
 *      quantizes to all-zero q.
 *   R4 the epilogue is evaluated left to right with a rounding after every operation
 *      (no fused multiply-add); bias bf16 -> fp32 is exact.  Build with
 *      -ffp-contract=off so the compiler cannot fuse.
 *   R5 H is applied per 128-element block as an fp32 fast Walsh-Hadamard transform in
 *      natural (Sylvester) order, butterfly spans 1,2,4,...,64 in ascending order,
 *      (lo, hi) -> (lo + hi, lo - hi), followed by one multiply with fp32(1/sqrt(128)).
 *      x_rot stays fp32 (never rounded to bf16).
 *   R6 the clamp is symmetric, [-127, 127].
 *
 * Floating point: fp32 wherever the pages fix fp32 (the epilogue, the scales);
 * integer accumulation is done in int64 and checked to fit int32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- bf16 <-> fp32 (bf16 is the upper half of an IEEE binary32) ------------- */
static float bf16_bits_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* round-to-nearest-even of an fp32 to bf16; inputs here are finite */
static uint16_t f32_to_bf16_bits_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* round-to-nearest-even of an fp32 to IEEE binary16 (finite inputs; overflow gives
 * +-infinity, values below the smallest subnormal round to +-0 or the smallest one) */
static uint16_t f32_to_f16_bits_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    const uint32_t sign = (u >> 16) & 0x8000u;
    const uint32_t mag = u & 0x7FFFFFFFu;
    if (mag >= 0x47800000u) {          /* |f| >= 65536: overflow (65520 and up round here too) */
        return (uint16_t)(sign | 0x7C00u);
    }
    if (mag >= 0x38800000u) {          /* |f| >= 2^-14: normal half */
        uint32_t exp = (mag >> 23) - 127 + 15;
        uint32_t man = mag & 0x7FFFFFu;
        uint32_t h = (exp << 10) | (man >> 13);
        uint32_t rem = man & 0x1FFFu;  /* 13 dropped bits */
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u)))
            h += 1;                    /* may carry into the exponent: still correct, 0x7C00 = inf */
        return (uint16_t)(sign | h);
    }
    /* subnormal half: value = m * 2^-24 with m in [0, 1023] */
    {
        int e = (int)(mag >> 23);      /* biased fp32 exponent */
        if (e < 102)                   /* |f| < 2^-25: rounds to zero */
            return (uint16_t)sign;
        uint32_t man = (mag & 0x7FFFFFu) | 0x800000u;  /* 24-bit significand, value man * 2^(e-150) */
        int shift = 126 - e;           /* man * 2^(e-150) / 2^-24 = man >> (126 - e) */
        uint32_t h = man >> shift;
        uint32_t rem = man & ((1u << shift) - 1u);
        uint32_t halfway = 1u << (shift - 1);
        if (rem > halfway || (rem == halfway && (h & 1u)))
            h += 1;
        return (uint16_t)(sign | h);
    }
}

/* exported for the pins: the same conversions, callable from tests */
uint16_t ck_oracle_f32_to_f16(float f) { return f32_to_f16_bits_rne(f); }
float ck_oracle_bf16_to_f32(uint16_t h) { return bf16_bits_to_f32(h); }
uint16_t ck_oracle_f32_to_bf16(float f) { return f32_to_bf16_bits_rne(f); }

int ck_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- ConvRot: one 128-block of x @ H (reading R5) ----------------------------
 * (x @ H)[j] = sum_i x[i] * H[i][j] with H[i][j] = (-1)^popcount(i & j) / sqrt(128).
 * The transform below evaluates exactly that sum with the butterfly factorisation
 * of the Sylvester matrix. */
void ck_oracle_fwht128(float *v)
{
    const float c128 = (float)(1.0 / sqrt(128.0)); /* 0x3DB504F3 */
    for (int h = 1; h < 128; h *= 2) {
        for (int i = 0; i < 128; i++) {
            if ((i & h) == 0) {
                float lo = v[i];
                float hi = v[i + h];
                v[i] = lo + hi;
                v[i + h] = lo - hi;
            }
        }
    }
    for (int i = 0; i < 128; i++)
        v[i] = v[i] * c128;
}

/* quantize one value with the row scale s (readings R1, R2, R3, R6) */
static int8_t quantize_value(float v, float s)
{
    if (s == 0.0f)
        return 0;
    float r = nearbyintf(v / s);
    if (r > 127.0f)
        r = 127.0f;
    if (r < -127.0f)
        r = -127.0f;
    return (int8_t)(int)r;
}

/* load row m of x as fp32, rotated if asked (ConvRot needs K % 128 == 0) */
static void load_row(const uint16_t *x, int64_t m, int64_t K, int rotate, float *v)
{
    for (int64_t k = 0; k < K; k++)
        v[k] = bf16_bits_to_f32(x[m * K + k]);
    if (rotate)
        for (int64_t b = 0; b < K; b += 128)
            ck_oracle_fwht128(v + b);
}

/* Per-row quantize (issue #278, quantize_int8_rowwise):
 *   x_scale[m] = max_k |v[m,k]| / 127 (fp32), q = clamp(rint(v / x_scale), -127, 127).
 * x: bf16 bits [M,K] row-major.  q: int8 [M,K].  xs: fp32 [M].
 * Returns 0, or -1 on a bad argument. */
int ck_oracle_quantize_rowwise(const uint16_t *x, int64_t M, int64_t K, int rotate,
                               int8_t *q, float *xs)
{
    if (M < 0 || K <= 0 || (rotate && K % 128 != 0))
        return -1;
    int bad = 0;
#pragma omp parallel
    {
        float *v = (float *)malloc((size_t)K * sizeof(float));
        if (!v) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t m = 0; m < M; m++) {
                load_row(x, m, K, rotate, v);
                float amax = 0.0f;
                for (int64_t k = 0; k < K; k++) {
                    float a = fabsf(v[k]);
                    if (a > amax)
                        amax = a;
                }
                float s = amax / 127.0f;
                xs[m] = s;
                for (int64_t k = 0; k < K; k++)
                    q[m * K + k] = quantize_value(v[k], s);
            }
            free(v);
        }
    }
    return bad ? -1 : 0;
}

/* Tensorwise quantize (issue #280, tensor-wide scales): one scale for the whole
 * tensor, x_scale = max_{m,k} |x[m,k]| / 127, then the same per-element rule. */
int ck_oracle_quantize_tensorwise(const uint16_t *x, int64_t M, int64_t K, int8_t *q, float *xs1)
{
    if (M < 0 || K <= 0)
        return -1;
    int64_t total = M * K;
    float amax = 0.0f;
    for (int64_t i = 0; i < total; i++) {
        float a = fabsf(bf16_bits_to_f32(x[i]));
        if (a > amax)
            amax = a;
    }
    float s = amax / 127.0f;
    xs1[0] = s;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < total; i++)
        q[i] = quantize_value(bf16_bits_to_f32(x[i]), s);
    return 0;
}

/* INT8 x INT8 -> int32 GEMM, acc[m,n] = sum_k q[m,k] * w[n,k] (issue #280, "Exactness":
 * the int32 accumulation is exact).  q: [M,K], w: [N,K] (both K contiguous),
 * acc: [M,N].  The sum is formed in int64 so it can never wrap; |acc| <= 127*127*K,
 * which fits int32 for K <= 133144 (checked).  Returns 0, -1 on a bad argument, -2 if
 * a sum did not fit int32. */
int ck_oracle_gemm_s32(const int8_t *q, const int8_t *w, int32_t *acc, int64_t M, int64_t N, int64_t K)
{
    if (M < 0 || N < 0 || K <= 0)
        return -1;
    int overflow = 0;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++) {
        for (int64_t n = 0; n < N; n++) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; k++)
                s += (int64_t)q[m * K + k] * (int64_t)w[n * K + k];
            if (s > INT32_MAX || s < INT32_MIN) {
#pragma omp atomic write
                overflow = 1;
            }
            acc[m * N + n] = (int32_t)s;
        }
    }
    return overflow ? -2 : 0;
}

/* fp32 dequant epilogue (issue #280, "Kernel used" / "Exactness"; reading R4):
 *   t = float(acc); t = t * xs; t = t * ws; if bias: t = t + float(bias); y = bf16(t).
 * scalar_scales != 0: xs and ws each hold one value (tensorwise).
 * bias may be NULL. */
void ck_oracle_dequant(const int32_t *acc, const float *xs, const float *ws, const uint16_t *bias,
                       int scalar_scales, int64_t M, int64_t N, uint16_t *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++) {
        float xsm = scalar_scales ? xs[0] : xs[m];
        for (int64_t n = 0; n < N; n++) {
            float wsn = scalar_scales ? ws[0] : ws[n];
            float t = (float)acc[m * N + n];
            t = t * xsm;
            t = t * wsn;
            if (bias)
                t = t + bf16_bits_to_f32(bias[n]);
            y[m * N + n] = f32_to_bf16_bits_rne(t);
        }
    }
}

/* The same epilogue with the output type of the pages' int8_linear(..., out_dtype):
 * out_dtype 0 = bf16, 1 = fp16, 2 = fp32; y holds M*N values of that type.  The fp32
 * value t is the same in every case; only the final rounding differs (none for fp32). */
void ck_oracle_dequant_typed(const int32_t *acc, const float *xs, const float *ws, const uint16_t *bias,
                             int scalar_scales, int64_t M, int64_t N, int out_dtype, void *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++) {
        float xsm = scalar_scales ? xs[0] : xs[m];
        for (int64_t n = 0; n < N; n++) {
            float wsn = scalar_scales ? ws[0] : ws[n];
            float t = (float)acc[m * N + n];
            t = t * xsm;
            t = t * wsn;
            if (bias)
                t = t + bf16_bits_to_f32(bias[n]);
            if (out_dtype == 2)
                ((float *)y)[m * N + n] = t;
            else if (out_dtype == 1)
                ((uint16_t *)y)[m * N + n] = f32_to_f16_bits_rne(t);
            else
                ((uint16_t *)y)[m * N + n] = f32_to_bf16_bits_rne(t);
        }
    }
}

/* The epilogue with a residual added (issue #280, section "Kernel used", mentions
 * residual-fused calls of the dequant GEMM).  Reading R15: the residual r[m,n] is given
 * in the output type and added in fp32 after the bias, one more separately rounded
 * operation:  y = out((((float(acc) * xs) * ws) + bias) + r).  r holds fp32 values (the
 * caller converts its bf16 / fp16 / fp32 tensor exactly). */
void ck_oracle_dequant_residual(const int32_t *acc, const float *xs, const float *ws, const uint16_t *bias,
                                const float *r, int scalar_scales, int64_t M, int64_t N, int out_dtype, void *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++) {
        float xsm = scalar_scales ? xs[0] : xs[m];
        for (int64_t n = 0; n < N; n++) {
            float wsn = scalar_scales ? ws[0] : ws[n];
            float t = (float)acc[m * N + n];
            t = t * xsm;
            t = t * wsn;
            if (bias)
                t = t + bf16_bits_to_f32(bias[n]);
            t = t + r[m * N + n];
            if (out_dtype == 2)
                ((float *)y)[m * N + n] = t;
            else if (out_dtype == 1)
                ((uint16_t *)y)[m * N + n] = f32_to_f16_bits_rne(t);
            else
                ((uint16_t *)y)[m * N + n] = f32_to_bf16_bits_rne(t);
        }
    }
}

/* The whole linear layer in one call.  mode: 0 tensorwise, 1 per-row, 2 ConvRot
 * (for ConvRot, w is the pre-rotated, pre-quantized W_rot and is used as is).
 * Optional outputs q_out [M,K], xs_out [M] (or [1]) and acc_out [M,N] may be NULL.
 * Returns 0 or a negative error. */
int ck_oracle_int8_linear(const uint16_t *x, const int8_t *w, const float *ws, const uint16_t *bias,
                          int64_t M, int64_t N, int64_t K, int mode, uint16_t *y,
                          int8_t *q_out, float *xs_out, int32_t *acc_out)
{
    if (mode < 0 || mode > 2)
        return -1;
    int8_t *q = q_out ? q_out : (int8_t *)malloc((size_t)(M * K));
    float *xs = xs_out ? xs_out : (float *)malloc(sizeof(float) * (size_t)(mode == 0 ? 1 : M));
    int32_t *acc = acc_out ? acc_out : (int32_t *)malloc(sizeof(int32_t) * (size_t)(M * N));
    int rc = 0;
    if (!q || !xs || !acc)
        rc = -3;
    if (rc == 0)
        rc = (mode == 0) ? ck_oracle_quantize_tensorwise(x, M, K, q, xs)
                         : ck_oracle_quantize_rowwise(x, M, K, mode == 2, q, xs);
    if (rc == 0)
        rc = ck_oracle_gemm_s32(q, w, acc, M, N, K);
    if (rc == 0)
        ck_oracle_dequant(acc, xs, ws, bias, mode == 0, M, N, y);
    if (!q_out)
        free(q);
    if (!xs_out)
        free(xs);
    if (!acc_out)
        free(acc);
    return rc;
}

/* ConvRot weight preparation (issue #278, "Suggested fix": the stored weight is
 * W_rot = W @ H^T, quantized per output row, and used as is by the GEMM).  H is
 * symmetric, so row n of W @ H^T is row n of W times H: the same block transform as
 * the activations.  Then w_scale[n] = max_k |W_rot[n,k]| / 127 and
 * w[n,k] = clamp(rint(W_rot[n,k] / w_scale[n]), -127, 127)  (readings R1-R3, R5, R6).
 * W: fp32 [N,K]; w: int8 [N,K]; ws: fp32 [N].  K % 128 == 0. */
int ck_oracle_prepare_convrot_weight(const float *W, int64_t N, int64_t K, int8_t *w, float *ws)
{
    if (N < 0 || K <= 0 || K % 128 != 0)
        return -1;
    int bad = 0;
#pragma omp parallel
    {
        float *v = (float *)malloc((size_t)K * sizeof(float));
        if (!v) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t n = 0; n < N; n++) {
                memcpy(v, W + n * K, (size_t)K * sizeof(float));
                for (int64_t b = 0; b < K; b += 128)
                    ck_oracle_fwht128(v + b);
                float amax = 0.0f;
                for (int64_t k = 0; k < K; k++) {
                    float a = fabsf(v[k]);
                    if (a > amax)
                        amax = a;
                }
                float s = amax / 127.0f;
                ws[n] = s;
                for (int64_t k = 0; k < K; k++)
                    w[n * K + k] = quantize_value(v[k], s);
            }
            free(v);
        }
    }
    return bad ? -1 : 0;
}

/* W8A16 linear: the 16-bit-activation path of issue #278 (section "Suggested fix":
 * dequantize the INT8 weight on the fly and run the GEMM on 16-bit tensor cores; the
 * stored weight keeps its INT8 footprint; for ConvRot the activation is rotated online,
 * x_rot = x @ H, the GEMM runs in the rotated basis and the weight is not rotated back).
 * Readings where the pages are silent:
 *   R12 the activation is not quantized: a = x as given (bf16), or for ConvRot
 *       a = bf16_rne(x @ H) with the fp32 block transform of R5 (16-bit tensor-core
 *       operands hold bf16, so the rotated activation is rounded once);
 *   R13 "dequantize on the fly" multiplies each code by w_scale[n]; this oracle keeps
 *       the exact real-number result of that definition,
 *           y[m,n] = w_scale[n] * sum_k a[m,k] * w[n,k] + bias[n],
 *       which equals sum_k a[m,k] * (w[n,k] * w_scale[n]) + bias[n] exactly;
 *   R14 tensorwise mode has one w_scale, per-row and ConvRot one per output row.
 * The sum is taken in double: every product a*w is exact in double (8 + 7 significant
 * bits) and K <= 131072 partial sums of magnitude < 2^53 ulps stay exact enough that
 * the result is the real value to within 2^-50 relative of sum |a*w|.  The caller gets
 * y (double, before any output rounding) and mag[m,n] = |w_scale[n]| * sum_k |a*w|,
 * which bounds the rounding error of any fp32 evaluation of the same sum.
 * x: bf16 bits [M,K]; w: int8 [N,K]; ws: fp32 [N] or [1]; bias: bf16 bits [N] or NULL.
 * Returns 0, or -1 on a bad argument / allocation failure. */
int ck_oracle_w8a16_linear(const uint16_t *x, const int8_t *w, const float *ws, const uint16_t *bias,
                           int64_t M, int64_t N, int64_t K, int mode, double *y, double *mag)
{
    if (M < 0 || N < 0 || K <= 0 || mode < 0 || mode > 2 || (mode == 2 && K % 128 != 0))
        return -1;
    int bad = 0;
#pragma omp parallel
    {
        float *v = (float *)malloc((size_t)K * sizeof(float));
        double *a = (double *)malloc((size_t)K * sizeof(double));
        if (!v || !a) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t m = 0; m < M; m++) {
                load_row(x, m, K, mode == 2, v);
                for (int64_t k = 0; k < K; k++)
                    a[k] = mode == 2 ? (double)bf16_bits_to_f32(f32_to_bf16_bits_rne(v[k])) : (double)v[k];
                for (int64_t n = 0; n < N; n++) {
                    double s = 0.0, sa = 0.0;
                    for (int64_t k = 0; k < K; k++) {
                        double p = a[k] * (double)w[n * K + k];
                        s += p;
                        sa += fabs(p);
                    }
                    double wsn = (double)(mode == 0 ? ws[0] : ws[n]);
                    double b = bias ? (double)bf16_bits_to_f32(bias[n]) : 0.0;
                    y[m * N + n] = wsn * s + b;
                    mag[m * N + n] = fabs(wsn) * sa;
                }
            }
        }
        free(v);
        free(a);
    }
    return bad ? -1 : 0;
}
