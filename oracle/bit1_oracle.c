/*
 * bit1_oracle.c -- plain, slow, scalar CPU oracle for the true 1-bit
 * (sign bit + one fp16 scale per 128 inputs) linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg load this library.  It shares no
 * code, header, table or constant with the CUDA library: it decodes fp16 and
 * bf16 itself, extracts one bit at a time, accumulates in fp64 and rounds with
 * its own routines.
 *
 * Sources (web pages describing the method):
 *  [27B-bin]  "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진 및 삼진 저비트 LLM",
 *             section "이진(Binary) 가중치 형식" (binary weight format):
 *             w_i = s_g * b_i, b_i in {-1,+1}, one FP16 scale per group of 128,
 *             b_eff = 1 + 16/128 = 1.125 bits/weight.
 *  [27B-kern] same page, section "하이브리드 어텐션을 위한 저비트 커널":
 *             packed sign codes are decoded and the group FP16 scale is applied
 *             inside the fused matmul; accumulation stays in high precision.
 *  [27B-ter]  same page, section "삼진(Ternary) 가중치 형식" (ternary weight
 *             format): w_i = s_g * t_i, t_i in {-1, 0, +1}, one FP16 scale per
 *             group of 128, b_eff ~ log2(3) + 16/128 ~ 1.71 bits/weight.
 *  [27B-store] same page, section "저장 공간과 실제 배포 크기": binary weights
 *             are deployed in the native 1-bit layout; today's kernels keep
 *             each ternary value in a 2-bit slot (deployed ~7.2 GB against
 *             the ~5.9 GB minimum).
 *  [Bankai]   "LocalLLaMA, true 1-bit LLM용 XOR patch 방식 \"Bankai\" 실험에 주목",
 *             section "LocalLLaMA가 본 핵심 포인트": a patch is a list of
 *             (layer, projection, row) entries whose binary weights are
 *             flipped; applying and removing are the same XOR.
 *  [27B-arch] same page, section "Bonsai 27B의 표현 방식": the base model
 *             keeps its architecture, whose MLP is SwiGLU; the MLP
 *             projections are binary like every other matrix.
 *  [8B-what]  "PrismML Bonsai — 1.15GB짜리 8B 모델이 말이 되나?", section
 *             "1-bit이 뭔지부터": weights are {-1,+1}; multiplies become
 *             additions and subtractions.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes):
 *  - bit 1 means +1, bit 0 means -1.
 *  - bits are stored row-major [N][K/8], k ascending, least significant bit
 *    first inside each byte: bit(n,k) = (bits[n*K/8 + k/8] >> (k%8)) & 1.
 *  - scales are stored row-major [N][K/128] as IEEE binary16 bit patterns.
 *  - packing: bit = !(w < 0) (so +0, -0 -> 1); scale = fp16 round-to-nearest-
 *    even of the mean of |w| over the group, the 128 magnitudes summed in
 *    fp64 in ascending k order and divided by 128.  A NaN weight gives
 *    status 5 (ENAN); a scale that is not finite gives status 3 (ERANGE).
 *  - K must be a positive multiple of 128.
 *  - a patch entry flips all K bits of its row; scales are untouched;
 *    duplicate rows flip once per occurrence.
 *
 * Ternary ([27B-ter], [27B-store]).  Reading of the 2-bit slot, which the
 * pages do not lay out: two bit planes a and b, each in the binary layout
 * above, with t = (a + b) / 2 when a bit is read as +-1 (bit 1 -> +1):
 * (1,1) -> +1, (0,0) -> -1, (1,0) and (0,1) -> 0.  Codes to planes:
 * a = (t >= 0), b = (t > 0).  Both planes share the one scale array.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ESHAPE 2
#define ORC_ERANGE 3
#define ORC_ENAN 5

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F16 2

/* ---- number decoding (exact) ------------------------------------------ */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);              /* zero / subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);  /* (1024+m) * 2^(e-15-10) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double orc_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int m = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);             /* m * 2^(-126-7) */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 128), e - 134);  /* (128+m) * 2^(e-127-7) */
    return sign ? -v : v;
}

static double orc_f32_to_double(const void *p)
{
    float f;
    memcpy(&f, p, 4);
    return (double)f;
}

/* ---- rounding fp64 -> narrow formats, round to nearest, ties to even ---- */

/* Generic: |a| rounded to a grid of significand width `p` bits with minimum
 * normal exponent `emin` and largest finite value `maxv`.  Returns the rounded
 * magnitude (possibly INFINITY). */
static double orc_round_grid(double a, int p, int emin, double maxv)
{
    int e;
    double q, n, r;
    if (a == 0.0)
        return 0.0;
    frexp(a, &e);         /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;               /* a in [2^e, 2^(e+1)) */
    if (e < emin)
        e = emin;         /* subnormal range: fixed quantum */
    q = ldexp(1.0, e - (p - 1));
    n = nearbyint(a / q); /* a/q is exact (power-of-two scaling); RNE */
    r = n * q;
    if (r > maxv)
        return INFINITY;
    return r;
}

uint16_t orc_double_to_half(double v)
{
    int sign = signbit(v) ? 1 : 0;
    double a = fabs(v), r;
    int e, n;
    if (isnan(v))
        return (uint16_t)((sign << 15) | 0x7e00);
    r = orc_round_grid(a, 11, -14, 65504.0);
    if (isinf(r))
        return (uint16_t)((sign << 15) | 0x7c00);
    if (r < ldexp(1.0, -14)) {               /* subnormal or zero */
        n = (int)(r * ldexp(1.0, 24));
        return (uint16_t)((sign << 15) | n);
    }
    frexp(r, &e);
    e -= 1;                                   /* r in [2^e, 2^(e+1)) */
    n = (int)(r * ldexp(1.0, 10 - e)) - 1024; /* fraction field */
    return (uint16_t)((sign << 15) | ((e + 15) << 10) | n);
}

uint16_t orc_double_to_bf16(double v)
{
    int sign = signbit(v) ? 1 : 0;
    double a = fabs(v), r;
    int e, n;
    double maxv = ldexp(255.0, 120);          /* (2 - 2^-7) * 2^127 */
    if (isnan(v))
        return (uint16_t)((sign << 15) | 0x7fc0);
    r = orc_round_grid(a, 8, -126, maxv);
    if (isinf(r))
        return (uint16_t)((sign << 15) | 0x7f80);
    if (r < ldexp(1.0, -126)) {
        n = (int)(r * ldexp(1.0, 133));
        return (uint16_t)((sign << 15) | n);
    }
    frexp(r, &e);
    e -= 1;
    n = (int)(r * ldexp(1.0, 7 - e)) - 128;
    return (uint16_t)((sign << 15) | ((e + 127) << 7) | n);
}

/* ---- the weight format ---------------------------------------------- */

/* Bytes of one packed matrix: N*K/8 sign bytes + N*(K/128) fp16 scales
 * ([27B-bin]: 1 + 16/128 = 1.125 bits per weight). */
int64_t orc_footprint_bytes(int64_t N, int64_t K)
{
    return N * K / 8 + 2 * N * (K / 128);
}

/* One sign bit, read on its own. */
static int orc_bit(const uint8_t *bits, int64_t K, int64_t n, int64_t k)
{
    return (bits[n * (K / 8) + k / 8] >> (k % 8)) & 1;
}

static int orc_check_shape(int64_t B, int64_t N, int64_t K)
{
    if (B < 1 || N < 1 || K < 128 || K % 128 != 0)
        return ORC_ESHAPE;
    return ORC_OK;
}

/* ---- the linear layer -------------------------------------------------
 * y[b,n] = sum_g s[n,g] * sum_{k in group g} (bit(n,k) ? +x[b,k] : -x[b,k])
 * ([27B-bin] weight definition, [27B-kern] scale applied per group inside
 * the product, high-precision accumulation; [8B-what] no multiply per
 * weight).  Scalar loops, fp64 accumulation, the group partial sum first and
 * then one multiply by the group's scale.  Rows [n0, n1) only. */
static void orc_gemv_rows(const uint8_t *bits, const uint16_t *scales,
                          const uint16_t *x, int64_t B, int64_t N, int64_t K,
                          int64_t n0, int64_t n1, double *y)
{
    int64_t G = K / 128;
    for (int64_t b = 0; b < B; b++) {
        for (int64_t n = n0; n < n1; n++) {
            double acc = 0.0;
            for (int64_t g = 0; g < G; g++) {
                double s = orc_half_to_double(scales[n * G + g]);
                double part = 0.0;
                for (int64_t k = 128 * g; k < 128 * g + 128; k++) {
                    double xv = orc_bf16_to_double(x[b * K + k]);
                    if (orc_bit(bits, K, n, k))
                        part += xv;
                    else
                        part -= xv;
                }
                acc += s * part;
            }
            y[b * N + n] = acc;
        }
    }
}

int orc_gemv(const uint8_t *bits, const uint16_t *scales, const uint16_t *x,
             int64_t B, int64_t N, int64_t K, double *y)
{
    int st = orc_check_shape(B, N, K);
    if (st != ORC_OK)
        return st;
    if (!bits || !scales || !x || !y)
        return ORC_EINVAL;
    orc_gemv_rows(bits, scales, x, B, N, K, 0, N, y);
    return ORC_OK;
}

/* Selected rows only: y[b * n_sel + i] = row rows[i] of the product.  Used to
 * check full-size problems on sampled outputs. */
int orc_gemv_select(const uint8_t *bits, const uint16_t *scales,
                    const uint16_t *x, int64_t B, int64_t N, int64_t K,
                    const int64_t *rows, int64_t n_sel, double *y)
{
    int st = orc_check_shape(B, N, K);
    double *tmp;
    if (st != ORC_OK)
        return st;
    if (!bits || !scales || !x || !y || (n_sel > 0 && !rows))
        return ORC_EINVAL;
    for (int64_t i = 0; i < n_sel; i++)
        if (rows[i] < 0 || rows[i] >= N)
            return ORC_ERANGE;
    tmp = (double *)malloc(sizeof(double) * (size_t)B * (size_t)N);
    if (!tmp)
        return ORC_EINVAL;
    for (int64_t i = 0; i < n_sel; i++) {
        int64_t n = rows[i];
        orc_gemv_rows(bits, scales, x, B, N, K, n, n + 1, tmp);
        for (int64_t b = 0; b < B; b++)
            y[b * n_sel + i] = tmp[b * N + n];
    }
    free(tmp);
    return ORC_OK;
}

/* ---- gate/up pair with the SwiGLU activation ------------------------------
 * [27B-arch]: the MLP is SwiGLU, h = silu(gate x) * (up x), fed to the down
 * projection.  Reading of the layout, which the pages do not give: the gate
 * and up matrices are stored as one matrix with interleaved rows, row 2n the
 * gate and row 2n+1 the up projection of output n.  h[b,n] = silu(g) * u with
 * the textbook silu(g) = g / (1 + exp(-g)), in fp64 on the exact GEMV
 * results.  N2 (the interleaved row count) must be even. */
int orc_gemv_swiglu(const uint8_t *bits, const uint16_t *scales, const uint16_t *x,
                    int64_t B, int64_t N2, int64_t K, double *h)
{
    int st = orc_check_shape(B, N2, K);
    double *y;
    if (st != ORC_OK)
        return st;
    if (N2 % 2 != 0)
        return ORC_ESHAPE;
    if (!bits || !scales || !x || !h)
        return ORC_EINVAL;
    y = (double *)malloc(sizeof(double) * (size_t)B * (size_t)N2);
    if (!y)
        return ORC_EINVAL;
    orc_gemv_rows(bits, scales, x, B, N2, K, 0, N2, y);
    for (int64_t b = 0; b < B; b++) {
        for (int64_t n = 0; n < N2 / 2; n++) {
            double g = y[b * N2 + 2 * n], u = y[b * N2 + 2 * n + 1];
            h[b * (N2 / 2) + n] = g / (1.0 + exp(-g)) * u;
        }
    }
    free(y);
    return ORC_OK;
}

/* Selected hidden units only: h[b * n_sel + i] = h[b, units[i]] of the
 * interleaved pair above, from rows 2 units[i] and 2 units[i] + 1 alone.
 * Used to check full-size problems on sampled outputs. */
int orc_gemv_swiglu_select(const uint8_t *bits, const uint16_t *scales, const uint16_t *x,
                           int64_t B, int64_t N2, int64_t K, const int64_t *units,
                           int64_t n_sel, double *h)
{
    int st = orc_check_shape(B, N2, K);
    double *y;
    if (st != ORC_OK)
        return st;
    if (N2 % 2 != 0)
        return ORC_ESHAPE;
    if (!bits || !scales || !x || !h || (n_sel > 0 && !units))
        return ORC_EINVAL;
    for (int64_t i = 0; i < n_sel; i++)
        if (units[i] < 0 || units[i] >= N2 / 2)
            return ORC_ERANGE;
    y = (double *)malloc(sizeof(double) * (size_t)B * (size_t)N2);
    if (!y)
        return ORC_EINVAL;
    for (int64_t i = 0; i < n_sel; i++) {
        int64_t n = units[i];
        orc_gemv_rows(bits, scales, x, B, N2, K, 2 * n, 2 * n + 2, y);
        for (int64_t b = 0; b < B; b++) {
            double g = y[b * N2 + 2 * n], u = y[b * N2 + 2 * n + 1];
            h[b * n_sel + i] = g / (1.0 + exp(-g)) * u;
        }
    }
    free(y);
    return ORC_OK;
}

/* ---- ternary linear layer ------------------------------------------------
 * y[b,n] = sum_g s[n,g] * sum_{k in group g} t(n,k) * x[b,k] ([27B-ter]);
 * t read from the two planes one weight at a time; fp64 accumulation, the
 * group partial first, then one multiply by the scale.  Rows [n0, n1). */
static int orc_trit(const uint8_t *pa, const uint8_t *pb, int64_t K, int64_t n, int64_t k)
{
    int va = orc_bit(pa, K, n, k) ? 1 : -1;
    int vb = orc_bit(pb, K, n, k) ? 1 : -1;
    return (va + vb) / 2;
}

static void orc_gemv_ternary_rows(const uint8_t *pa, const uint8_t *pb, const uint16_t *scales,
                                  const uint16_t *x, int64_t B, int64_t N, int64_t K,
                                  int64_t n0, int64_t n1, double *y)
{
    int64_t G = K / 128;
    for (int64_t b = 0; b < B; b++) {
        for (int64_t n = n0; n < n1; n++) {
            double acc = 0.0;
            for (int64_t g = 0; g < G; g++) {
                double s = orc_half_to_double(scales[n * G + g]);
                double part = 0.0;
                for (int64_t k = 128 * g; k < 128 * g + 128; k++) {
                    int t = orc_trit(pa, pb, K, n, k);
                    double xv = orc_bf16_to_double(x[b * K + k]);
                    if (t > 0)
                        part += xv;
                    else if (t < 0)
                        part -= xv;
                }
                acc += s * part;
            }
            y[b * N + n] = acc;
        }
    }
}

int orc_gemv_ternary(const uint8_t *pa, const uint8_t *pb, const uint16_t *scales,
                     const uint16_t *x, int64_t B, int64_t N, int64_t K, double *y)
{
    int st = orc_check_shape(B, N, K);
    if (st != ORC_OK)
        return st;
    if (!pa || !pb || !scales || !x || !y)
        return ORC_EINVAL;
    orc_gemv_ternary_rows(pa, pb, scales, x, B, N, K, 0, N, y);
    return ORC_OK;
}

/* Ternary gate/up pair with the SwiGLU activation ([27B-ter], [27B-arch]):
 * the interleaved layout of orc_gemv_swiglu on ternary rows. */
int orc_gemv_ternary_swiglu(const uint8_t *pa, const uint8_t *pb, const uint16_t *scales,
                            const uint16_t *x, int64_t B, int64_t N2, int64_t K, double *h)
{
    int st = orc_check_shape(B, N2, K);
    double *y;
    if (st != ORC_OK)
        return st;
    if (N2 % 2 != 0)
        return ORC_ESHAPE;
    if (!pa || !pb || !scales || !x || !h)
        return ORC_EINVAL;
    y = (double *)malloc(sizeof(double) * (size_t)B * (size_t)N2);
    if (!y)
        return ORC_EINVAL;
    orc_gemv_ternary_rows(pa, pb, scales, x, B, N2, K, 0, N2, y);
    for (int64_t b = 0; b < B; b++) {
        for (int64_t n = 0; n < N2 / 2; n++) {
            double gt = y[b * N2 + 2 * n], up = y[b * N2 + 2 * n + 1];
            h[b * (N2 / 2) + n] = gt / (1.0 + exp(-gt)) * up;
        }
    }
    free(y);
    return ORC_OK;
}

int orc_gemv_ternary_select(const uint8_t *pa, const uint8_t *pb, const uint16_t *scales,
                            const uint16_t *x, int64_t B, int64_t N, int64_t K,
                            const int64_t *rows, int64_t n_sel, double *y)
{
    int st = orc_check_shape(B, N, K);
    double *tmp;
    if (st != ORC_OK)
        return st;
    if (!pa || !pb || !scales || !x || !y || (n_sel > 0 && !rows))
        return ORC_EINVAL;
    for (int64_t i = 0; i < n_sel; i++)
        if (rows[i] < 0 || rows[i] >= N)
            return ORC_ERANGE;
    tmp = (double *)malloc(sizeof(double) * (size_t)B * (size_t)N);
    if (!tmp)
        return ORC_EINVAL;
    for (int64_t i = 0; i < n_sel; i++) {
        int64_t n = rows[i];
        orc_gemv_ternary_rows(pa, pb, scales, x, B, N, K, n, n + 1, tmp);
        for (int64_t b = 0; b < B; b++)
            y[b * n_sel + i] = tmp[b * N + n];
    }
    free(tmp);
    return ORC_OK;
}

/* Ternary codes [N][K] (int8, each -1, 0 or +1) to the two planes, one
 * weight at a time; ERANGE (planes untouched) if any code is another value. */
int orc_ternary_planes(const int8_t *t, int64_t N, int64_t K, uint8_t *pa, uint8_t *pb)
{
    int st = orc_check_shape(1, N, K);
    if (st != ORC_OK)
        return st;
    if (!t || !pa || !pb)
        return ORC_EINVAL;
    for (int64_t i = 0; i < N * K; i++)
        if (t[i] < -1 || t[i] > 1)
            return ORC_ERANGE;
    memset(pa, 0, (size_t)(N * K / 8));
    memset(pb, 0, (size_t)(N * K / 8));
    for (int64_t n = 0; n < N; n++) {
        for (int64_t k = 0; k < K; k++) {
            int8_t v = t[n * K + k];
            if (v >= 0)
                pa[n * (K / 8) + k / 8] |= (uint8_t)(1u << (k % 8));
            if (v > 0)
                pb[n * (K / 8) + k / 8] |= (uint8_t)(1u << (k % 8));
        }
    }
    return ORC_OK;
}

/* Bytes of a ternary matrix in 2-bit slots: two sign planes plus the scales. */
int64_t orc_ternary_footprint_bytes(int64_t N, int64_t K)
{
    return 2 * (N * K / 8) + 2 * N * (K / 128);
}

/* ---- ternary, five codes per byte ----------------------------------------
 * The native packing closer to log2(3) bits ([27B-ter]; [27B-store] says the
 * deployed 2-bit slots exceed the information-theoretic minimum until native
 * ternary kernels exist).  Reading (the pages give no layout): each group of
 * 128 codes of a row is 26 bytes; byte j < 25 holds codes 5j .. 5j+4 and byte
 * 25 holds codes 125 .. 127, each byte the base-3 number
 *     v = sum_i (t_i + 1) * 3^i   (i = 0 for the lowest k),
 * so a 5-code byte is 0 .. 242 and the last byte 0 .. 26.  Row n, group g
 * starts at byte (n * (K/128) + g) * 26.  With the scales: 1.75 bits/weight. */
static int orc_t5_digits(int64_t j)
{
    return j < 25 ? 5 : 3;
}

int orc_t5_pack(const int8_t *t, int64_t N, int64_t K, uint8_t *out)
{
    int st = orc_check_shape(1, N, K);
    int64_t G = K / 128;
    if (st != ORC_OK)
        return st;
    if (!t || !out)
        return ORC_EINVAL;
    for (int64_t i = 0; i < N * K; i++)
        if (t[i] < -1 || t[i] > 1)
            return ORC_ERANGE;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t g = 0; g < G; g++) {
            uint8_t *grp = out + (n * G + g) * 26;
            int64_t k = 128 * g;
            for (int64_t j = 0; j < 26; j++) {
                int v = 0, p = 1;
                for (int i = 0; i < orc_t5_digits(j); i++) {
                    v += (t[n * K + k] + 1) * p;
                    p *= 3;
                    k++;
                }
                grp[j] = (uint8_t)v;
            }
        }
    }
    return ORC_OK;
}

/* Code t(n, k) of a packed matrix, or 2 if its byte is out of range. */
static int orc_t5_code(const uint8_t *p, int64_t K, int64_t n, int64_t k)
{
    int64_t G = K / 128, g = k / 128, r = k % 128;
    int64_t j = r / 5;
    int i = (int)(r % 5), v = p[(n * G + g) * 26 + j];
    if (v > (j < 25 ? 242 : 26))
        return 2;
    while (i-- > 0)
        v /= 3;
    return v % 3 - 1;
}

int orc_t5_unpack(const uint8_t *p, int64_t N, int64_t K, int8_t *t)
{
    int st = orc_check_shape(1, N, K);
    if (st != ORC_OK)
        return st;
    if (!p || !t)
        return ORC_EINVAL;
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) {
            int c = orc_t5_code(p, K, n, k);
            if (c == 2)
                return ORC_ERANGE;
            t[n * K + k] = (int8_t)c;
        }
    return ORC_OK;
}

/* y[b,n] = sum_g s[n,g] * sum_{k in g} t(n,k) x[b,k], codes read one at a
 * time from the packed bytes; fp64, group partial first.  ERANGE (y
 * untouched) if any byte is out of range. */
int orc_gemv_t5(const uint8_t *p, const uint16_t *scales, const uint16_t *x,
                int64_t B, int64_t N, int64_t K, double *y)
{
    int st = orc_check_shape(B, N, K);
    int64_t G = K / 128;
    if (st != ORC_OK)
        return st;
    if (!p || !scales || !x || !y)
        return ORC_EINVAL;
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++)
            if (orc_t5_code(p, K, n, k) == 2)
                return ORC_ERANGE;
    for (int64_t b = 0; b < B; b++) {
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0;
            for (int64_t g = 0; g < G; g++) {
                double s = orc_half_to_double(scales[n * G + g]);
                double part = 0.0;
                for (int64_t k = 128 * g; k < 128 * g + 128; k++) {
                    int c = orc_t5_code(p, K, n, k);
                    double xv = orc_bf16_to_double(x[b * K + k]);
                    if (c > 0)
                        part += xv;
                    else if (c < 0)
                        part -= xv;
                }
                acc += s * part;
            }
            y[b * N + n] = acc;
        }
    }
    return ORC_OK;
}

/* Bytes of a matrix packed five codes per byte: 26 per group plus the scale. */
int64_t orc_t5_footprint_bytes(int64_t N, int64_t K)
{
    return N * (K / 128) * 26 + 2 * N * (K / 128);
}

/* Same function, rows split over `nthreads` POSIX threads: parallel dispatch
 * of the scalar loop above, nothing else (used only to time the oracle on
 * all host cores). */
struct orc_job {
    const uint8_t *bits;
    const uint16_t *scales;
    const uint16_t *x;
    int64_t B, N, K, n0, n1;
    double *y;
};

static void *orc_job_run(void *p)
{
    struct orc_job *j = (struct orc_job *)p;
    orc_gemv_rows(j->bits, j->scales, j->x, j->B, j->N, j->K, j->n0, j->n1, j->y);
    return NULL;
}

int orc_gemv_threads(const uint8_t *bits, const uint16_t *scales,
                     const uint16_t *x, int64_t B, int64_t N, int64_t K,
                     double *y, int nthreads)
{
    int st = orc_check_shape(B, N, K);
    pthread_t *th;
    struct orc_job *jobs;
    if (st != ORC_OK)
        return st;
    if (!bits || !scales || !x || !y)
        return ORC_EINVAL;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > N)
        nthreads = (int)N;
    th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    jobs = (struct orc_job *)calloc((size_t)nthreads, sizeof(struct orc_job));
    if (!th || !jobs) {
        free(th);
        free(jobs);
        return ORC_EINVAL;
    }
    for (int t = 0; t < nthreads; t++) {
        jobs[t].bits = bits;
        jobs[t].scales = scales;
        jobs[t].x = x;
        jobs[t].B = B;
        jobs[t].N = N;
        jobs[t].K = K;
        jobs[t].n0 = N * t / nthreads;
        jobs[t].n1 = N * (t + 1) / nthreads;
        jobs[t].y = y;
        pthread_create(&th[t], NULL, orc_job_run, &jobs[t]);
    }
    for (int t = 0; t < nthreads; t++)
        pthread_join(th[t], NULL);
    free(th);
    free(jobs);
    return ORC_OK;
}

/* ---- the Bankai XOR patch ---------------------------------------------
 * [Bankai]: each listed row has all of its binary weights flipped; applying
 * the same list again removes the patch.  All rows are checked first; if any
 * is outside [0, N) nothing is modified and ERANGE is returned.  Then, one
 * entry at a time and one byte at a time, bits[row][j] ^= 0xFF. */
int orc_xor_patch(uint8_t *bits, int64_t N, int64_t K, const int32_t *rows,
                  int64_t n_rows)
{
    int st = orc_check_shape(1, N, K);
    if (st != ORC_OK)
        return st;
    if (n_rows < 0 || (n_rows > 0 && (!bits || !rows)))
        return ORC_EINVAL;
    for (int64_t i = 0; i < n_rows; i++)
        if (rows[i] < 0 || (int64_t)rows[i] >= N)
            return ORC_ERANGE;
    for (int64_t i = 0; i < n_rows; i++) {
        int64_t r = rows[i];
        for (int64_t j = 0; j < K / 8; j++)
            bits[r * (K / 8) + j] ^= 0xFF;
    }
    return ORC_OK;
}

/* ---- the g128x storage layout -------------------------------------------
 * Not from the pages (they fix no bit layout beyond "packed 1-bit"): a
 * storage format of the library under test, a permutation of the 128 sign
 * bits of every group, written here from its stated definition so that the
 * library's conversion can be checked bit for bit.  Group bit b is bit b % 8
 * of byte b / 8 of the group's 16 bytes.  For input k of the group:
 *   inputs 0..71, six per field f = k / 6: byte f (of bytes 0..11), bit
 *   1 + k % 6 (bits 1..6 of the byte, in input order);
 *   inputs 72..95, six per field j = (k - 72) / 6 with i = (k - 72) % 6:
 *   in the bytes of 32-bit word i / 2 (bytes 4 (i / 2) .. 4 (i / 2) + 3),
 *   bit 7 of its byte j when i is even, bit 0 of its byte (j + 1) mod 4
 *   when i is odd;
 *   inputs 96..127: bit k (unchanged).
 * One byte and one bit at a time. */
static int orc_g128x_bit(int k)
{
    if (k < 72)
        return (k / 6) * 8 + 1 + k % 6;
    if (k < 96) {
        int j = (k - 72) / 6, i = (k - 72) % 6;
        int word = i / 2;
        if (i % 2 == 0)
            return word * 32 + j * 8 + 7;
        return word * 32 + ((j + 1) % 4) * 8 + 0;
    }
    return k;
}

static int orc_g128x_convert(const uint8_t *in, int64_t N, int64_t K, uint8_t *out, int to_g128x)
{
    int st = orc_check_shape(1, N, K);
    if (st != ORC_OK)
        return st;
    if (!in || !out)
        return ORC_EINVAL;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t g = 0; g < K / 128; g++) {
            const uint8_t *src = in + n * (K / 8) + 16 * g;
            uint8_t grp[16] = {0};
            for (int k = 0; k < 128; k++) {
                int from = to_g128x ? k : orc_g128x_bit(k);
                int to = to_g128x ? orc_g128x_bit(k) : k;
                if ((src[from / 8] >> (from % 8)) & 1)
                    grp[to / 8] |= (uint8_t)(1u << (to % 8));
            }
            memcpy(out + n * (K / 8) + 16 * g, grp, 16);
        }
    }
    return ORC_OK;
}

int orc_g128x_repack(const uint8_t *in, int64_t N, int64_t K, uint8_t *out)
{
    return orc_g128x_convert(in, N, K, out, 1);
}

int orc_g128x_unpack(const uint8_t *in, int64_t N, int64_t K, uint8_t *out)
{
    return orc_g128x_convert(in, N, K, out, 0);
}

/* ---- packing ----------------------------------------------------------
 * Floating-point weights [N][K] (fp32, bf16 or fp16 bit patterns) -> sign
 * bits and fp16 group scales, by the readings listed at the top. */
int orc_pack(const void *w, int dtype, int64_t N, int64_t K, uint8_t *bits,
             uint16_t *scales)
{
    int st = orc_check_shape(1, N, K);
    int nan_seen = 0, range_bad = 0;
    int64_t G = K / 128;
    if (st != ORC_OK)
        return st;
    if (!w || !bits || !scales)
        return ORC_EINVAL;
    if (dtype != ORC_F32 && dtype != ORC_BF16 && dtype != ORC_F16)
        return ORC_EINVAL;
    memset(bits, 0, (size_t)(N * K / 8));
    for (int64_t n = 0; n < N; n++) {
        for (int64_t g = 0; g < G; g++) {
            double sum = 0.0, mean;
            uint16_t h;
            for (int64_t k = 128 * g; k < 128 * g + 128; k++) {
                int64_t idx = n * K + k;
                double v;
                if (dtype == ORC_F32)
                    v = orc_f32_to_double((const uint8_t *)w + 4 * idx);
                else if (dtype == ORC_BF16)
                    v = orc_bf16_to_double(((const uint16_t *)w)[idx]);
                else
                    v = orc_half_to_double(((const uint16_t *)w)[idx]);
                if (isnan(v))
                    nan_seen = 1;
                if (!(v < 0.0))
                    bits[n * (K / 8) + k / 8] |= (uint8_t)(1u << (k % 8));
                sum += fabs(v);
            }
            mean = sum / 128.0;
            h = orc_double_to_half(mean);
            if ((h & 0x7c00) == 0x7c00)
                range_bad = 1;
            scales[n * G + g] = h;
        }
    }
    if (nan_seen)
        return ORC_ENAN;
    if (range_bad)
        return ORC_ERANGE;
    return ORC_OK;
}
