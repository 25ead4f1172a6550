/*
 * mpq_oracle.c -- plain, slow, single-threaded CPU oracle for fine-grained FP8
 * quantization and block-scaled FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the reference the CUDA path is checked
 * against.  Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark may load it.  It shares no code, header, table or constant with the
 * CUDA library and includes nothing from it.
 *
 * What it follows (the source pages are scraped copies of the FP8 mixed-precision
 * training description of an MoE LLM technical report):
 *   - page 1 (xn--9g3bo1gtkw0l8ubf92bgle.kr, qna board post 131281), second
 *     paragraph: the scaling factor is derived from the online
 *     maximum absolute value and the activation or weight is quantized online into
 *     FP8; FP8 GEMMs take FP8 inputs and produce BF16 or FP32 outputs.
 *   - page 3 (blog.cameseeing.com freeboard 1171527), first paragraph: the input
 *     is aligned to the FP8 range by scaling its maximum absolute value to the
 *     largest representable FP8 value.
 *   - page 2 (xn--jj0bz6z98ct0a29q.com board 62 368261), last paragraph: groups of
 *     128 activation values; backward re-quantization into 128x1 tiles.
 *   - page 4 (why-be.co.kr as_center 59061), first paragraph: partial sums are
 *     promoted to FP32 every 128 elements of K and accumulated in full FP32;
 *     second paragraph: integral power-of-2 scaling factors.
 *   - The E4M3 format itself (bias 7, no infinities, S.1111.111 = NaN, largest
 *     finite 448) is the OCP 8-bit floating point specification; the group shapes
 *     1x128 (activations) and 128x128 (weights) and "scale = amax / 448" read the
 *     subscripts the scraped pages lost (their text keeps only "128 elements" and
 *     "128x1 tiles").
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - rounding of the cast is round-to-nearest-even, overflow saturates to +-448;
 *   - the quotient x / s is one correctly rounded IEEE binary32 division, then the
 *     E4M3 rounding (double rounding is the contract);
 *   - an all-zero group gets scale 1.0;
 *   - power-of-2 scales round up: s = 2^e with e the smallest integer such that
 *     amax <= 448 * 2^e, so no element saturates;
 *   - zero keeps its sign (-0 -> 0x80), NaN inputs are out of contract;
 *   - a positive scale never drops below 2^-149 (see mpqo_group_scale);
 *   - re-quantization dequantizes with one binary32 product dec(q) * s.
 *
 * Build: gcc -O2 -fPIC -shared -ffp-contract=off (no -ffast-math: IEEE division,
 * subnormals kept).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

/* ---------------------------------------------------------------- E4M3 codec */

/* OCP E4M3: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.
 * exponent 0 -> subnormal m * 2^-9; exponent 15 with mantissa 7 -> NaN. */
double mpqo_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = (double)m * ldexp(1.0, -9);
    else
        v = (1.0 + (double)m / 8.0) * ldexp(1.0, e - 7);
    return s ? -v : v;
}

/* Non-negative finite values, code 0x00 .. 0x7E, ascending. */
static double g_pos[127];
static int g_pos_ready = 0;

static void init_pos(void)
{
    if (g_pos_ready)
        return;
    for (int c = 0; c <= 0x7E; ++c)
        g_pos[c] = mpqo_e4m3_decode((uint8_t)c);
    g_pos_ready = 1;
}

/* Round a binary32 value to the nearest E4M3 value, ties to the even code,
 * saturating at +-448.  Works on magnitudes against the decoded value table. */
uint8_t mpqo_e4m3_encode(float v)
{
    init_pos();
    if (isnan(v))
        return 0x7F; /* out of contract */
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0)
        return sign | 0x7E;
    /* largest code c with g_pos[c] <= a (binary search, table ascending) */
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (g_pos[mid] <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    int c = lo;
    if (g_pos[c] == a)
        return sign | (uint8_t)c;
    /* a < 448 so c + 1 <= 0x7E exists */
    double dlo = a - g_pos[c];
    double dhi = g_pos[c + 1] - a;
    if (dlo < dhi)
        return sign | (uint8_t)c;
    if (dhi < dlo)
        return sign | (uint8_t)(c + 1);
    return sign | (uint8_t)((c & 1) ? c + 1 : c); /* tie: even mantissa */
}

/* ------------------------------------------------------------- group scales */

static float bf16_to_float(uint16_t b)
{
    union { uint32_t u; float f; } x;
    x.u = (uint32_t)b << 16;
    return x.f;
}

/* Scale of one quantization group from its maximum absolute value.
 * Floor: a scale that would be 0 (amax/448 below half the smallest subnormal) or a power
 * of 2 below 2^-149 (not a binary32 number) becomes 2^-149, the smallest positive
 * binary32.  BF16 groups never reach it (their amax is at least 2^-133); groups of
 * dequantized FP8 values can. */
float mpqo_group_scale(float amax, int pow2)
{
    if (amax == 0.0f)
        return 1.0f;
    if (!pow2) {
        float s = amax / 448.0f; /* one IEEE binary32 division */
        return s > 0.0f ? s : ldexpf(1.0f, -149);
    }
    int e = -149;
    while ((double)amax > ldexp(448.0, e))
        ++e;
    return ldexpf(1.0f, e); /* 2^e */
}

static uint8_t quant_one(float x, float s)
{
    float y = x / s; /* correctly rounded binary32 quotient */
    return mpqo_e4m3_encode(y);
}

/* ------------------------------------------------------------- quantizers */

/* Row-wise 1x128 groups: group (r, kb) = x[r, kb*128 .. kb*128+127].
 * q[r, c] row-major (ldq), s[kb * lds + r] (K-block-major scales). */
void mpqo_quant_tile_1x128(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx,
                           uint8_t *q, int64_t ldq, float *s, int64_t lds, int pow2)
{
    int64_t nkb = cols / 128;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t kb = 0; kb < nkb; ++kb) {
            const uint16_t *g = x + r * ldx + kb * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float a = fabsf(bf16_to_float(g[i]));
                if (a > amax)
                    amax = a;
            }
            float sc = mpqo_group_scale(amax, pow2);
            s[kb * lds + r] = sc;
            for (int i = 0; i < 128; ++i)
                q[r * ldq + kb * 128 + i] = quant_one(bf16_to_float(g[i]), sc);
        }
    }
}

/* Column-wise 128x1 groups (along rows, i.e. along tokens): group (rb, c) =
 * x[rb*128 .. rb*128+127, c].  Output is stored transposed so that the group is
 * contiguous: qT[c, rb*128 + i] (ldqT), sT[rb * ldsT + c]. */
void mpqo_quant_tile_128x1(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx,
                           uint8_t *qT, int64_t ldqT, float *sT, int64_t ldsT, int pow2)
{
    int64_t nrb = rows / 128;
    for (int64_t c = 0; c < cols; ++c) {
        for (int64_t rb = 0; rb < nrb; ++rb) {
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float a = fabsf(bf16_to_float(x[(rb * 128 + i) * ldx + c]));
                if (a > amax)
                    amax = a;
            }
            float sc = mpqo_group_scale(amax, pow2);
            sT[rb * ldsT + c] = sc;
            for (int i = 0; i < 128; ++i)
                qT[c * ldqT + rb * 128 + i] =
                    quant_one(bf16_to_float(x[(rb * 128 + i) * ldx + c]), sc);
        }
    }
}

/* Re-quantization of cached FP8 codes into 128x1 groups.  Page 2 ("9 Amazing Deepseek
 * Hacks"), last paragraph: in the backward pass the FP8 matrix is read out, dequantized,
 * transposed and quantized again into 128x1 tiles; page 1, second paragraph: activations
 * are cached in FP8 for the backward pass of the Linear operator.
 * Input: the row-wise 1x128 quantization of a [rows, cols] matrix, codes q[t, c] (ldq) and
 * scales s[(c/128) * lds + t].  Each element is dequantized to binary32,
 * xhat = dec(q) * s (one IEEE binary32 product), and the 128x1 groups of xhat along t are
 * quantized as mpqo_quant_tile_128x1 quantizes BF16 values.  Output stored transposed:
 * qT[c, t] (ldqT), sT[(t/128) * ldsT + c]. */
void mpqo_requant_tile_128x1(const uint8_t *q, int64_t rows, int64_t cols, int64_t ldq,
                             const float *s, int64_t lds, uint8_t *qT, int64_t ldqT,
                             float *sT, int64_t ldsT, int pow2)
{
    int64_t nrb = rows / 128;
    for (int64_t c = 0; c < cols; ++c) {
        for (int64_t rb = 0; rb < nrb; ++rb) {
            float xh[128];
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                int64_t t = rb * 128 + i;
                float d = (float)mpqo_e4m3_decode(q[t * ldq + c]); /* exact */
                xh[i] = d * s[(c / 128) * lds + t];
                float a = fabsf(xh[i]);
                if (a > amax)
                    amax = a;
            }
            float sc = mpqo_group_scale(amax, pow2);
            sT[rb * ldsT + c] = sc;
            for (int i = 0; i < 128; ++i)
                qT[c * ldqT + rb * 128 + i] = quant_one(xh[i], sc);
        }
    }
}

/* ------------------------------------------- SwiGLU feeding the down projection */

/* exp(x) in binary32 by Cody and Waite's argument reduction (W. J. Cody, W. Waite,
 * "Software Manual for the Elementary Functions", 1980): n = rint(x log2 e),
 * r = x - n ln2 with ln2 split into a 15-bit head (n * head is exact) and a tail, then the
 * degree-7 Taylor polynomial of e^r (|r| <= ln2/2, truncation error below 2^-27) in Horner
 * form with fused multiply-adds, scaled by 2^n.  This exact sequence of binary32 operations
 * is the definition the GPU path follows; its accuracy against the true exponential is
 * pinned by the tests (within 2 ulp).  x is clamped to [-104, 89]: below, e^x rounds to 0;
 * above, it overflows to infinity, as it does after the clamp. */
float mpqo_exp_f32(float x)
{
    const float l2e = 0x1.715476p+0f, ln2_hi = 0x1.62e4p-1f, ln2_lo = 0x1.7f7d1cp-20f;
    if (x < -104.0f)
        x = -104.0f;
    if (x > 89.0f)
        x = 89.0f;
    const float nf = nearbyintf(x * l2e); /* ties to even */
    const int n = (int)nf;
    float r = fmaf(-nf, ln2_hi, x);
    r = fmaf(-nf, ln2_lo, r);
    float p = 0x1.a01a02p-13f;            /* 1/7! */
    p = fmaf(p, r, 0x1.6c16c2p-10f);      /* 1/6! */
    p = fmaf(p, r, 0x1.111112p-7f);       /* 1/5! */
    p = fmaf(p, r, 0x1.555556p-5f);       /* 1/4! */
    p = fmaf(p, r, 0x1.555556p-3f);       /* 1/3! */
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    /* p * 2^n, with one rounding: the first factor below is exact */
    if (n > 127)
        return (p * 0x1p64f) * ldexpf(1.0f, n - 64);
    if (n < -126)
        return (p * ldexpf(1.0f, n + 64)) * 0x1p-64f;
    return p * ldexpf(1.0f, n);
}

/* silu(g) = g / (1 + e^-g): one binary32 addition and one IEEE division. */
float mpqo_silu_f32(float g)
{
    const float den = 1.0f + mpqo_exp_f32(-g);
    return g / den;
}

/* SwiGLU of the up-projection output and its 1x128 quantization, the input of the down
 * projection.  Page 1, first paragraph: the SwiGLU operator's inputs are cached and its
 * output recomputed in the backward pass; page 4, second paragraph: the activation before
 * the MoE down projection uses integral power-of-2 scales.
 * hcat[r, 0 .. W) is the gate, hcat[r, W .. 2W) the up value (BF16 bits, ldh >= 2W);
 * x[r, c] = silu(gate[r, c]) * up[r, c] (binary32, one rounded product); its 1x128 groups
 * are quantized like mpqo_quant_tile_1x128's: q[r, c] (ldq), s[(c/128) * lds + r]. */
void mpqo_swiglu_quant_1x128(const uint16_t *hcat, int64_t rows, int64_t width, int64_t ldh, uint8_t *q,
                             int64_t ldq, float *s, int64_t lds, int pow2)
{
    int64_t nkb = width / 128;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t kb = 0; kb < nkb; ++kb) {
            float x[128];
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                const int64_t c = kb * 128 + i;
                const float g = bf16_to_float(hcat[r * ldh + c]);
                const float u = bf16_to_float(hcat[r * ldh + width + c]);
                x[i] = mpqo_silu_f32(g) * u;
                float a = fabsf(x[i]);
                if (a > amax)
                    amax = a;
            }
            float sc = mpqo_group_scale(amax, pow2);
            s[kb * lds + r] = sc;
            for (int i = 0; i < 128; ++i)
                q[r * ldq + kb * 128 + i] = quant_one(x[i], sc);
        }
    }
}

/* 128x128 blocks: block (i, j) = w[i*128 .. +127, j*128 .. +127].
 * q[r, c] (ldq); optional transposed codes qT[c, r] (ldqT); s[i * lds + j]. */
void mpqo_quant_block_128x128(const uint16_t *w, int64_t rows, int64_t cols, int64_t ldw,
                              uint8_t *q, int64_t ldq, uint8_t *qT, int64_t ldqT,
                              float *s, int64_t lds, int pow2)
{
    for (int64_t i = 0; i < rows / 128; ++i) {
        for (int64_t j = 0; j < cols / 128; ++j) {
            float amax = 0.0f;
            for (int64_t r = i * 128; r < i * 128 + 128; ++r)
                for (int64_t c = j * 128; c < j * 128 + 128; ++c) {
                    float a = fabsf(bf16_to_float(w[r * ldw + c]));
                    if (a > amax)
                        amax = a;
                }
            float sc = mpqo_group_scale(amax, pow2);
            s[i * lds + j] = sc;
            for (int64_t r = i * 128; r < i * 128 + 128; ++r)
                for (int64_t c = j * 128; c < j * 128 + 128; ++c) {
                    uint8_t code = quant_one(bf16_to_float(w[r * ldw + c]), sc);
                    q[r * ldq + c] = code;
                    if (qT)
                        qT[c * ldqT + r] = code;
                }
        }
    }
}

/* ------------------------------------------------------------------- GEMM */

/* Operation codes; they select only where the B-side scale of (n, k) lives.
 *   FPROP (0): sB[(n/128) * ldsb + k/128]   (128x128 weight blocks, [N/128][K/128])
 *   DGRAD (1): sB[(k/128) * ldsb + n/128]   (same blocks seen through the
 *              transposed weight, [K/128][N/128])
 *   WGRAD (2): sB[(k/128) * ldsb + n]       (128x1 token tiles, [K/128][N])
 * The A-side scale of (m, k) is always sA[(k/128) * ldsa + m]. */
static double scale_b(int op, const float *sB, int64_t ldsb, int64_t n, int64_t k)
{
    if (op == 0)
        return (double)sB[(n / 128) * ldsb + k / 128];
    if (op == 1)
        return (double)sB[(k / 128) * ldsb + n / 128];
    return (double)sB[(k / 128) * ldsb + n];
}

/* All 256 decoded codes, filled once from mpqo_e4m3_decode (lookup for speed only). */
static double g_dec[256];
static int g_dec_ready = 0;

static void init_dec(void)
{
    if (g_dec_ready)
        return;
    for (int c = 0; c < 256; ++c)
        g_dec[c] = mpqo_e4m3_decode((uint8_t)c);
    g_dec_ready = 1;
}

/* One output element: sum over k of (dec(A[m,k]) sA) (dec(B[n,k]) sB), in FP64,
 * in k order, plus the sum of magnitudes of the terms (for the tolerance). */
static void dot_one(int op, int64_t K, const uint8_t *A, int64_t lda, const float *sA,
                    int64_t ldsa, const uint8_t *B, int64_t ldb, const float *sB,
                    int64_t ldsb, int64_t m, int64_t n, double *ref, double *absref)
{
    double acc = 0.0, aacc = 0.0;
    init_dec();
    for (int64_t k = 0; k < K; ++k) {
        double a = g_dec[A[m * lda + k]] * (double)sA[(k / 128) * ldsa + m];
        double b = g_dec[B[n * ldb + k]] * scale_b(op, sB, ldsb, n, k);
        acc += a * b;
        aacc += fabs(a * b);
    }
    *ref = acc;
    *absref = aacc;
}

/* C[m, n] = sum_k A[m, k] B[n, k] with both operands K-major, all elements. */
void mpqo_gemm_ref(int op, int64_t M, int64_t N, int64_t K,
                   const uint8_t *A, int64_t lda, const float *sA, int64_t ldsa,
                   const uint8_t *B, int64_t ldb, const float *sB, int64_t ldsb,
                   double *ref, double *absref, int64_t ldr)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            dot_one(op, K, A, lda, sA, ldsa, B, ldb, sB, ldsb, m, n,
                    &ref[m * ldr + n], &absref[m * ldr + n]);
}

/* The same at a list of (m, n) positions. */
void mpqo_gemm_ref_at(int op, int64_t K,
                      const uint8_t *A, int64_t lda, const float *sA, int64_t ldsa,
                      const uint8_t *B, int64_t ldb, const float *sB, int64_t ldsb,
                      const int64_t *ms, const int64_t *ns, int64_t count,
                      double *ref, double *absref)
{
    for (int64_t i = 0; i < count; ++i)
        dot_one(op, K, A, lda, sA, ldsa, B, ldb, sB, ldsb, ms[i], ns[i], &ref[i], &absref[i]);
}

/* Grouped (MoE experts): expert g owns rows [off[g], off[g+1]) of A and C and
 * its own weight B_g = B + g * N * ldb with block scales sB_g = sB + g * nb * ldsb
 * (nb = N / 128 rows of the [N/128][K/128] scale grid).  FPROP scaling. */
void mpqo_grouped_gemm_ref(int64_t G, const int64_t *off, int64_t N, int64_t K,
                           const uint8_t *A, int64_t lda, const float *sA, int64_t ldsa,
                           const uint8_t *B, int64_t ldb, const float *sB, int64_t ldsb,
                           double *ref, double *absref, int64_t ldr)
{
    for (int64_t g = 0; g < G; ++g) {
        int64_t m0 = off[g], m1 = off[g + 1];
        if (m1 <= m0)
            continue;
        mpqo_gemm_ref(0, m1 - m0, N, K, A + m0 * lda, lda, sA + m0, ldsa,
                      B + g * N * ldb, ldb, sB + g * (N / 128) * ldsb, ldsb,
                      ref + m0 * ldr, absref + m0 * ldr, ldr);
    }
}
