/*
 * KroQuant MXFP4 activation quantizer -- CPU reference ("oracle").
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * Source of every step: "KroQuant: Kronecker-Structured Block Transforms for
 * Efficient Post-Training Quantization of Diffusion Transformers"
 * (arXiv 2607.21446v1), cited below as [KQ] with the section / equation.
 *
 * Arithmetic is IEEE fp64 throughout.  bf16 activations and fp32 factor
 * entries convert to fp64 exactly.  Nothing here is blocked, fused or
 * reordered beyond what the definitions state: the Kronecker block is
 * expanded entry by entry (eq. 12), applied as a dense 32x32 row-vector
 * product (eq. 4, K1's A_tile @ K), and each 32-element block is then
 * quantized on its own (Sec. 3.1, MXFP4 per the OCP MX format named in
 * Sec. 4.1 "Data format").
 *
 * Readings taken where the pages are silent:
 *   - shared exponent e = floor(log2 amax) - 2 (2 = emax of E2M1), clamped to
 *     the E8M0 range [-127, 127]; amax == 0 gives e = -127;
 *   - e2m1 rounding is round-to-nearest, ties to the even code, with
 *     saturation to +-6; the sign of y is kept, also for a zero magnitude;
 *   - packing: byte k of a row holds code 2k in bits 0-3 and code 2k+1 in
 *     bits 4-7.
 *
 * Parity: every function here is pinned by tests that do not use it as
 * their own reference (closed forms, a brute-force twin, library routines).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define KQO_EXPORT __attribute__((visibility("default")))

/* --- input conversion ---------------------------------------------------- */

static double bf16_bits_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;     /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

KQO_EXPORT double kqo_bf16_to_f64(uint16_t h) { return bf16_bits_to_f64(h); }

/* IEEE 754 binary16: sign, 5-bit exponent with bias 15, 10-bit fraction;
 * exponent 0 holds zero and the subnormals f * 2^-24, exponent 31 Inf/NaN. */
static double f16_bits_to_f64(uint16_t h)
{
    int sign = h >> 15, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f / 2^10) * 2^(e - 15) */
    return sign ? -v : v;
}

KQO_EXPORT double kqo_f16_to_f64(uint16_t h) { return f16_bits_to_f64(h); }

/* Format of the 16-bit activations the transforms read: 0 = bf16, 1 = fp16.
 * Process-wide; the Python wrapper sets it around each call. */
static int g_input_f16 = 0;

KQO_EXPORT void kqo_set_input_format(int f16) { g_input_f16 = f16 != 0; }

static double in_to_f64(uint16_t h) { return g_input_f16 ? f16_bits_to_f64(h) : bf16_bits_to_f64(h); }

/* --- [KQ] Sec. 3.2, eq. (6): unit-|det| LU factor ----------------------------
 * lu = {a, b, c}; G = [[1,0],[c,1]] . [[a,b],[0,u22]] with
 *   u22 = -1/a  (det_sign = -1, the paper's form, eq. 6)
 *   u22 = +1/a  (det_sign = +1, the unit-determinant form of the workloads).
 * G is written row-major: G[0]=G00, G[1]=G01, G[2]=G10, G[3]=G11.
 */
KQO_EXPORT void kqo_lu_to_factor(const double lu[3], int det_sign, double G[4])
{
    double a = lu[0], b = lu[1], c = lu[2];
    double u22 = (det_sign < 0 ? -1.0 : 1.0) / a;
    /* L . U, entry by entry (the zero products of the triangular factors
     * are left out) */
    G[0] = a;              /* 1*a + 0*0   */
    G[1] = b;              /* 1*b + 0*u22 */
    G[2] = c * a;          /* c*a + 1*0   */
    G[3] = c * b + u22;    /* c*b + 1*u22 */
}

/* --- [KQ] Sec. 3.5.1, eq. (12): entry-wise Kronecker expansion ---------------
 * K[r][c] = prod_{k=1..5} G_k[ bit_{5-k}(r), bit_{5-k}(c) ]
 * G holds the five factors G_1..G_5 as [5][2][2] row-major; G_1 pairs with
 * bit 4 (the most significant bit) of the row and column index.
 */
KQO_EXPORT void kqo_expand_block(const double *G, double *K)
{
    for (int r = 0; r < 32; ++r)
        for (int c = 0; c < 32; ++c) {
            double p = 1.0;
            for (int k = 1; k <= 5; ++k) {
                int bit = 5 - k;
                int rb = (r >> bit) & 1, cb = (c >> bit) & 1;
                p *= G[(k - 1) * 4 + rb * 2 + cb];
            }
            K[r * 32 + c] = p;
        }
}

/* Closed-form normalised Walsh-Hadamard block ([KQ] Sec. 3.2, "Hadamard
 * initialization"): H32[r][c] = (-1)^popcount(r & c) / sqrt(32). */
KQO_EXPORT void kqo_hadamard_block(double *K)
{
    double s = 1.0 / sqrt(32.0);
    for (int r = 0; r < 32; ++r)
        for (int c = 0; c < 32; ++c)
            K[r * 32 + c] = (__builtin_popcount((unsigned)(r & c)) & 1) ? -s : s;
}

/* --- [KQ] eq. (4) with K1's orientation A_tile @ K (Sec. 3.5.1) --------------
 * y[i][32j + c] = sum_r a[i][32j + r] * K_j[r][c]
 * bound[i][32j + c] = sum_r |a[i][32j + r] * K_j[r][c]|   (error scale)
 * Kall holds nb dense blocks [nb][32][32].
 */
static void apply_dense_blocks(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                               const double *Kall, double *y, double *bound)
{
    int64_t nb = d / 32;
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < m; ++i) {
        double a[32];
        for (int64_t j = 0; j < nb; ++j) {
            const double *K = Kall + j * 1024;
            for (int r = 0; r < 32; ++r)
                a[r] = in_to_f64(A[i * lda + j * 32 + r]);
            for (int c = 0; c < 32; ++c) {
                double acc = 0.0, mag = 0.0;
                for (int r = 0; r < 32; ++r) {
                    double t = a[r] * K[r * 32 + c];
                    acc += t;
                    mag += fabs(t);
                }
                y[i * d + j * 32 + c] = acc;
                if (bound) bound[i * d + j * 32 + c] = mag;
            }
        }
    }
}

/* Any dense per-block matrices Kall [nb][32][32] (used for the weight side
 * W T^{-T} of eq. 1, whose blocks are K_j^{-T}). */
KQO_EXPORT void kqo_transform_dense(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                    const double *Kall, double *y, double *bound)
{
    apply_dense_blocks(A, m, d, lda, Kall, y, bound);
}

/* KroQuant transform: factors [nb][5][2][2] (fp64), one set per 32-block
 * (eq. 4: T = diag(K^(1), ..., K^(nb)), eq. 5: K = G1 (x) ... (x) G5).
 * Kscratch must hold nb*1024 doubles. */
KQO_EXPORT void kqo_transform_kron(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                   const double *factors, double *Kscratch,
                                   double *y, double *bound)
{
    int64_t nb = d / 32;
    for (int64_t j = 0; j < nb; ++j)
        kqo_expand_block(factors + j * 20, Kscratch + j * 1024);
    apply_dense_blocks(A, m, d, lda, Kscratch, y, bound);
}

/* Fixed block-Hadamard baseline ([KQ] Sec. 4.3, Table 2 "Hadamard (32x32)"). */
KQO_EXPORT void kqo_transform_hadamard(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                       double *Kscratch, double *y, double *bound)
{
    int64_t nb = d / 32;
    kqo_hadamard_block(Kscratch);
    for (int64_t j = 1; j < nb; ++j)
        memcpy(Kscratch + j * 1024, Kscratch, 1024 * sizeof(double));
    apply_dense_blocks(A, m, d, lda, Kscratch, y, bound);
}

/* Full-row Walsh-Hadamard baseline ([KQ] Sec. 4.4, Table 3 "FWHT"; d a
 * power of two): y = a . H_d / sqrt(d) with the Sylvester-order Hadamard
 * matrix H_d[r][c] = (-1)^popcount(r & c), computed by the fast transform --
 * log2(d) passes of butterflies (x, y) -> (x + y, x - y) over pairs h apart,
 * h = 1, 2, 4, ... (H_2n = [[H_n, H_n], [H_n, -H_n]]; H_d is symmetric, so
 * a . H_d = H_d . a) -- then one multiply by 1/sqrt(d).
 * bound = sum_r |a_r| / sqrt(d), the error scale of every output. */
KQO_EXPORT void kqo_transform_fwht(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                   double *y, double *bound)
{
    const double inv = 1.0 / sqrt((double)d);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < m; ++i) {
        double *v = y + i * d;
        double l1 = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            v[c] = in_to_f64(A[i * lda + c]);
            l1 += fabs(v[c]);
        }
        for (int64_t h = 1; h < d; h *= 2)
            for (int64_t base = 0; base < d; base += 2 * h)
                for (int64_t j = base; j < base + h; ++j) {
                    const double x = v[j], z = v[j + h];
                    v[j] = x + z;
                    v[j + h] = x - z;
                }
        for (int64_t c = 0; c < d; ++c) {
            v[c] *= inv;
            if (bound) bound[i * d + c] = l1 * inv;
        }
    }
}

/* Diagonal (per-channel scaling, SmoothQuant-style) baseline:
 * T = diag(s), y = a * s[c]  ([KQ] Sec. 4.4, the "Scale" kernel). */
KQO_EXPORT void kqo_transform_diag(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                   const double *s, double *y, double *bound)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < m; ++i)
        for (int64_t c = 0; c < d; ++c) {
            double t = in_to_f64(A[i * lda + c]) * s[c];
            y[i * d + c] = t;
            if (bound) bound[i * d + c] = fabs(t);
        }
}

/* Identity transform: the bare quantizer ("Q4", [KQ] Tables 3 and 4). */
KQO_EXPORT void kqo_transform_identity(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                       double *y, double *bound)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < m; ++i)
        for (int64_t c = 0; c < d; ++c) {
            double t = in_to_f64(A[i * lda + c]);
            y[i * d + c] = t;
            if (bound) bound[i * d + c] = fabs(t);
        }
}

/* --- MXFP4 block quantizer ([KQ] Sec. 3.1; OCP MX, Sec. 4.1) --------------- */

/* E8M0 shared exponent: e = floor(log2 amax) - 2, clamped to [-127, 127]. */
KQO_EXPORT int kqo_e8m0_exponent(double amax)
{
    if (!(amax > 0.0)) return -127;
    int ex;
    frexp(amax, &ex);               /* amax = f * 2^ex, f in [0.5, 1) */
    int e = (ex - 1) - 2;           /* floor(log2 amax) = ex - 1 */
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* e2m1 magnitude grid, code order: {0, .5, 1, 1.5, 2, 3, 4, 6}. */
KQO_EXPORT double kqo_e2m1_value(uint8_t code)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[code & 7];
    return (code & 8) ? -v : v;
}

/* e2m1 encode: round to nearest on the e2m1 grid, ties to the even code
 * (even mantissa bit), saturate at 6, keep the sign bit of v.
 * Between binades the grid spacing is 0.5 on [0,2), 1 on [2,4), 2 on [4,6];
 * rint() (round half to even) on the spacing gives the nearest grid point,
 * and an even multiple there is an even code. */
KQO_EXPORT uint8_t kqo_encode_e2m1(double v)
{
    uint8_t sign = signbit(v) ? 8 : 0;
    double a = fabs(v);
    double q;
    if (a > 6.0) {
        q = 6.0;
    } else {
        double step = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
        q = rint(a / step) * step;
    }
    uint8_t mag;
    int twice = (int)(q * 2.0);
    switch (twice) {
    case 0: mag = 0; break;    /* 0   */
    case 1: mag = 1; break;    /* 0.5 */
    case 2: mag = 2; break;    /* 1   */
    case 3: mag = 3; break;    /* 1.5 */
    case 4: mag = 4; break;    /* 2   */
    case 6: mag = 5; break;    /* 3   */
    case 8: mag = 6; break;    /* 4   */
    default: mag = 7; break;   /* 6   */
    }
    return (uint8_t)(sign | mag);
}

/* Scale-factor byte position.
 * layout 0: row-major [m][nb].
 * layout 1: the 128x4 tiled layout of block-scaled MMA operands -- tiles of
 *   128 rows x 4 block-columns, 512 bytes each, tiles ordered row-tile major;
 *   inside a tile, row i and block-column kb sit at
 *   (i % 32) * 16 + ((i % 128) / 32) * 4 + (kb % 4). */
KQO_EXPORT int64_t kqo_sf_offset(int64_t i, int64_t kb, int64_t nb, int layout)
{
    if (layout == 0) return i * nb + kb;
    int64_t ncb = (nb + 3) / 4;
    int64_t tile = (i / 128) * ncb + kb / 4;
    return tile * 512 + (i % 32) * 16 + ((i % 128) / 32) * 4 + (kb % 4);
}

KQO_EXPORT int64_t kqo_sf_bytes(int64_t m, int64_t nb, int layout)
{
    if (layout == 0) return m * nb;
    return ((m + 127) / 128) * ((nb + 3) / 4) * 512;
}

/* Scatter row-major scale bytes rm [m][nb] into `out` (kqo_sf_bytes(m, nb,
 * layout) bytes) at the positions of the given layout; positions that hold
 * no scale (the padding of the tiled layout) get `fill`. */
KQO_EXPORT void kqo_sf_place(const uint8_t *rm, int64_t m, int64_t nb, int layout, uint8_t fill,
                             uint8_t *out)
{
    memset(out, fill, (size_t)kqo_sf_bytes(m, nb, layout));
    for (int64_t i = 0; i < m; ++i)
        for (int64_t j = 0; j < nb; ++j) out[kqo_sf_offset(i, j, nb, layout)] = rm[i * nb + j];
}

/* Flags for the comparison rules (bit mask per element):
 *   1: |v| within 1e-3 relative of a rounding midpoint
 *   2: the block's amax within 1e-3 relative of a power of two
 *   4: sign of a zero code not decided: |y| <= 2^-16 * bound and the
 *      magnitude rounds to 0. */
static const double kMidpoints[7] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0};

/* Quantize y [m][d] (fp64) into packed codes q [m][ldq] and scales sf. */
KQO_EXPORT void kqo_quantize(const double *y, const double *bound, int64_t m, int64_t d,
                             uint8_t *q, int64_t ldq, uint8_t *sf, int layout,
                             uint8_t *flags)
{
    int64_t nb = d / 32;
    if (layout == 1) memset(sf, 0, (size_t)kqo_sf_bytes(m, nb, layout));
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < nb; ++j) {
            const double *yb = y + i * d + j * 32;
            double amax = 0.0;
            for (int c = 0; c < 32; ++c)
                if (fabs(yb[c]) > amax) amax = fabs(yb[c]);
            int e = kqo_e8m0_exponent(amax);
            sf[kqo_sf_offset(i, j, nb, layout)] = (uint8_t)(e + 127);
            int edge = 0;
            if (amax > 0.0) {
                int ex;
                double f = frexp(amax, &ex);      /* f in [0.5, 1) */
                edge = (f - 0.5 <= 1e-3 * 0.5) || (1.0 - f <= 1e-3 * 1.0);
            }
            uint8_t codes[32];
            for (int c = 0; c < 32; ++c) {
                double v = ldexp(yb[c], -e);      /* y / 2^e, exact */
                codes[c] = kqo_encode_e2m1(v);
                if (flags) {
                    uint8_t fl = edge ? 2 : 0;
                    double av = fabs(v);
                    for (int k = 0; k < 7; ++k)
                        if (fabs(av - kMidpoints[k]) <= 1e-3 * kMidpoints[k]) fl |= 1;
                    if (bound && (codes[c] & 7) == 0 &&
                        fabs(yb[c]) <= ldexp(bound[i * d + j * 32 + c], -16))
                        fl |= 4;
                    flags[i * d + j * 32 + c] = fl;
                }
            }
            for (int k = 0; k < 16; ++k)
                q[i * ldq + j * 16 + k] = (uint8_t)(codes[2 * k] | (codes[2 * k + 1] << 4));
        }
    }
}

/* Dequantize: value(code) * 2^(sf - 127). */
KQO_EXPORT void kqo_dequantize(const uint8_t *q, int64_t ldq, const uint8_t *sf, int layout,
                               int64_t m, int64_t d, double *out)
{
    int64_t nb = d / 32;
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < m; ++i)
        for (int64_t c = 0; c < d; ++c) {
            uint8_t byte = q[i * ldq + c / 2];
            uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
            int e = (int)sf[kqo_sf_offset(i, c / 32, nb, layout)] - 127;
            out[i * d + c] = ldexp(kqo_e2m1_value(code), e);
        }
}

/* Packed codes of the fp32 bit patterns first, first+1, ..., first+count-1
 * taken as values v with scale 2^0 (count even): the expected output of the
 * device encoder under an exhaustive sweep. */
KQO_EXPORT void kqo_encode_f32_range(uint32_t first, int64_t count, uint8_t *packed)
{
    #pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < count / 2; ++k) {
        uint8_t c[2];
        for (int t = 0; t < 2; ++t) {
            uint32_t u = first + (uint32_t)(2 * k + t);
            float f;
            memcpy(&f, &u, sizeof f);
            c[t] = kqo_encode_e2m1((double)f);
        }
        packed[k] = (uint8_t)(c[0] | (c[1] << 4));
    }
}

KQO_EXPORT void kqo_encode_e2m1_array(const double *v, int64_t n, uint8_t *codes)
{
    #pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < n; ++k) codes[k] = kqo_encode_e2m1(v[k]);
}

/* --- 16-bit side output ---------------------------------------------------- */

/* fp64 -> bf16 bit pattern, round to nearest with ties to even.  This is the
 * cast of the transformed activations to the 16-bit input dtype: [KQ] Sec.
 * 3.5.1 (K1 writes y back in the 16-bit type of its input) and App. D
 * "Quantization" (the activations that feed the low-rank branch of eq. (11)
 * stay in 16 bits; bf16 for SANA and FLUX).
 * bf16: 1 sign, 8 exponent, 7 fraction bits.  A finite magnitude is
 * k * 2^(e - 7) with k in [128, 255] in the binade [2^e, 2^(e+1)),
 * e in [-126, 127], and k * 2^-133, k in [0, 127], below 2^-126.  The value is
 * rounded to the nearest multiple of its binade's spacing (ties to an even
 * multiple, rint in the default rounding mode); a carry to k = 256 moves to
 * the next binade, and a rounded magnitude of 2^128 is infinity. */
KQO_EXPORT uint16_t kqo_f64_to_bf16(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    const double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    if (a == 0.0) return sign;
    int E;
    (void)frexp(a, &E);                 /* a in [2^(E-1), 2^E) */
    int e = E - 1;
    if (e < -126) e = -126;             /* subnormal range: spacing 2^-133 */
    const double spacing = ldexp(1.0, e - 7);
    const double r = rint(a / spacing) * spacing;   /* both steps exact */
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    if (r == 0.0) return sign;
    int E2;
    (void)frexp(r, &E2);
    const int e2 = E2 - 1;
    if (e2 < -126) return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -133)));
    const uint16_t field = (uint16_t)(e2 + 127);
    const uint16_t frac = (uint16_t)(r / ldexp(1.0, e2 - 7) - 128.0);
    return (uint16_t)(sign | (uint16_t)(field << 7) | frac);
}

KQO_EXPORT void kqo_f64_to_bf16_array(const double *x, int64_t n, uint16_t *out)
{
    #pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < n; ++k) out[k] = kqo_f64_to_bf16(x[k]);
}
