/*
 * kq.h -- C ABI of the GB300 (sm_103a) KroQuant MXFP4 activation quantizer.
 *
 * What it computes ("KroQuant: Kronecker-Structured Block Transforms for
 * Efficient Post-Training Quantization of Diffusion Transformers",
 * arXiv 2607.21446v1, cited below as [KQ]):
 *   - eq. (4): T = diag(K_1, ..., K_nb) is block diagonal with 32x32 blocks;
 *   - eq. (5): K_j = G1 (x) G2 (x) G3 (x) G4 (x) G5, five 2x2 factors;
 *   - eq. (12): K_j[r][c] = prod_k G_k[bit_{5-k}(r)][bit_{5-k}(c)], so G1
 *     acts on bit 4 (most significant) of the channel index within a block;
 *   - Sec. 3.5.1 (K1, "A_tile @ K"): every row a of A is transformed as the
 *     row vector y = a . K_j per 32-channel block j;
 *   - Sec. 3.1 and 4.1: y is quantized to MXFP4 -- per 32-element block one
 *     E8M0 scale 2^e with e = floor(log2 amax) - 2 (clamped to [-127, 127],
 *     e = -127 when amax = 0) and 32 FP4 E2M1 codes of y / 2^e, rounded to
 *     nearest with ties to even, saturated to +-6, sign kept (also -0).
 *
 * Data layout.
 *   A       bf16 bit patterns, row-major [m][lda], lda >= d.
 *   q       packed E2M1 codes, row-major [m][ldq] bytes, ldq >= d/2; byte k
 *           of a row holds code 2k in bits 0-3 and code 2k+1 in bits 4-7
 *           (code = sign << 3 | E2M1 magnitude index 0..7).
 *   sf      E8M0 scale bytes (e + 127), nb = d/32 per row, either
 *           KQ_SF_ROWMAJOR [m][nb], or KQ_SF_BLOCKED_128x4, the tiled layout
 *           that block-scaled MMA reads: tiles of 128 rows x 4 block-columns,
 *           512 bytes each, tiles in row-tile-major order; inside a tile the
 *           scale of (row i, block kb) sits at
 *           (i % 32) * 16 + ((i % 128) / 32) * 4 + (kb % 4).  Rows are padded
 *           to a multiple of 128 and block-columns to a multiple of 4; the
 *           library writes 0x00 into the padding.  kq_sf_bytes() gives the size.
 *   factors fp32 raw 2x2 entries [nb][5][2][2]: factor k of block j is
 *           factors[((j*5 + k)*2 + r)*2 + c] = G_{k+1}[r][c].  Any raw
 *           entries are accepted (both determinant-sign conventions of the
 *           LU form, eq. 6, and the Hadamard factor of Sec. 3.2).
 *
 * Ownership and execution.  The caller allocates and owns every buffer.
 * Entry points taking a cudaStream_t validate their arguments on the host,
 * then enqueue work on that stream and return without synchronizing;
 * results are valid once the stream reaches that point.  They never
 * allocate, free or synchronize.  Device-pointer arguments must be device
 * (or managed) memory of the current device.
 *
 * Errors.  Argument checks run before anything is enqueued; a failed check
 * returns its status and enqueues nothing.  A launch failure reported by the
 * CUDA runtime returns KQ_ERR_CUDA.  m = 0 is a valid no-op (KQ_OK).
 * A kernel that finds its data pipeline stalled for longer than about one
 * second stops waiting and writes the E8M0 NaN byte 0xFF as the scale of
 * every block it could not finish (finite inputs never produce 0xFF).
 */
#ifndef KQ_H
#define KQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define KQ_API __attribute__((visibility("default")))
#else
#define KQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kq_status {
    KQ_OK = 0,
    KQ_ERR_NULL = 1,        /* a required pointer is NULL */
    KQ_ERR_SHAPE = 2,       /* m < 0, d <= 0, d % 32 != 0, lda < d, ldq < d/2, nb <= 0 */
    KQ_ERR_ALIGN = 3,       /* a pointer or leading dimension breaks the alignment rules */
    KQ_ERR_LAYOUT = 4,      /* unknown kq_sf_layout / kq_kfmt / variant / sign value */
    KQ_ERR_CUDA = 5,        /* the CUDA runtime or driver reported an error */
    KQ_ERR_UNSUPPORTED = 6  /* the current device is not sm_103 (GB300) */
} kq_status;

typedef enum kq_sf_layout {
    KQ_SF_ROWMAJOR = 0,
    KQ_SF_BLOCKED_128x4 = 1
} kq_sf_layout;

typedef enum kq_kfmt {
    KQ_K_FP32 = 0,      /* dense K_j, fp32 row-major [nb][32][32] */
    KQ_K_BF16X3 = 1     /* operand records of the tensor-core kernel (opaque,
                           6144 bytes per block): the dense 32x32 K_j as a
                           three-term bf16 split hi + mid + lo, in the
                           shared-memory operand layout of its MMAs */
} kq_kfmt;

/* Input formats of kq_quantize_mxfp4_ex: A holds bf16 or fp16 bit patterns. */
typedef enum {
    KQ_IN_BF16 = 0,
    KQ_IN_F16 = 1
} kq_in_format;

/* Transforms of kq_quantize_mxfp4_ex (the CUDA-core kernels). */
typedef enum {
    KQ_TRANSFORM_KRON = 0,      /* eq. (12) from the raw factors (butterfly) */
    KQ_TRANSFORM_DIAG = 1,      /* y = a * s[c] */
    KQ_TRANSFORM_HADAMARD = 2,  /* H32 / sqrt(32) per block */
    KQ_TRANSFORM_IDENTITY = 3,  /* the bare quantizer */
    KQ_TRANSFORM_FWHT = 4       /* H_d / sqrt(d) over the row */
} kq_transform;

/* Alignment rules shared by the quantizer entry points:
 *   A, q, sf, y_debug, factors, s, K_expanded: 16-byte aligned;
 *   lda % 8 == 0 (16-byte row pitch), ldq % 16 == 0. */

/*
 * kq_quantize_mxfp4 -- the KroQuant online activation quantizer.
 * [KQ] eq. (4), (5), (12); Sec. 3.5 (one pass: transform, then the fused
 * MXFP4 quantizer); Sec. 3.1 / 4.1 (MXFP4).
 *   A          device, bf16 [m][lda] (read only)
 *   m, d, lda  rows, channels (d % 32 == 0), row pitch in elements
 *   factors    device, fp32 [d/32][5][2][2] raw factor entries, or NULL
 *   K_expanded device, output of kq_expand_blocks(..., KQ_K_BF16X3, ...), or
 *              NULL.  With K_expanded != NULL the transform runs on the
 *              tensor cores (tcgen05.mma, fp32 accumulation in TMEM) against
 *              the dense 32x32 K_j as three bf16 terms -- the fastest path.
 *              Otherwise, with factors != NULL, the same tensor-core kernel
 *              builds the three bf16 terms of each K_j itself, from the raw
 *              factors (eq. 12 as fp32 products, [KQ] Sec. 3.5.1 "K2": no
 *              expanded blocks in memory); with both NULL the transform is
 *              the identity (the bare quantizer, "Q4" of [KQ] Tables 3 and
 *              4).  Both paths compute y to about fp32 precision (|error| <=
 *              2^-16 * sum_r |a_r K_rc|); the CUDA-core butterfly on the raw
 *              factors is kq_quantize_mxfp4_ex(..., KQ_TRANSFORM_KRON, ...).
 *   q, ldq     device, packed codes [m][ldq] (written)
 *   sf         device, scales in sf_layout (written; kq_sf_bytes() bytes)
 *   y_debug    device fp32 [m][d] or NULL: if given, receives y = a . K_j
 *              exactly as it enters the quantizer (for verification)
 *   stream     CUDA stream (0 = legacy default stream)
 */
KQ_API kq_status kq_quantize_mxfp4(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                            const float *factors, const void *K_expanded,
                            uint8_t *q, int64_t ldq, uint8_t *sf, kq_sf_layout sf_layout,
                            float *y_debug, cudaStream_t stream);

/*
 * kq_quantize_mxfp4_dual -- kq_quantize_mxfp4 on the tensor-core path that
 * also writes the 16-bit side output A T in the same pass: [KQ] eq. (11)
 * evaluates Q(A T) x Q(W~ - L R) + (A T) L R, the low-rank branch taking
 * A T in 16 bits (App. D "Quantization"; bf16 for SANA and FLUX), cast from
 * the transform's fp32 result as K1 does (Sec. 3.5.1).
 *   K_expanded  device, output of kq_expand_blocks(..., KQ_K_BF16X3, ...)
 *               (required)
 *   at, ldat    device, bf16 [m][ldat] (written, columns < d): at[i][c] is y
 *               rounded to bf16 (nearest, ties to even) -- the same y that is
 *               quantized into q / sf.  ldat >= d, ldat % 8 == 0, 16-byte
 *               aligned.  A block that timed out (see Errors above) gets
 *               bf16 NaNs.
 *   other arguments as kq_quantize_mxfp4.
 */
KQ_API kq_status kq_quantize_mxfp4_dual(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                 const void *K_expanded, uint8_t *q, int64_t ldq, uint8_t *sf,
                                 kq_sf_layout sf_layout, uint16_t *at, int64_t ldat,
                                 float *y_debug, cudaStream_t stream);

/*
 * kq_quantize_mxfp4_shared -- kq_quantize_mxfp4 with one factor set shared
 * by every 32-channel block, K_j = K for all j ([KQ] Sec. 3.5.1 on K2: the case where
 * several column blocks use one set of Kronecker factors, so that storing
 * the transform per block is wasted).
 *   factors     device fp32 [5][2][2]: the shared G1..G5, or NULL
 *   K_expanded  device, kq_expand_blocks(factors, 1, KQ_K_BF16X3, ...)
 *               (kq_expanded_bytes(1, KQ_K_BF16X3) bytes), or NULL; with it
 *               the tensor cores read that record for every block,
 *               otherwise they build it from `factors` (the K2 form of
 *               kq_quantize_mxfp4).  One of the two is required
 *               (KQ_ERR_NULL).
 *   other arguments as kq_quantize_mxfp4; the result equals
 *   kq_quantize_mxfp4 given the set repeated d/32 times.
 */
KQ_API kq_status kq_quantize_mxfp4_shared(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                          const float *factors, const void *K_expanded,
                                          uint8_t *q, int64_t ldq, uint8_t *sf,
                                          kq_sf_layout sf_layout, float *y_debug,
                                          cudaStream_t stream);

/*
 * kq_quantize_mxfp4_ex -- the CUDA-core quantizers with the input format
 * chosen: bf16, or fp16 as PixArt-Sigma runs and as [KQ] times its kernels
 * (Sec. 4.1 "Data format", Sec. 4.4: FP16 activations).  fp16 values enter
 * the transform exactly (every fp16 is an fp32).
 *   A          device, [m][lda] 16-bit patterns in in_format
 *   transform  KQ_TRANSFORM_*; param = factors [d/32][5][2][2] (KRON) or
 *              s [d] (DIAG), device fp32, 16-byte aligned; NULL otherwise
 *              (ignored).  FWHT needs a power-of-two d in [128, 16384].
 *   other arguments as kq_quantize_mxfp4.  An unknown format or transform
 *   gives KQ_ERR_LAYOUT.  The tensor-core path (kq_quantize_mxfp4 with
 *   K_expanded) reads bf16 only: its MMA takes both operands in one type.
 */
KQ_API kq_status kq_quantize_mxfp4_ex(const uint16_t *A, kq_in_format in_format, int64_t m,
                                      int64_t d, int64_t lda, kq_transform transform,
                                      const float *param, uint8_t *q, int64_t ldq, uint8_t *sf,
                                      kq_sf_layout sf_layout, float *y_debug,
                                      cudaStream_t stream);

/*
 * kq_smooth_quantize_mxfp4 -- diagonal-scale baseline: T = diag(s),
 * y[i][c] = a[i][c] * s[c], then the same MXFP4 quantizer ([KQ] Sec. 4.4,
 * "Scale", per-channel scaling of SmoothQuant; a SmoothQuant user passes
 * s = 1/gamma with gamma of Appendix D.2).
 *   s  device fp32 [d]; other arguments as kq_quantize_mxfp4.
 */
KQ_API kq_status kq_smooth_quantize_mxfp4(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                   const float *s, uint8_t *q, int64_t ldq, uint8_t *sf,
                                   kq_sf_layout sf_layout, float *y_debug, cudaStream_t stream);

/*
 * kq_hadamard_quantize_mxfp4 -- fixed block-Hadamard baseline: every K_j is
 * the normalised 32-point Walsh-Hadamard matrix H32 / sqrt(32) (Sylvester
 * order, H32[r][c] = (-1)^popcount(r & c)), [KQ] Sec. 3.2 "Hadamard
 * initialization" and Table 2 "Hadamard (32x32)".  Arguments as
 * kq_quantize_mxfp4.
 */
KQ_API kq_status kq_hadamard_quantize_mxfp4(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                     uint8_t *q, int64_t ldq, uint8_t *sf,
                                     kq_sf_layout sf_layout, float *y_debug, cudaStream_t stream);

/*
 * kq_fwht_quantize_mxfp4 -- full-row Walsh-Hadamard baseline: every row is
 * transformed by the normalised d-point Walsh-Hadamard matrix,
 * y = a . H_d / sqrt(d), H_d[r][c] = (-1)^popcount(r & c) (Sylvester order),
 * then quantized like kq_quantize_mxfp4 ([KQ] Sec. 4.4 and Table 3, "FWHT";
 * it needs a power-of-two d).  d must be a power of two with
 * 128 <= d <= 16384 (KQ_ERR_SHAPE otherwise); other arguments as
 * kq_quantize_mxfp4.
 */
KQ_API kq_status kq_fwht_quantize_mxfp4(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                 uint8_t *q, int64_t ldq, uint8_t *sf,
                                 kq_sf_layout sf_layout, float *y_debug, cudaStream_t stream);

/*
 * kq_w4a4_gemm -- the W4A4 product that consumes the quantizer's output,
 * [KQ] eq. (11) (Q(A T) x Q(W~)) and eq. (2):
 *     c[i][j] = sum_k deq(qa)[i][k] * deq(qw)[j][k]      (C = A_q W_q^T)
 * with deq = e2m1(code) * 2^(sf - 127) as in kq_dequantize.  Runs on the
 * FP4 tensor cores (tcgen05.mma kind::mxf4, block-scaled: the instruction
 * reads the packed codes and applies the E8M0 scales itself), fp32
 * accumulation in TMEM.  The element products are exact; only the fp32
 * accumulation rounds.
 *   qa, ldqa   device, packed codes of the m x k left operand [m][ldqa]
 *              (as kq_quantize_mxfp4 writes them; ldqa >= k/2, ldqa % 16 == 0)
 *   sfa        device, its scales in KQ_SF_BLOCKED_128x4 (kq_sf_bytes(m, k))
 *   qw, ldqw   device, packed codes of the n x k right operand (weights,
 *              output channel j in row j)
 *   sfw        device, its scales in KQ_SF_BLOCKED_128x4 (kq_sf_bytes(n, k))
 *   m, n, k    k % 32 == 0, k > 0; m, n >= 0 (m or n = 0: no-op)
 *   c, ldc     device fp32 [m][ldc] (written, columns < n), ldc >= n,
 *              ldc % 4 == 0, 16-byte aligned
 * Scale bytes of padding blocks (columns past k) are not used; 0xFF (the
 * E8M0 NaN) in a used block yields NaN.  A kernel that finds its pipeline
 * stalled for about one second stops; the output tiles it had not written
 * are then left as they were.
 */
KQ_API kq_status kq_w4a4_gemm(const uint8_t *qa, int64_t ldqa, const uint8_t *sfa,
                              const uint8_t *qw, int64_t ldqw, const uint8_t *sfw,
                              int64_t m, int64_t n, int64_t k, float *c, int64_t ldc,
                              cudaStream_t stream);

/*
 * kq_bf16_gemm -- the unquantized reference product of [KQ] eq. (2),
 * c = A W^T, on the same tensor-core kernel: bf16 operands, fp32
 * accumulation.
 *   a, lda     device, bf16 [m][lda] (lda >= k, lda % 8 == 0)
 *   w, ldw     device, bf16 [n][ldw] (ldw >= k, ldw % 8 == 0)
 *   m, n, k    k > 0; m, n >= 0 (m or n = 0: no-op)
 *   c, ldc     as kq_w4a4_gemm
 */
KQ_API kq_status kq_bf16_gemm(const uint16_t *a, int64_t lda, const uint16_t *w, int64_t ldw,
                              int64_t m, int64_t n, int64_t k, float *c, int64_t ldc,
                              cudaStream_t stream);

/*
 * kq_layer_error -- the squared Frobenius norms behind [KQ] eq. (2):
 *     out[0] = sum_ij (c[i][j] - c_ref[i][j])^2   (||E(T)||_F^2 when c is
 *              the W4A4 product and c_ref = A W^T)
 *     out[1] = sum_ij c_ref[i][j]^2
 * accumulated in fp64 (squares of fp32 differences are exact in fp64; the
 * order of the additions is not fixed).
 *   c, ldc, c_ref, ldr  device fp32 [m][ldc], [m][ldr] (ld >= n, % 4 == 0,
 *                       16-byte aligned)
 *   out                 device double[2] (overwritten; 8-byte aligned)
 */
KQ_API kq_status kq_layer_error(const float *c, int64_t ldc, const float *c_ref, int64_t ldr,
                                int64_t m, int64_t n, double *out, cudaStream_t stream);

/*
 * kq_expand_blocks -- [KQ] Sec. 3.5.1 K1 (the dense 32x32 blocks are kept
 * in device memory): expand the raw factors into dense blocks by eq. (12),
 * computed in fp64 and then rounded to the requested format.
 *   factors  device fp32 [nb][5][2][2]
 *   nb       number of 32-channel blocks (> 0)
 *   fmt      KQ_K_FP32 (row-major [nb][32][32] fp32) or KQ_K_BF16X3 (the
 *            tensor-core operand records consumed by kq_quantize_mxfp4)
 *   K_out    device, kq_expanded_bytes(nb, fmt) bytes, 16-byte aligned
 */
KQ_API kq_status kq_expand_blocks(const float *factors, int64_t nb, kq_kfmt fmt, void *K_out,
                           cudaStream_t stream);

/* Bytes kq_expand_blocks writes for nb blocks in format fmt (0 if invalid). */
KQ_API size_t kq_expanded_bytes(int64_t nb, kq_kfmt fmt);

/*
 * kq_dequantize -- MXFP4 decode: out[i][c] = e2m1(code) * 2^(sf - 127),
 * exact in fp32 (OCP MX element x shared scale; [KQ] Sec. 3.1, Q_b returns
 * the dequantized matrix).
 *   q, ldq, sf, sf_layout  as written by the quantizers (device)
 *   m, d                   shape of the quantized matrix
 *   out                    device fp32 [m][d] (16-byte aligned)
 */
KQ_API kq_status kq_dequantize(const uint8_t *q, int64_t ldq, const uint8_t *sf,
                        kq_sf_layout sf_layout, int64_t m, int64_t d, float *out,
                        cudaStream_t stream);

/* Bytes of the scale array for an m x d matrix (padded for the blocked
 * layout); 0 if the arguments are invalid. */
KQ_API size_t kq_sf_bytes(int64_t m, int64_t d, kq_sf_layout sf_layout);

/* Static, never-NULL description of a status code. */
KQ_API const char *kq_status_string(kq_status status);

/*
 * Host helpers (host memory, synchronous, no CUDA calls).
 *
 * kq_lu_to_factors -- [KQ] eq. (6): lu [nb][5][3] = (a, b, c) per factor,
 *   G = [[1, 0], [c, 1]] . [[a, b], [0, det_sign / a]], evaluated in fp64 and
 *   rounded once to fp32 into factors [nb][5][2][2].  det_sign = -1 is the
 *   paper's form (det G = -1), +1 the unit-determinant form.  a == 0 gives
 *   KQ_ERR_SHAPE.
 */
KQ_API kq_status kq_lu_to_factors(const float *lu, int64_t nb, int det_sign, float *factors);

/*
 * kq_invert_transpose_factors -- factors of K_j^{-T} = (x)_k G_k^{-T}
 *   ([KQ] Sec. 3.2: the inverse of a Kronecker product is the Kronecker
 *   product of the inverses; eq. (1): the weights take W T^{-T}).  Each 2x2
 *   inverse-transpose is evaluated in fp64 and rounded once to fp32.  A
 *   singular factor gives KQ_ERR_SHAPE.  Feed the result to
 *   kq_quantize_mxfp4 to quantize the rows of W T^{-T}.
 */
KQ_API kq_status kq_invert_transpose_factors(const float *factors, int64_t nb, float *out);

#ifdef __cplusplus
}
#endif

#endif /* KQ_H */
