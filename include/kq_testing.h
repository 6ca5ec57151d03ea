/*
 * kq_testing.h -- verification and benchmarking hooks of libkq_gb300.so.
 *
 * These entry points are not part of the library's interface (include/kq.h):
 * they choose an implementation explicitly, run one stage of a kernel alone,
 * or make a pipeline wait run out on purpose, so that the tests can check
 * each implementation and each error path against the CPU oracle, and the
 * benchmark can time the alternatives.  Conventions (ownership, streams,
 * argument checks, status codes) are those of include/kq.h.
 */
#ifndef KQ_TESTING_H
#define KQ_TESTING_H

#include "kq.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * kq_quantize_mxfp4_variant -- kq_quantize_mxfp4 with the block-transform
 *   implementation chosen explicitly: variant 0 = in-register butterfly
 *   from the raw factors (needs factors), 2 = identity, 3 = tcgen05 tensor
 *   cores with TMEM accumulators on the pre-expanded operand records (needs
 *   K_expanded), 4 = the same tensor-core kernel with the records built in
 *   the kernel from the raw factors ([KQ] Sec. 3.5.1 "K2": K_j constructed on
 *   the fly from its Kronecker factors, no expanded blocks in memory; needs
 *   factors).  Other values (including 1, the warp-level mma.sync variant,
 *   which is no longer built): KQ_ERR_LAYOUT.
 */
KQ_API kq_status kq_quantize_mxfp4_variant(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                           const float *factors, const void *K_expanded,
                                           uint8_t *q, int64_t ldq, uint8_t *sf,
                                           kq_sf_layout sf_layout, float *y_debug, int variant,
                                           cudaStream_t stream);

/*
 * kq_w4a4_gemm_variant -- kq_w4a4_gemm with the implementation chosen:
 *   variant 0 = block-scaled FP4 MMA (kind::mxf4, the default), 1 = every
 *   operand tile dequantized to bf16 in shared memory (exact) and multiplied
 *   with kind::f16 -- an independent route to the same sums, for checking;
 *   2 / 3 = the FP4 kernel with its tile width fixed at 128 / 256 columns of
 *   C (variant 0 picks the width from the number of tiles per SM and K).
 *   Other values: KQ_ERR_LAYOUT.
 */
KQ_API kq_status kq_w4a4_gemm_variant(const uint8_t *qa, int64_t ldqa, const uint8_t *sfa,
                                      const uint8_t *qw, int64_t ldqw, const uint8_t *sfw,
                                      int64_t m, int64_t n, int64_t k, float *c, int64_t ldc,
                                      int variant, cudaStream_t stream);

/*
 * kq_test_encode_e2m1 -- runs the quantizers' E2M1 encoder on the fp32 bit
 *   patterns first, first+1, ..., first+count-1 with the scale fixed at 2^0
 *   (v = y), writing count/2 packed bytes (code of the even pattern in bits
 *   0-3).  count must be a multiple of 8; out is device memory, 16-byte
 *   aligned.  Used for the exhaustive rounding check.
 */
KQ_API kq_status kq_test_encode_e2m1(uint32_t first, int64_t count, uint8_t *out,
                                     cudaStream_t stream);

/*
 * kq_test_quantize_stall -- the tensor-core quantizer (kq_quantize_mxfp4 on
 *   K_expanded) with its pipeline made to stall on purpose: the producer of
 *   the CTA that owns tile `skip_tile` (row tile * column tiles + column
 *   tile, in 128-row x 64-channel tiles; the tiled scale layout also counts
 *   its padding column tiles; with G = min(tiles, SMs) CTAs, CTA c owns the
 *   tiles c, c + G, c + 2G, ... in that order) arms that tile's ring stage
 *   but never issues its loads, and every wait of the kernel gives up after
 *   wait_limit_ns nanoseconds (1 ms to 1 s, KQ_ERR_SHAPE otherwise) instead
 *   of one second.  The kernel then takes the path a real stall would take:
 *   it returns, with the E8M0 NaN byte 0xFF as the scale (and zero codes) of
 *   every block it did not finish.  Nothing faults: no access goes out of
 *   bounds and every wait ends.  skip_tile = -1 runs the kernel normally
 *   with the given limit.
 */
KQ_API kq_status kq_test_quantize_stall(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                        const void *K_expanded, uint8_t *q, int64_t ldq,
                                        uint8_t *sf, kq_sf_layout sf_layout, int64_t skip_tile,
                                        uint64_t wait_limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KQ_TESTING_H */
