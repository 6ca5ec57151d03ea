// Internal declarations shared by the translation units of the library.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kq.h"
#include "kq_testing.h"
#include "kq_records.h"

namespace kq {

enum Transform : int {
    kKron = 0,      // five 2x2 factors per block, in-register butterfly
    kDiag = 1,      // y = a * s[c]
    kHadamard = 2,  // y = a . H32 / sqrt(32)
    kIdentity = 3   // y = a
};

// Arguments of the TMA-fed quantizer kernels.
struct QuantParams {
    int64_t m;          // rows
    int64_t m_rows;     // rows the grid covers (m, or m padded to 128 for the blocked layout)
    int64_t d;          // channels
    int64_t nb;         // d / 32
    int64_t ncol_tiles; // ceil(nb / 4)
    int64_t nrow_tiles; // ceil(m_rows / BR)
    int64_t ntiles;
    const float *factors;  // kKron: [nb][5][2][2]
    const float *s;        // kDiag: [d]
    uint8_t *q;
    int64_t ldq;
    uint8_t *sf;
    int sf_layout;
    int64_t ncb;        // ceil(nb / 4), for the blocked layout
    float *y_debug;     // [m][d] or null
    int shared_params;  // 1: every block takes block 0's factors / operand records
    int in_f16;         // 1: A holds fp16 bit patterns (CUDA-core kernels), 0: bf16
    // tcgen05 kernel only:
    uint64_t wait_limit_ns; // bound of every pipeline wait
    int64_t skip_tile;      // verification hook: a tile whose loads are never issued (-1: none)
};

// Per-device facts the launchers need.
struct DeviceInfo {
    int sm_count;
    bool supported;  // compute capability 10.3
};

kq_status device_info(DeviceInfo &info);
kq_status make_tensor_map_2d_bf16(CUtensorMap *map, const void *base, int64_t rows, int64_t cols,
                                  int64_t ld_elems, uint32_t box_cols, uint32_t box_rows);
kq_status make_tensor_map_2d_u8(CUtensorMap *map, void *base, int64_t rows, int64_t cols,
                                int64_t ld_bytes, uint32_t box_cols, uint32_t box_rows,
                                CUtensorMapSwizzle swizzle);
kq_status make_tensor_map_2d_f32(CUtensorMap *map, void *base, int64_t rows, int64_t cols,
                                 int64_t ld_elems, uint32_t box_cols, uint32_t box_rows,
                                 CUtensorMapSwizzle swizzle);
kq_status check_launch();

// The kernels walk tiles in 32-bit arithmetic: row and column tile indices,
// and the walk's start and stride (at most twice the grid), must fit in int.
inline bool tiles_fit_int32(const QuantParams &p, int grid)
{
    const int64_t lim = (int64_t(1) << 30);
    return p.nrow_tiles < lim && p.ncol_tiles < lim && p.ntiles < lim && grid < (1 << 20);
}

// Launches a persistent quantizer kernel with programmatic stream
// serialization: the launch may begin while the previous kernel of the
// stream is still running; the kernel orders its global-memory accesses
// after that kernel with griddepcontrol.wait.
template <typename... KArgs, typename... Args>
kq_status launch_pdl(void (*kern)(KArgs...), int grid, int block, size_t smem,
                     cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...) == cudaSuccess ? KQ_OK : KQ_ERR_CUDA;
}

kq_status launch_quant_tma(Transform t, const uint16_t *A, int64_t lda, const QuantParams &p,
                           cudaStream_t stream);
// The tcgen05 operand records of kq_expand_blocks (KQ_K_BF16X3).
kq_status launch_umma_records(const float *factors, int64_t nb, void *out, cudaStream_t stream);
// Full-row Walsh-Hadamard + MXFP4 (d a power of two, 128 <= d <= 16384).
kq_status launch_quant_fwht(const uint16_t *A, int64_t lda, const QuantParams &p,
                            cudaStream_t stream);
// at != nullptr: also write the bf16 side output A T ([m][ldat], the DUAL kernel);
// K_expanded == nullptr: the K2 form, building the operand records in the
// kernel from p.factors (no side output)
kq_status launch_quant_umma(const uint16_t *A, int64_t lda, const void *K_expanded,
                            const QuantParams &p, uint16_t *at, int64_t ldat, cudaStream_t stream);

// C = A_q W_q^T from packed codes + 128x4 tiled scales (variant 0: block-scaled
// kind::mxf4 MMA; 1: dequantized to bf16 in shared memory, kind::f16), and
// C = A W^T in bf16 (tcgen05 GEMM); the fp64 error sums of eq. (2).
kq_status launch_w4a4_gemm(const uint8_t *qa, int64_t ldqa, const uint8_t *sfa, const uint8_t *qw,
                           int64_t ldqw, const uint8_t *sfw, int64_t m, int64_t n, int64_t k,
                           float *c, int64_t ldc, int variant, cudaStream_t stream);
kq_status launch_bf16_gemm(const uint16_t *a, int64_t lda, const uint16_t *w, int64_t ldw,
                           int64_t m, int64_t n, int64_t k, float *c, int64_t ldc,
                           cudaStream_t stream);
kq_status launch_layer_error(const float *c, int64_t ldc, const float *r, int64_t ldr, int64_t m,
                             int64_t n, double *out, cudaStream_t stream);

kq_status validate_quant_args(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                              const uint8_t *q, int64_t ldq, const uint8_t *sf,
                              kq_sf_layout layout, const float *y_debug);
void fill_quant_params(QuantParams &p, int64_t m, int64_t d, int64_t rows_per_tile, uint8_t *q,
                       int64_t ldq, uint8_t *sf, kq_sf_layout layout, float *y_debug);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace kq
