// C ABI entry points of the KroQuant MXFP4 quantizer, the argument checks,
// device facts, TMA descriptors, and the auxiliary kernels (dequantize,
// dense block expansion, encoder sweep).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {

// ---------------------------------------------------------------------------
// device facts

kq_status device_info(DeviceInfo &info)
{
    static std::once_flag once[64];
    static DeviceInfo cache[64];
    static cudaError_t errs[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KQ_ERR_CUDA;
    std::call_once(once[dev], [dev] {
        int major = 0, minor = 0, sms = 0;
        cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        errs[dev] = e;
        cache[dev].sm_count = sms;
        cache[dev].supported = (major == 10 && minor == 3);
    });
    if (errs[dev] != cudaSuccess) return KQ_ERR_CUDA;
    info = cache[dev];
    return info.supported ? KQ_OK : KQ_ERR_UNSUPPORTED;
}

kq_status check_launch()
{
    return cudaGetLastError() == cudaSuccess ? KQ_OK : KQ_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// TMA descriptor (driver entry point fetched through the runtime, so the
// library needs no link-time dependency on libcuda)

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

kq_status make_tensor_map_2d_bf16(CUtensorMap *map, const void *base, int64_t rows, int64_t cols,
                                  int64_t ld_elems, uint32_t box_cols, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (fn == nullptr) return KQ_ERR_CUDA;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_elems) * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KQ_OK : KQ_ERR_CUDA;
}

kq_status make_tensor_map_2d_u8(CUtensorMap *map, void *base, int64_t rows, int64_t cols,
                                int64_t ld_bytes, uint32_t box_cols, uint32_t box_rows,
                                CUtensorMapSwizzle swizzle)
{
    auto fn = encode_fn();
    if (fn == nullptr) return KQ_ERR_CUDA;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_bytes)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KQ_OK : KQ_ERR_CUDA;
}

kq_status make_tensor_map_2d_f32(CUtensorMap *map, void *base, int64_t rows, int64_t cols,
                                 int64_t ld_elems, uint32_t box_cols, uint32_t box_rows,
                                 CUtensorMapSwizzle swizzle)
{
    auto fn = encode_fn();
    if (fn == nullptr) return KQ_ERR_CUDA;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_elems) * 4};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KQ_OK : KQ_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// argument checks (host only; nothing is enqueued when they fail)

kq_status validate_quant_args(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                              const uint8_t *q, int64_t ldq, const uint8_t *sf,
                              kq_sf_layout layout, const float *y_debug)
{
    if (m < 0 || d <= 0 || d % 32 != 0 || lda < d || ldq < d / 2) return KQ_ERR_SHAPE;
    // 2-D TMA coordinates are int32; the row pitch must stay below 2^40 bytes
    if (m > 0x7fffffffLL || d > 0x7fffffffLL || lda > (1LL << 38)) return KQ_ERR_SHAPE;
    if (layout != KQ_SF_ROWMAJOR && layout != KQ_SF_BLOCKED_128x4) return KQ_ERR_LAYOUT;
    if (m == 0) return KQ_OK;
    if (A == nullptr || q == nullptr || sf == nullptr) return KQ_ERR_NULL;
    if (!aligned16(A) || !aligned16(q) || !aligned16(sf) || lda % 8 != 0 || ldq % 16 != 0)
        return KQ_ERR_ALIGN;
    if (y_debug != nullptr && !aligned16(y_debug)) return KQ_ERR_ALIGN;
    return KQ_OK;
}

void fill_quant_params(QuantParams &p, int64_t m, int64_t d, int64_t rows_per_tile, uint8_t *q,
                       int64_t ldq, uint8_t *sf, kq_sf_layout layout, float *y_debug)
{
    p.m = m;
    p.m_rows = (layout == KQ_SF_BLOCKED_128x4) ? ((m + 127) / 128) * 128 : m;
    p.d = d;
    p.nb = d / 32;
    p.ncol_tiles = (p.nb + 3) / 4;
    p.nrow_tiles = (p.m_rows + rows_per_tile - 1) / rows_per_tile;
    p.ntiles = p.nrow_tiles * p.ncol_tiles;
    p.factors = nullptr;
    p.s = nullptr;
    p.q = q;
    p.ldq = ldq;
    p.sf = sf;
    p.sf_layout = static_cast<int>(layout);
    p.ncb = (p.nb + 3) / 4;
    p.y_debug = y_debug;
    p.shared_params = 0;
    p.in_f16 = 0;
    p.wait_limit_ns = kWaitLimitNs;
    p.skip_tile = -1;
}

// ---------------------------------------------------------------------------
// auxiliary kernels

namespace {

// fp32 bits of an E2M1 code: sign | magnitude from the 2-bit exponent
// (bias 1) and 1-bit mantissa; exponent 0 is the subnormal 0 / 0.5.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c)
{
    const uint32_t E = (c >> 1) & 3u, M = c & 1u, sgn = (c & 8u) << 28;
    const uint32_t mag = E ? (((E + 126u) << 23) | (M << 22)) : (M ? 0x3F000000u : 0u);
    return __uint_as_float(sgn | mag);
}

// 2^(byte - 127) as fp32; byte 0 is the subnormal 2^-127.
__device__ __forceinline__ float e8m0_to_f32(uint32_t byte)
{
    return __uint_as_float(byte ? (byte << 23) : 0x00400000u);
}

__global__ void dequant_kernel(const uint8_t *__restrict__ q, int64_t ldq,
                               const uint8_t *__restrict__ sf, int layout, int64_t m, int64_t nb,
                               float *__restrict__ out)
{
    const int64_t n = m * nb, ncb = (nb + 3) / 4;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = idx / nb, j = idx % nb;
        const uint4 c = *reinterpret_cast<const uint4 *>(q + row * ldq + j * 16);
        const uint32_t byte = layout == KQ_SF_ROWMAJOR ? sf[row * nb + j]
                                                       : sf[sf_blocked_offset(row, j, ncb)];
        const float scale = e8m0_to_f32(byte);
        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
        float *o = out + row * (nb * 32) + j * 32;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float v[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) v[t] = e2m1_to_f32((words[k] >> (4 * t)) & 15u) * scale;
            stg_f4(o + 8 * k, make_float4(v[0], v[1], v[2], v[3]));
            stg_f4(o + 8 * k + 4, make_float4(v[4], v[5], v[6], v[7]));
        }
    }
}

// Dense K_j by eq. (12), one thread per entry, product in fp64.
__global__ void expand_kernel(const float *__restrict__ factors, int64_t nb,
                              void *__restrict__ out)
{
    const int64_t n = nb * 1024;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t j = idx >> 10;
        const int r = static_cast<int>((idx >> 5) & 31), c = static_cast<int>(idx & 31);
        const float *f = factors + j * 20;
        double k = 1.0;
#pragma unroll
        for (int t = 0; t < 5; ++t) {
            const int bit = 4 - t;
            k *= static_cast<double>(f[t * 4 + ((r >> bit) & 1) * 2 + ((c >> bit) & 1)]);
        }
        static_cast<float *>(out)[idx] = static_cast<float>(k);
    }
}

// The quantizers' encoder on consecutive fp32 bit patterns at scale 2^0.
__global__ void encode_sweep_kernel(uint32_t first, int64_t n8, uint32_t *__restrict__ out)
{
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint32_t b = first + static_cast<uint32_t>(8 * i);
        float2 Y[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
            Y[t] = make_float2(__uint_as_float(b + 2 * t), __uint_as_float(b + 2 * t + 1));
        const float s = inv_scale(127u);
        const float2 s2 = make_float2(s, s);
        float2 V[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) V[t] = __fmul2_rn(Y[t], s2);
        out[i] = e2m1x8(V[0].x, V[0].y, V[1].x, V[1].y, V[2].x, V[2].y, V[3].x, V[3].y);
    }
}

int grid_for(int64_t work, int threads)
{
    DeviceInfo info{};
    int sms = 148;
    if (device_info(info) == KQ_OK) sms = info.sm_count;
    const int64_t blocks = (work + threads - 1) / threads;
    return static_cast<int>(std::min<int64_t>(std::max<int64_t>(blocks, 1), 8LL * sms));
}

}  // namespace
}  // namespace kq

using namespace kq;

namespace {

// The quantizer entry points: argument checks, then the implementation
// `variant` (0 butterfly, 2 identity, 3 tcgen05 on the expanded records,
// 4 tcgen05 building the records in the kernel from the raw factors, K2).
// `extra` carries the tcgen05 kernel's wait limit and verification hook (its
// other fields are filled here).
kq_status quantize_variant(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                           const float *factors, const void *K_expanded, uint8_t *q, int64_t ldq,
                           uint8_t *sf, kq_sf_layout sf_layout, float *y_debug, int variant,
                           const QuantParams &extra, cudaStream_t stream)
{
    if (variant != 0 && variant != 2 && variant != 3 && variant != 4) return KQ_ERR_LAYOUT;
    kq_status st = validate_quant_args(A, m, d, lda, q, ldq, sf, sf_layout, y_debug);
    if (st != KQ_OK) return st;
    if ((variant == 0 || variant == 4) && factors == nullptr) return KQ_ERR_NULL;
    if (variant == 3 && K_expanded == nullptr) return KQ_ERR_NULL;
    if ((variant == 0 || variant == 4) && !aligned16(factors)) return KQ_ERR_ALIGN;
    if (variant == 3 && !aligned16(K_expanded)) return KQ_ERR_ALIGN;
    if (m == 0) return KQ_OK;
    DeviceInfo info;
    if ((st = device_info(info)) != KQ_OK) return st;
    QuantParams p;
    fill_quant_params(p, m, d, 128, q, ldq, sf, sf_layout, y_debug);
    if (variant == 3 || variant == 4) {
        p.wait_limit_ns = extra.wait_limit_ns;
        p.skip_tile = extra.skip_tile;
        if (variant == 4) p.factors = factors;
        return launch_quant_umma(A, lda, variant == 3 ? K_expanded : nullptr, p, nullptr, 0,
                                 stream);
    }
    if (variant == 0) {
        p.factors = factors;
        return launch_quant_tma(kKron, A, lda, p, stream);
    }
    return launch_quant_tma(kIdentity, A, lda, p, stream);
}

// The fastest implementation the arguments allow: tcgen05 on the expanded
// blocks, else tcgen05 building the blocks from the raw factors (K2), else
// identity.  Measured on GB300 (steady state, FLUX-shaped activations): the
// records path is the fastest on every shape from 256 x 1152 to 65536 x
// 12288; from the raw factors alone, K2 beats the CUDA-core butterfly from
// 1024 x 3072 up (32.0 against 36.2 us at 4608 x 12288) and ties it below.
int default_variant(const float *factors, const void *K_expanded)
{
    return K_expanded != nullptr ? 3 : (factors != nullptr ? 4 : 2);
}

// The tcgen05 kernel's default wait limit and no skipped tile.
QuantParams hook_params()
{
    QuantParams p{};
    p.wait_limit_ns = kWaitLimitNs;
    p.skip_tile = -1;
    return p;
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI

extern "C" {

kq_status kq_quantize_mxfp4_variant(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                    const float *factors, const void *K_expanded, uint8_t *q,
                                    int64_t ldq, uint8_t *sf, kq_sf_layout sf_layout,
                                    float *y_debug, int variant, cudaStream_t stream)
{
    return quantize_variant(A, m, d, lda, factors, K_expanded, q, ldq, sf, sf_layout, y_debug,
                            variant, hook_params(), stream);
}

kq_status kq_quantize_mxfp4(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                            const float *factors, const void *K_expanded, uint8_t *q, int64_t ldq,
                            uint8_t *sf, kq_sf_layout sf_layout, float *y_debug,
                            cudaStream_t stream)
{
    return quantize_variant(A, m, d, lda, factors, K_expanded, q, ldq, sf, sf_layout, y_debug,
                            default_variant(factors, K_expanded), hook_params(), stream);
}

kq_status kq_quantize_mxfp4_dual(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                 const void *K_expanded, uint8_t *q, int64_t ldq, uint8_t *sf,
                                 kq_sf_layout sf_layout, uint16_t *at, int64_t ldat,
                                 float *y_debug, cudaStream_t stream)
{
    kq_status st = validate_quant_args(A, m, d, lda, q, ldq, sf, sf_layout, y_debug);
    if (st != KQ_OK) return st;
    if (ldat < d || ldat > (1LL << 38)) return KQ_ERR_SHAPE;
    if (m == 0) return KQ_OK;
    if (K_expanded == nullptr || at == nullptr) return KQ_ERR_NULL;
    if (!aligned16(K_expanded) || !aligned16(at) || ldat % 8 != 0) return KQ_ERR_ALIGN;
    QuantParams p;
    fill_quant_params(p, m, d, 128, q, ldq, sf, sf_layout, y_debug);
    return launch_quant_umma(A, lda, K_expanded, p, at, ldat, stream);
}

kq_status kq_test_quantize_stall(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                 const void *K_expanded, uint8_t *q, int64_t ldq, uint8_t *sf,
                                 kq_sf_layout sf_layout, int64_t skip_tile,
                                 uint64_t wait_limit_ns, cudaStream_t stream)
{
    if (wait_limit_ns < 1000000ull || wait_limit_ns > kWaitLimitNs) return KQ_ERR_SHAPE;
    QuantParams p = hook_params();
    p.skip_tile = skip_tile;
    p.wait_limit_ns = wait_limit_ns;
    return quantize_variant(A, m, d, lda, nullptr, K_expanded, q, ldq, sf, sf_layout, nullptr,
                            3, p, stream);
}

kq_status kq_fwht_quantize_mxfp4(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                 uint8_t *q, int64_t ldq, uint8_t *sf, kq_sf_layout sf_layout,
                                 float *y_debug, cudaStream_t stream)
{
    kq_status st = validate_quant_args(A, m, d, lda, q, ldq, sf, sf_layout, y_debug);
    if (st != KQ_OK) return st;
    if (d < 128 || d > 16384 || (d & (d - 1)) != 0) return KQ_ERR_SHAPE;
    if (m == 0) return KQ_OK;
    QuantParams p;
    fill_quant_params(p, m, d, 128, q, ldq, sf, sf_layout, y_debug);
    return launch_quant_fwht(A, lda, p, stream);
}

kq_status kq_w4a4_gemm_variant(const uint8_t *qa, int64_t ldqa, const uint8_t *sfa,
                               const uint8_t *qw, int64_t ldqw, const uint8_t *sfw, int64_t m,
                               int64_t n, int64_t k, float *c, int64_t ldc, int variant,
                               cudaStream_t stream)
{
    if (variant < 0 || variant > 3) return KQ_ERR_LAYOUT;
    if (m < 0 || n < 0 || k <= 0 || k % 32 != 0 || ldqa < k / 2 || ldqw < k / 2 || ldc < n)
        return KQ_ERR_SHAPE;
    // int32 TMA coordinates; row pitches below 2^40 bytes
    if (m > 0x7fffffffLL || n > 0x7fffffffLL || k > 0x7fffffffLL || ldqa > (1LL << 38) ||
        ldqw > (1LL << 38) || ldc > (1LL << 38))
        return KQ_ERR_SHAPE;
    if (m == 0 || n == 0) return KQ_OK;
    if (qa == nullptr || sfa == nullptr || qw == nullptr || sfw == nullptr || c == nullptr)
        return KQ_ERR_NULL;
    if (!aligned16(qa) || !aligned16(qw) || !aligned16(sfa) || !aligned16(sfw) || !aligned16(c) ||
        ldqa % 16 != 0 || ldqw % 16 != 0 || ldc % 4 != 0)
        return KQ_ERR_ALIGN;
    return launch_w4a4_gemm(qa, ldqa, sfa, qw, ldqw, sfw, m, n, k, c, ldc, variant, stream);
}

kq_status kq_w4a4_gemm(const uint8_t *qa, int64_t ldqa, const uint8_t *sfa, const uint8_t *qw,
                       int64_t ldqw, const uint8_t *sfw, int64_t m, int64_t n, int64_t k,
                       float *c, int64_t ldc, cudaStream_t stream)
{
    return kq_w4a4_gemm_variant(qa, ldqa, sfa, qw, ldqw, sfw, m, n, k, c, ldc, 0, stream);
}

kq_status kq_bf16_gemm(const uint16_t *a, int64_t lda, const uint16_t *w, int64_t ldw, int64_t m,
                       int64_t n, int64_t k, float *c, int64_t ldc, cudaStream_t stream)
{
    if (m < 0 || n < 0 || k <= 0 || lda < k || ldw < k || ldc < n) return KQ_ERR_SHAPE;
    if (m > 0x7fffffffLL || n > 0x7fffffffLL || k > 0x7fffffffLL || lda > (1LL << 38) ||
        ldw > (1LL << 38) || ldc > (1LL << 38))
        return KQ_ERR_SHAPE;
    if (m == 0 || n == 0) return KQ_OK;
    if (a == nullptr || w == nullptr || c == nullptr) return KQ_ERR_NULL;
    if (!aligned16(a) || !aligned16(w) || !aligned16(c) || lda % 8 != 0 || ldw % 8 != 0 ||
        ldc % 4 != 0)
        return KQ_ERR_ALIGN;
    return launch_bf16_gemm(a, lda, w, ldw, m, n, k, c, ldc, stream);
}

kq_status kq_layer_error(const float *c, int64_t ldc, const float *c_ref, int64_t ldr, int64_t m,
                         int64_t n, double *out, cudaStream_t stream)
{
    if (m < 0 || n < 0 || ldc < n || ldr < n) return KQ_ERR_SHAPE;
    if (out == nullptr) return KQ_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(out) & 7u) != 0) return KQ_ERR_ALIGN;
    if (m > 0 && n > 0) {
        if (c == nullptr || c_ref == nullptr) return KQ_ERR_NULL;
        if (!aligned16(c) || !aligned16(c_ref) || ldc % 4 != 0 || ldr % 4 != 0)
            return KQ_ERR_ALIGN;
    }
    return launch_layer_error(c, ldc, c_ref, ldr, m, n, out, stream);
}

kq_status kq_quantize_mxfp4_shared(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                   const float *factors, const void *K_expanded, uint8_t *q,
                                   int64_t ldq, uint8_t *sf, kq_sf_layout sf_layout,
                                   float *y_debug, cudaStream_t stream)
{
    kq_status st = validate_quant_args(A, m, d, lda, q, ldq, sf, sf_layout, y_debug);
    if (st != KQ_OK) return st;
    if (m == 0) return KQ_OK;
    if (factors == nullptr && K_expanded == nullptr) return KQ_ERR_NULL;
    if ((factors != nullptr && !aligned16(factors)) || (K_expanded != nullptr && !aligned16(K_expanded)))
        return KQ_ERR_ALIGN;
    DeviceInfo info;
    if ((st = device_info(info)) != KQ_OK) return st;
    QuantParams p;
    fill_quant_params(p, m, d, 128, q, ldq, sf, sf_layout, y_debug);
    p.shared_params = 1;
    p.factors = factors;
    // the records path on the record, else K2 building every block's
    // records from the one factor set
    return launch_quant_umma(A, lda, K_expanded, p, nullptr, 0, stream);
}

kq_status kq_quantize_mxfp4_ex(const uint16_t *A, kq_in_format in_format, int64_t m, int64_t d,
                               int64_t lda, kq_transform transform, const float *param,
                               uint8_t *q, int64_t ldq, uint8_t *sf, kq_sf_layout sf_layout,
                               float *y_debug, cudaStream_t stream)
{
    if (in_format != KQ_IN_BF16 && in_format != KQ_IN_F16) return KQ_ERR_LAYOUT;
    if (transform < KQ_TRANSFORM_KRON || transform > KQ_TRANSFORM_FWHT) return KQ_ERR_LAYOUT;
    kq_status st = validate_quant_args(A, m, d, lda, q, ldq, sf, sf_layout, y_debug);
    if (st != KQ_OK) return st;
    if (transform == KQ_TRANSFORM_FWHT && (d < 128 || d > 16384 || (d & (d - 1)) != 0))
        return KQ_ERR_SHAPE;
    if (m == 0) return KQ_OK;
    const bool needs_param = transform == KQ_TRANSFORM_KRON || transform == KQ_TRANSFORM_DIAG;
    if (needs_param && param == nullptr) return KQ_ERR_NULL;
    if (needs_param && !aligned16(param)) return KQ_ERR_ALIGN;
    DeviceInfo info;
    if ((st = device_info(info)) != KQ_OK) return st;
    QuantParams p;
    fill_quant_params(p, m, d, 128, q, ldq, sf, sf_layout, y_debug);
    p.in_f16 = in_format == KQ_IN_F16 ? 1 : 0;
    switch (transform) {
    case KQ_TRANSFORM_KRON: p.factors = param; return launch_quant_tma(kKron, A, lda, p, stream);
    case KQ_TRANSFORM_DIAG: p.s = param; return launch_quant_tma(kDiag, A, lda, p, stream);
    case KQ_TRANSFORM_HADAMARD: return launch_quant_tma(kHadamard, A, lda, p, stream);
    case KQ_TRANSFORM_IDENTITY: return launch_quant_tma(kIdentity, A, lda, p, stream);
    default: return launch_quant_fwht(A, lda, p, stream);
    }
}

kq_status kq_smooth_quantize_mxfp4(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                   const float *s, uint8_t *q, int64_t ldq, uint8_t *sf,
                                   kq_sf_layout sf_layout, float *y_debug, cudaStream_t stream)
{
    kq_status st = validate_quant_args(A, m, d, lda, q, ldq, sf, sf_layout, y_debug);
    if (st != KQ_OK) return st;
    if (m == 0) return KQ_OK;
    if (s == nullptr) return KQ_ERR_NULL;
    if (!aligned16(s)) return KQ_ERR_ALIGN;
    DeviceInfo info;
    if ((st = device_info(info)) != KQ_OK) return st;
    QuantParams p;
    fill_quant_params(p, m, d, 128, q, ldq, sf, sf_layout, y_debug);
    p.s = s;
    return launch_quant_tma(kDiag, A, lda, p, stream);
}

kq_status kq_hadamard_quantize_mxfp4(const uint16_t *A, int64_t m, int64_t d, int64_t lda,
                                     uint8_t *q, int64_t ldq, uint8_t *sf, kq_sf_layout sf_layout,
                                     float *y_debug, cudaStream_t stream)
{
    kq_status st = validate_quant_args(A, m, d, lda, q, ldq, sf, sf_layout, y_debug);
    if (st != KQ_OK) return st;
    if (m == 0) return KQ_OK;
    DeviceInfo info;
    if ((st = device_info(info)) != KQ_OK) return st;
    QuantParams p;
    fill_quant_params(p, m, d, 128, q, ldq, sf, sf_layout, y_debug);
    return launch_quant_tma(kHadamard, A, lda, p, stream);
}

kq_status kq_dequantize(const uint8_t *q, int64_t ldq, const uint8_t *sf, kq_sf_layout sf_layout,
                        int64_t m, int64_t d, float *out, cudaStream_t stream)
{
    if (m < 0 || d <= 0 || d % 32 != 0 || ldq < d / 2) return KQ_ERR_SHAPE;
    if (sf_layout != KQ_SF_ROWMAJOR && sf_layout != KQ_SF_BLOCKED_128x4) return KQ_ERR_LAYOUT;
    if (m == 0) return KQ_OK;
    if (q == nullptr || sf == nullptr || out == nullptr) return KQ_ERR_NULL;
    if (!aligned16(q) || !aligned16(out) || ldq % 16 != 0) return KQ_ERR_ALIGN;
    DeviceInfo info;
    kq_status st = device_info(info);
    if (st != KQ_OK) return st;
    const int64_t work = m * (d / 32);
    dequant_kernel<<<grid_for(work, 256), 256, 0, stream>>>(q, ldq, sf, static_cast<int>(sf_layout),
                                                            m, d / 32, out);
    return check_launch();
}

kq_status kq_expand_blocks(const float *factors, int64_t nb, kq_kfmt fmt, void *K_out,
                           cudaStream_t stream)
{
    if (nb <= 0) return KQ_ERR_SHAPE;
    if (fmt != KQ_K_FP32 && fmt != KQ_K_BF16X3) return KQ_ERR_LAYOUT;
    if (factors == nullptr || K_out == nullptr) return KQ_ERR_NULL;
    if (!aligned16(factors) || !aligned16(K_out)) return KQ_ERR_ALIGN;
    DeviceInfo info;
    kq_status st = device_info(info);
    if (st != KQ_OK) return st;
    if (fmt == KQ_K_BF16X3) return launch_umma_records(factors, nb, K_out, stream);
    expand_kernel<<<grid_for(nb * 1024, 256), 256, 0, stream>>>(factors, nb, K_out);
    return check_launch();
}

kq_status kq_test_encode_e2m1(uint32_t first, int64_t count, uint8_t *out, cudaStream_t stream)
{
    if (count < 0 || count % 8 != 0 || static_cast<uint64_t>(first) + count > (1ULL << 32))
        return KQ_ERR_SHAPE;
    if (count == 0) return KQ_OK;
    if (out == nullptr) return KQ_ERR_NULL;
    if (!aligned16(out)) return KQ_ERR_ALIGN;
    DeviceInfo info;
    kq_status st = device_info(info);
    if (st != KQ_OK) return st;
    encode_sweep_kernel<<<grid_for(count / 8, 256), 256, 0, stream>>>(
        first, count / 8, reinterpret_cast<uint32_t *>(out));
    return check_launch();
}

}  // extern "C"
