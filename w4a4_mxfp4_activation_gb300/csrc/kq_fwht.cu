// Full-row Walsh-Hadamard baseline with the fused MXFP4 quantizer, sm_103a.
//
// "KroQuant: Kronecker-Structured Block Transforms for Efficient Post-
// Training Quantization of Diffusion Transformers", Sec. 4.4 and Table 3:
// the FWHT baseline transforms every row by the normalised d-point
// Walsh-Hadamard matrix, y = a . H_d / sqrt(d) with H_d[r][c] =
// (-1)^popcount(r & c) (Sylvester order, d a power of two), and quantizes y
// to MXFP4 like the other kernels.  Unlike the block-diagonal transforms it
// couples every channel of a row with every other, so a row must be complete
// on chip before any output block is known.
//
// Layout of the work: a persistent CTA of 512 threads (two per SM)
// transforms 16384 elements per iteration (16384 / d rows).  Bit b of an
// element's index within the iteration is bit b of its channel for b < log2 d
// and a row bit above; the butterfly stages of H_d act on one channel bit
// each and commute, so they run in three register phases, 32 values per
// thread, joined by two exchanges through a shared fp32 buffer (padded to 36
// floats per 32, so every access pattern below is free of bank conflicts):
//   A. channel bits 0 and 10..13: the thread reads 16 adjacent bf16 (or fp16)
//      pairs 1024 elements apart from the staging tile (the iteration's rows,
//      copied in natural order by 16-byte cp.async during the previous
//      iteration), applies those stages and stores the 16 pairs;
//   B. bits 5..9: 32 values 32 apart (a warp reads 32 consecutive floats);
//   C. bits 1..4, then the quantizer: the thread's own 32-channel block, read
//      as 8 float4; it scales by 1/sqrt(d), quantizes and stores 16 bytes of
//      codes and one scale byte.
// Values travel as fp32 pairs, so every stage whose partner is not the other
// half of a pair is one packed fp32x2 add and one packed fused multiply-add
// (x + y, x - y) for two butterflies.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int kFThreads = 512;
constexpr int kFElems = 16384;                       // elements per iteration
constexpr int kFSmemFloats = kFElems + kFElems / 8;  // padded: 36 floats per 32
// 16-bit staging of the next iteration's rows, natural order: element e of
// the iteration (row_local * d + channel) at byte 2 e
constexpr int kFStageOff = kFSmemFloats * 4;
constexpr int kFSmemBytes = kFStageOff + kFElems * 2;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ int pad(int e) { return e + 4 * (e >> 5); }

// Butterflies (x, y) -> (x + y, x - y) on two pairs at once.
__device__ __forceinline__ void bfly2(float2 &a, float2 &b)
{
    const float2 x = a;
    a = __fadd2_rn(x, b);
    b = __ffma2_rn(b, make_float2(-1.0f, -1.0f), x);
}

// Butterfly stages on the pair-index bits h = 1, 2, 4, ... < N of v[0..N)
// that are set in `mask` (a compile-time constant at every call).
template <int N>
__device__ __forceinline__ void bfly_stages(float2 *v, int mask)
{
#pragma unroll
    for (int h = 1; h < N; h *= 2)
        if (mask & h)
#pragma unroll
            for (int k = 0; k < N; ++k)
                if ((k & h) == 0) bfly2(v[k], v[k + h]);
}

template <int LOGD, bool DEBUG>
__global__ void __launch_bounds__(kFThreads, 2) fwht_quant_kernel(const uint16_t *A, int64_t lda,
                                                                  const QuantParams p)
{
    constexpr int D = 1 << LOGD;
    constexpr int kRows = kFElems / D;               // rows per iteration
    constexpr int kChunksPerRow = D / 8;             // 16-byte chunks of a 16-bit row
    // which of the phase's index bits are channel bits (stages to apply):
    // A: pair index k bit i = channel bit 10 + i; B: bit i = channel bit 5 + i
    constexpr int kMaskA = LOGD >= 14 ? 15 : (LOGD > 10 ? (1 << (LOGD - 10)) - 1 : 0);
    constexpr int kMaskB = LOGD >= 10 ? 31 : (1 << (LOGD - 5)) - 1;
    extern __shared__ __align__(16) float fbuf[];
    const uint8_t *stg = reinterpret_cast<const uint8_t *>(fbuf) + kFStageOff;
    grid_dependency_wait();
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const bool f16 = p.in_f16 != 0;
    const float inv = 1.0f / sqrtf(static_cast<float>(D));   // exact when d = 4^k
    const int64_t groups = (p.m_rows + kRows - 1) / kRows;
    const uint32_t stg_s = smem_addr(stg);
    // copies of the rows of iteration g: chunk c = t + 512 i of the staging
    // tile (row c / kChunksPerRow, channels 8 (c % kChunksPerRow) ..); rows
    // past m are zero
    auto issue = [&](int64_t g) {
        if (g < groups) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = t + kFThreads * i;
                const int64_t r = g * kRows + c / kChunksPerRow;
                const uint32_t dst = stg_s + 16 * c;
                if (r < p.m)
                    cp_async16(dst, A + r * lda + 8 * (c % kChunksPerRow));
                else
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
            }
        }
        cp_async_commit();
    };
    const int ea = 2 * lane + 64 * warp;             // phase A: elements ea + 1024 k (+ 0, 1)
    const int eb = lane + 1024 * warp;               // phase B: elements eb + 32 j
    const int ec = 32 * t;                           // phase C: elements ec .. ec + 31
    const int64_t row_c = ec >> LOGD;                // row of the thread's block in the tile
    const int b = (ec & (D - 1)) >> 5;               // the block
    issue(blockIdx.x);
    for (int64_t grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        cp_async_wait_all();
        __syncthreads();   // the tile has landed; the last iteration's phase C is done with fbuf
        // ---- phase A: channel bits 0, 10..13
        {
            const uint32_t *st32 = reinterpret_cast<const uint32_t *>(stg);
            float2 v[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint32_t w = st32[(ea + 1024 * k) >> 1];
                v[k] = f16 ? make_float2(f16_lo(w), f16_hi(w)) : make_float2(bf16_lo(w), bf16_hi(w));
                v[k] = make_float2(v[k].x + v[k].y, v[k].x - v[k].y);          // bit 0
            }
            bfly_stages<16>(v, kMaskA);
#pragma unroll
            for (int k = 0; k < 16; ++k)
                *reinterpret_cast<float2 *>(fbuf + pad(ea + 1024 * k)) = v[k];
        }
        __syncthreads();   // phase A's values are in fbuf; the staging tile is free
        issue(grp + gridDim.x);                      // next tile in flight during B and C
        // ---- phase B: channel bits 5..9 (pairs j, j + 16: bit 9 inside a pair)
        {
            float2 v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = make_float2(fbuf[pad(eb + 32 * j)], fbuf[pad(eb + 32 * (j + 16))]);
            bfly_stages<16>(v, kMaskB & 15);
            if (kMaskB & 16) {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = make_float2(v[j].x + v[j].y, v[j].x - v[j].y);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                fbuf[pad(eb + 32 * j)] = v[j].x;
                fbuf[pad(eb + 32 * (j + 16))] = v[j].y;
            }
        }
        __syncthreads();   // phase B's values are in fbuf
        // ---- phase C: channel bits 1..4 of the thread's block, then quantize
        float2 Y[16];
        {
            const float4 *own4 = reinterpret_cast<const float4 *>(fbuf + pad(ec));
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 w = own4[k];
                Y[2 * k] = make_float2(w.x, w.y);
                Y[2 * k + 1] = make_float2(w.z, w.w);
            }
            bfly_stages<16>(Y, 15);
#pragma unroll
            for (int k = 0; k < 16; ++k) Y[k] = __fmul2_rn(Y[k], make_float2(inv, inv));
        }
        const int64_t row = grp * kRows + row_c;
        if (row < p.m_rows) {
            if (DEBUG && row < p.m) {
                float *yd = p.y_debug + row * p.d + b * 32;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    stg_f4(yd + 4 * k, make_float4(Y[2 * k].x, Y[2 * k].y, Y[2 * k + 1].x,
                                                   Y[2 * k + 1].y));
            }
            uint32_t byte;
            const uint4 codes = quantize_block(Y, byte);
            if (row < p.m) stg128_cs(p.q + row * p.ldq + b * 16, codes);
            if (p.sf_layout == KQ_SF_ROWMAJOR) {
                if (row < p.m) p.sf[row * p.nb + b] = static_cast<uint8_t>(byte);
            } else {
                p.sf[sf_blocked_offset(row, b, p.ncb)] = static_cast<uint8_t>(byte);
            }
        }
    }
    cp_async_wait_all();
}

struct FSlot {
    std::once_flag once[64];
    int occupancy[64] = {};
    cudaError_t err[64] = {};
};

template <int LOGD, bool DEBUG>
kq_status launch_fwht_t(const uint16_t *A, int64_t lda, const QuantParams &p, int sm_count,
                        cudaStream_t stream)
{
    auto kern = fwht_quant_kernel<LOGD, DEBUG>;
    static FSlot slot;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KQ_ERR_CUDA;
    std::call_once(slot.once[dev], [&] {
        slot.err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kFSmemBytes);
        if (slot.err[dev] == cudaSuccess)
            slot.err[dev] = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &slot.occupancy[dev], kern, kFThreads, kFSmemBytes);
    });
    if (slot.err[dev] != cudaSuccess || slot.occupancy[dev] < 1) return KQ_ERR_CUDA;
    constexpr int kRows = kFElems >> LOGD;
    const int64_t groups = (p.m_rows + kRows - 1) / kRows;
    if (groups == 0) return KQ_OK;
    const int grid = static_cast<int>(
        std::min<int64_t>(groups, static_cast<int64_t>(slot.occupancy[dev]) * sm_count));
    return launch_pdl(kern, grid, kFThreads, static_cast<size_t>(kFSmemBytes), stream, A, lda, p);
}

template <bool DEBUG>
kq_status launch_fwht_d(const uint16_t *A, int64_t lda, const QuantParams &p, int sm_count,
                        cudaStream_t stream)
{
    switch (p.d) {
    case 128: return launch_fwht_t<7, DEBUG>(A, lda, p, sm_count, stream);
    case 256: return launch_fwht_t<8, DEBUG>(A, lda, p, sm_count, stream);
    case 512: return launch_fwht_t<9, DEBUG>(A, lda, p, sm_count, stream);
    case 1024: return launch_fwht_t<10, DEBUG>(A, lda, p, sm_count, stream);
    case 2048: return launch_fwht_t<11, DEBUG>(A, lda, p, sm_count, stream);
    case 4096: return launch_fwht_t<12, DEBUG>(A, lda, p, sm_count, stream);
    case 8192: return launch_fwht_t<13, DEBUG>(A, lda, p, sm_count, stream);
    case 16384: return launch_fwht_t<14, DEBUG>(A, lda, p, sm_count, stream);
    default: return KQ_ERR_SHAPE;
    }
}

}  // namespace

kq_status launch_quant_fwht(const uint16_t *A, int64_t lda, const QuantParams &p,
                            cudaStream_t stream)
{
    DeviceInfo info;
    kq_status st = device_info(info);
    if (st != KQ_OK) return st;
    if (p.y_debug != nullptr) return launch_fwht_d<true>(A, lda, p, info.sm_count, stream);
    return launch_fwht_d<false>(A, lda, p, info.sm_count, stream);
}

}  // namespace kq
