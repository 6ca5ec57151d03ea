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
// Layout of the work: a persistent CTA of 512 threads transforms 16384
// elements per iteration (16384 / d rows).  The butterfly stages of H_d act on
// one bit of the channel index each and commute, so they run in the order
// that keeps shared-memory traffic lowest:
//   1. the iteration's rows arrive by 16-byte cp.async copies into a bf16
//      staging tile in natural order (consecutive threads, consecutive
//      chunks), issued during the previous iteration;
//   2. the stages with pairs 32 apart and more run as passes: a thread
//      gathers r values at the pass's stride (lanes at consecutive channels,
//      so every access is conflict-free), applies log2(r) stages in registers
//      and writes them to a shared fp32 buffer padded to 36 floats per 32 --
//      the first pass reads the bf16 staging tile, a second one (d > 1024)
//      the fp32 buffer;
//   3. each thread then reads one 32-channel block of a row, applies the five
//      stages with pairs 1..16 apart in registers, multiplies by 1/sqrt(d),
//      quantizes and stores 16 bytes of codes and one scale byte.
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
// bf16 staging of the next iteration's rows, natural order: element e of the
// iteration (row_local * d + channel) at byte 2 e
constexpr int kFStageOff = kFSmemFloats * 4;
constexpr int kFSmemBytes = kFStageOff + kFElems * 2;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ int pad(int e) { return e + 4 * (e >> 5); }

// In-place unnormalised Walsh-Hadamard transform of n = 2^k values (Sylvester
// order): butterflies (x, y) -> (x + y, x - y) over pairs h = 1, 2, ..., n/2 apart.
template <int N>
__device__ __forceinline__ void wht_regs(float (&v)[32])
{
#pragma unroll
    for (int h = 1; h < N; h *= 2)
#pragma unroll
        for (int j = 0; j < N; ++j)
            if ((j & h) == 0) {
                const float x = v[j], z = v[j + h];
                v[j] = x + z;
                v[j + h] = x - z;
            }
}

// One pass over the stages with pairs S, 2S, ..., (R/2)S apart: groups of R
// values at stride S; group g of a row = (lo, hi) with lo = g % S (the lanes
// of a warp take consecutive lo, i.e. consecutive channels) and base
// lo + hi * S * R.  FROM_STAGING: the values come from the 16-bit staging
// tile (bf16, or fp16 when f16); they always go to the padded fp32 buffer.
template <int D, int S, int R, bool FROM_STAGING>
__device__ __forceinline__ void wht_pass(float *buf, const uint16_t *stg, int row_local, int tr,
                                         bool f16)
{
    static_assert(S % 32 == 0, "pass strides are multiples of 32");
    constexpr int kThreadsPerRow = D / 32;
    constexpr int kGroupsPerThread = (D / R) / kThreadsPerRow;
    static_assert(kGroupsPerThread >= 1, "every thread takes at least one group");
#pragma unroll 1
    for (int q = 0; q < kGroupsPerThread; ++q) {
        const int g = tr + q * kThreadsPerRow;
        const int e0 = row_local * D + (g % S) + (g / S) * S * R;
        // S is a multiple of 32, so the padded index of e0 + k S is
        // pad(e0) + k (S + S / 8)
        float *pb = buf + pad(e0);
        float v[32];
        if constexpr (FROM_STAGING) {
            const uint16_t *sb = stg + e0;
            if (f16) {
#pragma unroll
                for (int k = 0; k < R; ++k) v[k] = __half2float(__ushort_as_half(sb[k * S]));
            } else {
#pragma unroll
                for (int k = 0; k < R; ++k) v[k] = __uint_as_float(static_cast<uint32_t>(sb[k * S]) << 16);
            }
        } else {
#pragma unroll
            for (int k = 0; k < R; ++k) v[k] = pb[k * (S + S / 8)];
        }
        wht_regs<R>(v);
#pragma unroll
        for (int k = 0; k < R; ++k) pb[k * (S + S / 8)] = v[k];
    }
}

template <int LOGD, bool DEBUG>
__global__ void __launch_bounds__(kFThreads, 2) fwht_quant_kernel(const uint16_t *A, int64_t lda,
                                                                  const QuantParams p)
{
    constexpr int D = 1 << LOGD;
    constexpr int kRows = kFElems / D;               // rows per iteration
    constexpr int kThreadsPerRow = D / 32;
    constexpr int kChunksPerRow = D / 8;             // 16-byte chunks of a bf16 row
    extern __shared__ float fbuf[];
    uint16_t *stg = reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(fbuf) + kFStageOff);
    grid_dependency_wait();
    const int t = threadIdx.x;
    const int row_local = t / kThreadsPerRow, tr = t % kThreadsPerRow;
    const int b = tr;                                // the thread's 32-channel block in step 3
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
    issue(blockIdx.x);
    for (int64_t grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        const int64_t row = grp * kRows + row_local;
        cp_async_wait_all();
        __syncthreads();                             // every chunk of the tile has landed
        // stages with pairs 32 apart and more: the first pass reads the staging tile
        if constexpr (LOGD > 10) {
            wht_pass<D, 1024, (1 << (LOGD - 10)), true>(fbuf, stg, row_local, tr, f16);   // 1024..8192
            __syncthreads();
            issue(grp + gridDim.x);                  // staging consumed: next tile in flight
            wht_pass<D, 32, 32, false>(fbuf, stg, row_local, tr, f16);                    // 32..512
        } else {
            wht_pass<D, 32, (1 << (LOGD - 5)), true>(fbuf, stg, row_local, tr, f16);
            __syncthreads();
            issue(grp + gridDim.x);
        }
        __syncthreads();
        // the thread's own block: stages with pairs 1..16 apart, then quantize
        const int own = pad(row_local * D + b * 32);   // a multiple of 36: 16-byte aligned
        const float4 *own4 = reinterpret_cast<const float4 *>(fbuf + own);
        float v[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 w = own4[k];
            v[4 * k] = w.x;
            v[4 * k + 1] = w.y;
            v[4 * k + 2] = w.z;
            v[4 * k + 3] = w.w;
        }
        wht_regs<32>(v);
        float2 Y[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) Y[k] = make_float2(v[2 * k] * inv, v[2 * k + 1] * inv);
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
        __syncthreads();                             // the buffer is reused next iteration
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
