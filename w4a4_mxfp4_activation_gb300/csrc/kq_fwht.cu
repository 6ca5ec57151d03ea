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
// elements per iteration (16384 / d rows).  Thread t owns one 32-channel
// block of one row:
//   1. it takes the block from a shared staging area, where four 16-byte
//      cp.async copies brought it during the previous iteration's passes,
//      issues the copies for its block of the next iteration, runs the first
//      five butterfly stages (pairs 1..16 apart) in registers and writes the
//      32 values to a shared fp32 buffer padded to 36 floats per 32 (so that
//      a thread's own block moves in 16-byte vectors and both those and 32
//      lanes' strided scalar accesses are free of bank conflicts);
//   2. the stages with pairs 32..512 apart, then 1024..8192 apart, each run as
//      one pass: a thread gathers r values at the stage's stride into
//      registers, applies log2(r) stages, writes them back (r = 32, or less
//      in the last pass);
//   3. it reads its block back, multiplies by 1/sqrt(d), quantizes and
//      stores 16 bytes of codes and one scale byte.
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
// staging for the next iteration's bf16 input: chunk k (16 bytes) of thread t
// at k * 8 KB + 16 t, so that a warp's accesses are contiguous
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
// of a warp take consecutive lo) and base lo + hi * S * R.
template <int D, int S, int R>
__device__ __forceinline__ void wht_pass(float *buf, int row_local, int tr)
{
    static_assert(S % 32 == 0, "pass strides are multiples of 32");
    constexpr int kThreadsPerRow = D / 32;
    constexpr int kGroupsPerThread = 32 / R;
#pragma unroll 1
    for (int q = 0; q < kGroupsPerThread; ++q) {
        const int g = tr + q * kThreadsPerRow;
        // S is a multiple of 32, so the padded index of base + k S is
        // pad(base) + k (S + S / 8): one register and immediate offsets
        float *pb = buf + pad(row_local * D + (g % S) + (g / S) * S * R);
        float v[32];
#pragma unroll
        for (int k = 0; k < R; ++k) v[k] = pb[k * (S + S / 8)];
        wht_regs<R>(v);
#pragma unroll
        for (int k = 0; k < R; ++k) pb[k * (S + S / 8)] = v[k];
    }
}

template <int LOGD, bool DEBUG>
__global__ void __launch_bounds__(kFThreads, 2) fwht_quant_kernel(const uint16_t *__restrict__ A,
                                                                  int64_t lda, const QuantParams p)
{
    constexpr int D = 1 << LOGD;
    constexpr int kRows = kFElems / D;               // rows per iteration
    constexpr int kThreadsPerRow = D / 32;
    extern __shared__ float fbuf[];
    grid_dependency_wait();
    const int t = threadIdx.x;
    const int row_local = t / kThreadsPerRow, tr = t % kThreadsPerRow;
    const int b = tr;                                // the thread's 32-channel block
    const float inv = 1.0f / sqrtf(static_cast<float>(D));   // exact when d = 4^k
    const int64_t groups = (p.m_rows + kRows - 1) / kRows;
    const uint32_t stage = smem_addr(fbuf) + kFStageOff + 16 * t;
    // copies of this thread's block of rows group g into its staging chunks
    auto issue = [&](int64_t g) {
        const int64_t r = g * kRows + row_local;
        if (g < groups && r < p.m) {
            const uint16_t *src = A + r * lda + b * 32;
#pragma unroll
            for (int k = 0; k < 4; ++k) cp_async16(stage + k * 8192, src + 8 * k);
        }
        cp_async_commit();
    };
    issue(blockIdx.x);
    for (int64_t grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        const int64_t row = grp * kRows + row_local;
        float v[32];
        cp_async_wait_all();
        if (row < p.m) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 w = lds128(stage + k * 8192);
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[8 * k + 2 * e] = p.in_f16 ? f16_lo(u[e]) : bf16_lo(u[e]);
                    v[8 * k + 2 * e + 1] = p.in_f16 ? f16_hi(u[e]) : bf16_hi(u[e]);
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = 0.f;
        }
        issue(grp + gridDim.x);                      // in flight during the passes below
        wht_regs<32>(v);                             // pairs 1..16 apart
        const int own = pad(row_local * D + b * 32);   // a multiple of 36: 16-byte aligned
        float4 *own4 = reinterpret_cast<float4 *>(fbuf + own);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            own4[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        __syncthreads();
        if constexpr (LOGD > 5) {                    // pairs 32..512 apart
            constexpr int R1 = (LOGD - 5 >= 5) ? 32 : (1 << (LOGD - 5));
            wht_pass<D, 32, R1>(fbuf, row_local, tr);
            __syncthreads();
        }
        if constexpr (LOGD > 10) {                   // pairs 1024..8192 apart
            wht_pass<D, 1024, (1 << (LOGD - 10))>(fbuf, row_local, tr);
            __syncthreads();
        }
        float2 Y[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 w = own4[k];
            Y[2 * k] = make_float2(w.x * inv, w.y * inv);
            Y[2 * k + 1] = make_float2(w.z * inv, w.w * inv);
        }
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
