// Consumer of the quantizer's output: the W4A4 product of eq. (11) on the
// 5th-generation tensor cores, sm_103a, and the pieces of the layer error of
// eq. (2).
//
// "KroQuant: Kronecker-Structured Block Transforms for Efficient Post-
// Training Quantization of Diffusion Transformers", eq. (11) multiplies the
// MXFP4-quantized transformed activations by the MXFP4-quantized transformed
// weights, and eq. (2) measures the layer's error through that product:
//     C[i][n] = sum_k deq(A)[i][k] * deq(W)[n][k]
// from packed E2M1 codes ([rows][d/2] bytes, code 2k in the low nibble) and
// E8M0 scales in the 128x4 tiled layout of block-scaled MMA -- exactly the
// bytes kq_quantize_mxfp4 writes.  Three kernels:
//   w4a4_mxf4_kernel<NH, true>   the product on the FP4 tensor cores
//                                (tcgen05.mma kind::mxf4, block-scaled): the
//                                library's W4A4 GEMM;
//   w4a4_mxf4_kernel<NH, false>  the same structure on bf16 A and W (kind::f16):
//                                the unquantized reference product A W^T;
//   w4a4_gemm_kernel             a checking route for the W4A4 product: every
//                                operand tile dequantized to bf16 in shared
//                                memory (exact: an MXFP4 element times its
//                                power-of-two scale has at most two significant
//                                bits) and multiplied with kind::f16;
// and the fp64 error sums.  Every wait is bounded in time; a CTA that times
// out stops and leaves its remaining tiles unwritten, and the call reports
// nothing (results are then undefined), as for the quantizers.
//
// The checking kernel (persistent over 128 x 128 output tiles; K in steps of
// 64): warp 0 loads per K step the code tiles of A and W (TMA, 128 rows x 32
// bytes each) and their 512-byte scale tiles (bulk copies) into a 4-deep
// ring; warp 1 issues four M = 128, N = 128, K = 16 MMAs per K step into one
// of two TMEM accumulators; warps 2-5 dequantize (thread r turns row r of
// both code tiles into bf16 rows of the 128B-swizzled, double-buffered
// operand buffers); warps 6-9 read the accumulator back and store fp32 rows.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int kGBM = 128, kGBN = 128, kGBK = 64;
constexpr int kGThreads = 320;
constexpr int kGStages = 4;                   // code ring
constexpr int kGCodeBytes = 128 * 32;         // one operand's code tile per K step
constexpr int kGSfBytes = 512;                // one 128x4 scale tile
constexpr int kGStageBytes = 2 * kGCodeBytes + 2 * kGSfBytes;   // 9 KB
constexpr int kGOpBytes = kGBM * 128;         // 128 rows x 64 bf16 (one operand)
constexpr int kGOpOff = 0;                    // 2 buffers x (A, W): 64 KB, 1 KB aligned
constexpr int kGRingOff = 4 * kGOpBytes;
constexpr int kGBarOff = kGRingOff + kGStages * kGStageBytes;
constexpr int kGSmemBytes = kGBarOff + 1024 + 1024;
constexpr uint32_t kGTmemCols = 256;

__device__ __forceinline__ void g_tmem_alloc(uint32_t slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void g_tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void g_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void g_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ uint64_t g_desc(uint32_t saddr)
{
    // K-major, 128B swizzle: LBO 16 B (unused), SBO 1024 B (8 rows x 128 B)
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(16 >> 4) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f16: fp32 D, bf16 A and B, both K-major, N = 128, M = 128.
constexpr uint32_t kGIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) |
                             ((128u >> 4) << 24);

__device__ __forceinline__ void g_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(kGIdesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void g_mma_id(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void g_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void g_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// E2M1 code (bits 0-2 magnitude, bit 3 sign) times 2^(byte - 127), as fp32:
// exact (at most two significant bits; 2^-127 and below are fp32 subnormals).
__device__ __forceinline__ float e2m1_scaled(uint32_t code, float scale)
{
    const uint32_t mag = code & 7u;
    // magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 as fp32 bit patterns
    const uint32_t e = mag >> 1, half = mag & 1u;
    const uint32_t bits = mag < 2 ? (mag == 1 ? 0x3F000000u : 0u)
                                  : ((126u + e) << 23) | (half << 22);
    const float v = __uint_as_float(bits | ((code & 8u) << 28));
    return v * scale;
}

// 2^(byte - 127) as fp32 (byte 0: the subnormal 2^-127); byte 255 is the
// E8M0 NaN of the OCP MX format.
__device__ __forceinline__ float e8m0_value(uint32_t byte)
{
    return __uint_as_float(byte == 255u ? 0x7FC00000u : (byte ? byte << 23 : 0x00400000u));
}

struct GemmArgs {
    int64_t m, n, k;              // C is m x n, the contraction runs over k
    int64_t nb;                   // k / 32 scale blocks per row
    int64_t ncb;                  // ceil(nb / 4): 128x4 scale tiles per row band
    const uint8_t *sfa, *sfw;     // tiled scales (MXFP4 mode)
    float *c;
    int64_t ldc;
    int64_t mtiles, ntiles, ksteps;
};

__global__ void __launch_bounds__(kGThreads, 1)
    w4a4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                     const GemmArgs g)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    const uint32_t bar = base + kGBarOff;
    const uint32_t code_full = bar, code_empty = bar + 8 * kGStages;
    const uint32_t op_full = bar + 16 * kGStages, op_free = op_full + 16;
    const uint32_t acc_full = op_free + 16, acc_empty = acc_full + 16;
    const uint32_t tmem_slot = acc_empty + 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles = g.mtiles * g.ntiles;

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmW);
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(code_full + 8 * s, 1);
            mbar_init(code_empty + 8 * s, 128);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(op_full + 8 * b, 128);               // the dequantization threads
            mbar_init(op_free + 8 * b, 1);                 // MMA commit
            mbar_init(acc_full + 8 * b, 1);
            mbar_init(acc_empty + 8 * b, 128);
        }
        mbar_fence_init();
    }
    if (warp == 1) g_tmem_alloc(tmem_slot, kGTmemCols);
    g_fence_before();
    __syncthreads();
    g_fence_after();
    uint32_t tmem_base;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(tmem_base) : "r"(tmem_slot) : "memory");
    grid_dependency_wait();

    if (warp == 0) {
        if (lane == 0) {
            int64_t kk = 0;       // global K-step counter of this CTA
            bool ok = true;
            for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int64_t mt = t / g.ntiles, nt = t % g.ntiles;
                for (int64_t ks = 0; ks < g.ksteps && ok; ++ks, ++kk) {
                    const int s = static_cast<int>(kk % kGStages);
                    if (kk >= kGStages &&
                        !mbar_wait(code_empty + 8 * s, static_cast<uint32_t>(((kk / kGStages) - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = base + kGRingOff + s * kGStageBytes;
                    mbar_arrive_expect_tx(code_full + 8 * s, kGStageBytes);
                    tma_load_2d(st, &tmA, static_cast<int32_t>(ks * 32),
                                static_cast<int32_t>(mt * kGBM), code_full + 8 * s, 0);
                    tma_load_2d(st + kGCodeBytes, &tmW, static_cast<int32_t>(ks * 32),
                                static_cast<int32_t>(nt * kGBN), code_full + 8 * s, 0);
                    // the 128x4 scale tile holding this K step's two blocks
                    bulk_load(st + 2 * kGCodeBytes, g.sfa + (mt * g.ncb + ks / 2) * 512, 512,
                              code_full + 8 * s);
                    bulk_load(st + 2 * kGCodeBytes + kGSfBytes, g.sfw + (nt * g.ncb + ks / 2) * 512,
                              512, code_full + 8 * s);
                }
            }
            // the last copies issued into each buffer have landed before the
            // CTA may exit (they have, unless a wait above gave up)
            for (int64_t j = kk - 1; j >= 0 && j >= kk - kGStages; --j)
                (void)mbar_wait(code_full + 8 * static_cast<int>(j % kGStages),
                                static_cast<uint32_t>((j / kGStages) & 1));
        }
    } else if (warp == 1) {
        int64_t kk = 0, tc = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++tc) {
            const int a = static_cast<int>(tc & 1);
            if (tc >= 2)
                ok = __all_sync(0xffffffffu,
                                mbar_wait(acc_empty + 8 * a, static_cast<uint32_t>(((tc >> 1) - 1) & 1)));
            for (int64_t ks = 0; ks < g.ksteps && ok; ++ks, ++kk) {
                const int b = static_cast<int>(kk & 1);
                ok = __all_sync(0xffffffffu,
                                mbar_wait(op_full + 8 * b, static_cast<uint32_t>((kk >> 1) & 1)));
                if (!ok) break;
                g_fence_after();
                if (lane == 0) {
                    const uint32_t opa = base + kGOpOff + b * 2 * kGOpBytes;
                    for (int k = 0; k < 4; ++k)
                        g_mma(tmem_base + a * 128, g_desc(opa + 32 * k), g_desc(opa + kGOpBytes + 32 * k),
                              (ks > 0 || k > 0) ? 1u : 0u);
                    g_commit(op_free + 8 * b);
                    if (ks == g.ksteps - 1) g_commit(acc_full + 8 * a);
                }
                __syncwarp();
            }
        }
        if (tc >= 1 && ok)
            (void)mbar_wait(acc_full + 8 * static_cast<int>((tc - 1) & 1),
                            static_cast<uint32_t>(((tc - 1) >> 1) & 1));
    } else if (warp < 6) {
        {
            // dequantization: thread r owns row r of both code tiles
            const int r = threadIdx.x - 64;
            int64_t kk = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                for (int64_t ks = 0; ks < g.ksteps; ++ks, ++kk) {
                    const int s = static_cast<int>(kk % kGStages), b = static_cast<int>(kk & 1);
                    ok = mbar_wait(code_full + 8 * s, static_cast<uint32_t>((kk / kGStages) & 1));
                    if (ok && kk >= 2)
                        ok = mbar_wait(op_free + 8 * b, static_cast<uint32_t>(((kk >> 1) - 1) & 1));
                    if (!ok) break;
                    const uint32_t st = base + kGRingOff + s * kGStageBytes;
                    const uint32_t opa = base + kGOpOff + b * 2 * kGOpBytes;
                    // scale bytes of row r, blocks 2 ks and 2 ks + 1 (adjacent in the tile)
                    const int sfo = (r & 31) * 16 + (r >> 5) * 4 + static_cast<int>((ks & 1) * 2);
#pragma unroll
                    for (int op = 0; op < 2; ++op) {
                        const uint32_t codes = st + op * kGCodeBytes + r * 32;
                        uint32_t sfw2;
                        asm volatile("ld.shared.u16 %0, [%1];"
                                     : "=r"(sfw2)
                                     : "r"(st + 2 * kGCodeBytes + op * kGSfBytes + sfo)
                                     : "memory");
                        // blocks past k (the padding columns of the last scale tile)
                        // hold only zero codes; their scale bytes are not read
                        const float sc0 = 2 * ks < g.nb ? e8m0_value(sfw2 & 0xFFu) : 0.f;
                        const float sc1 = 2 * ks + 1 < g.nb ? e8m0_value(sfw2 >> 8) : 0.f;
                        const uint32_t orow = opa + op * kGOpBytes + r * 128;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {            // 16-byte halves of the 32-byte row
                            const uint4 w = lds128(codes + 16 * h);
                            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
                            const float sc = h ? sc1 : sc0;      // 32 codes per block
#pragma unroll
                            for (int q = 0; q < 4; ++q) {        // 8 codes -> 8 bf16 = one 16-byte chunk
                                uint32_t o[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const uint32_t byte = (wv[q] >> (8 * e)) & 0xFFu;
                                    const __nv_bfloat162 p = __floats2bfloat162_rn(
                                        e2m1_scaled(byte & 15u, sc), e2m1_scaled(byte >> 4, sc));
                                    o[e] = *reinterpret_cast<const uint32_t *>(&p);
                                }
                                const int chunk = 4 * h + q;
                                sts128(orow + ((chunk ^ (r & 7)) << 4), make_uint4(o[0], o[1], o[2], o[3]));
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(code_empty + 8 * s);
                    mbar_arrive(op_full + 8 * b);
                }
            }
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31
        const int qtr = warp & 3;
        const int row_in = qtr * 32 + lane;
        int64_t tc = 0;
        for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++tc) {
            const int a = static_cast<int>(tc & 1);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full + 8 * a,
                                                              static_cast<uint32_t>((tc >> 1) & 1)));
            if (!ok) break;
            g_fence_after();
            const int64_t mt = t / g.ntiles, nt = t % g.ntiles;
            const int64_t row = mt * kGBM + row_in;
            float *crow = g.c + row * g.ldc + nt * kGBN;
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t v[32];
                g_ld32(tmem_base + (static_cast<uint32_t>(qtr * 32) << 16) + a * 128 + cb * 32, v);
                if (row < g.m) {
                    const int64_t col0 = nt * kGBN + cb * 32;
                    if (col0 + 32 <= g.n) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            stg_f4(crow + cb * 32 + 4 * j,
                                   make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                               __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
                    } else {
                        for (int j = 0; j < 32 && col0 + j < g.n; ++j)
                            crow[cb * 32 + j] = __uint_as_float(v[j]);
                    }
                }
            }
            g_fence_before();
            mbar_arrive(acc_empty + 8 * a);
        }
    }

    g_fence_before();
    __syncthreads();
    if (warp == 1) {
        g_fence_after();
        g_tmem_dealloc(tmem_base, kGTmemCols);
    }
}

// ---- block-scaled FP4 kernel (tcgen05.mma kind::mxf4) ---------------------------
//
// The tensor cores read the packed E2M1 codes straight from shared memory and
// apply the E8M0 block scales themselves (one scale per 32 elements along K,
// two per K = 64 instruction), so nothing is dequantized on the CUDA cores.
// A CTA computes 128 x (128 NH) tiles of C (persistent over tiles, K in
// stages of 256 elements), NH = 1 or 2 halves of 128 W rows:
//   stage: A codes 128 rows x 128 B and W codes 128 NH rows x 128 B (TMA,
//   128-byte swizzle), the two 128x4 scale tiles of A and the 2 NH of W that
//   cover the stage's 8 blocks (bulk copies of the tiled layout, unchanged);
//   TMEM: 256 accumulator columns -- two 128-column buffers for NH = 1, one
//   256-column buffer for NH = 2 (one N = 256 instruction per K = 64, W row j
//   -> column j) -- then 8 + 8 NH columns per stage for the scales: A tile at
//   at column 4 at; W half h tile at at 8 + 4 (NH at + h) (tcgen05.cp
//   32x128b.warpx4 puts tile row r -- the scales of rows r, r + 32, r + 64,
//   r + 96 -- into lane r of every lane quarter; an N = 256 instruction reads
//   W rows 128-255 from the 4 columns after rows 0-127).
// A kind::mxf4 M = 128, K = 64 instruction occupies the tensor pipe for 128
// cycles at N = 128 and N = 256 alike, so the tile is as wide as one
// instruction allows (N = 256).  The pipe holds little work ahead of the
// issuing thread: every cycle that thread spends between two stages' MMAs
// (waits, address arithmetic, loop control) is a cycle the pipe may idle.  So
// a full stage is issued from straight-line code (loops with run-time bounds
// cost a quarter more per stage), a stage's scale copies are issued ahead of
// its four MMAs, by the MMA thread itself (in-order, no commit between them
// and the MMAs), each stage is released by its own commit, and the issuing
// warp is kept converged with its operands warp-uniform, one elected lane
// issuing.
// Roles: warp 0 producer, warp 1 scale copies + MMAs, 4 NH epilogue warps:
// NH per TMEM lane quarter, 128 columns each, read their part of the
// accumulator into registers and release it before they store, so the next
// tile's MMAs start while the stores drain.

constexpr int kXACodeBytes = 128 * 128;            // A codes per stage
constexpr uint32_t kXTmemCols = 512;
constexpr uint32_t kXSfCol = 256;                  // scale columns follow the accumulators

// MX = true: the FP4 product (codes + scale tiles, kind::mxf4, K = 256 per
// stage); MX = false: the bf16 product A W^T on the same structure (kind::f16,
// K = 64 per stage -- again 128 bytes of every operand row -- no scales).
template <int NH, bool MX>
struct XCfg {
    static constexpr int kBN = 128 * NH;                  // tile width (C columns, W rows)
    static constexpr int kBK = MX ? 256 : 64;             // K elements per stage
    static constexpr int kStages = 4;
    static constexpr int kEpiWarps = 4 * NH;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer, MMA, epilogue
    static constexpr int kAccBufs = NH == 1 ? 2 : 1;
    static constexpr int kWCodeBytes = kBN * 128;
    static constexpr int kSfaOff = kXACodeBytes + kWCodeBytes;
    static constexpr int kSfwOff = kSfaOff + 1024;        // A: two scale tiles; W: NH halves x 2
    static constexpr int kStageBytes = MX ? kSfwOff + 1024 * NH : kSfaOff;
    // per epilogue warp kBoxBufs staging boxes of 32 rows x kBoxCols fp32 for
    // the TMA stores of C (128-byte swizzle for 32 columns, 64-byte for 16);
    // the wide tile keeps 4 stages by storing narrower boxes, one at a time
    static constexpr int kBoxCols = NH == 1 ? 32 : 16;
    static constexpr int kBoxBufs = NH == 1 ? 2 : 1;
    static constexpr int kBoxBytes = 32 * kBoxCols * 4;
    static constexpr int kStagingOff = kStages * kStageBytes;
    static constexpr int kBarOff = kStagingOff + kEpiWarps * kBoxBufs * kBoxBytes;
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;
    static constexpr uint32_t kSfStride = 8 + 8 * NH;     // TMEM scale columns per stage
    static_assert(kStageBytes % 1024 == 0, "stages keep the 1 KB alignment of the swizzle");
    static_assert(kXSfCol + kSfStride * kStages <= kXTmemCols, "scale columns fit in TMEM");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");
};

// Shared-memory descriptor of a no-swizzle K-major matrix: core matrices of
// 8 rows x 16 bytes, SBO = distance between 8-row groups (one 16-byte chunk
// per row here, so the chunk stride is unused).
__device__ __forceinline__ uint64_t x_desc_noswz(uint32_t saddr, uint32_t sbo)
{
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(16 >> 4) << 16) |
           (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::mxf4: E2M1 A and B (format 1), both K-major,
// UE8M0 scales (bit 23), N = 128, M = 128, dense K = 64; the scale-data ids
// (bits 4-5 for B, 29-30 for A) pick the byte of the 32-bit TMEM scale word
// the instruction starts at.
__host__ __device__ constexpr uint32_t x_idesc(uint32_t sf_id)
{
    return (sf_id << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | (1u << 23) |
           ((128u >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void x_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                      uint32_t sfa, uint32_t sfb, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}

// elect.sync: one lane of the converged warp.
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(pred));
    return pred != 0;
}

__device__ __forceinline__ void x_cp_sf(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

template <int NH, bool MX>
__global__ void __launch_bounds__(XCfg<NH, MX>::kThreads, 1)
    w4a4_mxf4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmC, const GemmArgs g)
{
    using C = XCfg<NH, MX>;
    constexpr int kXStages = C::kStages, kXBN = C::kBN, kXWCodeBytes = C::kWCodeBytes;
    constexpr int kXBK = C::kBK;
    constexpr int kXSfaOff = C::kSfaOff, kXSfwOff = C::kSfwOff, kXStageBytes = C::kStageBytes;
    constexpr uint32_t kXSfStride = C::kSfStride;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    const uint32_t bar = base + C::kBarOff;
    const uint32_t full = bar, empty = bar + 8 * kXStages;
    const uint32_t acc_full = bar + 16 * kXStages, acc_empty = acc_full + 16;
    const uint32_t tmem_slot = acc_empty + 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles = g.mtiles * g.ntiles;
    const int64_t wrt = (g.n + 127) / 128;            // 128-row scale tiles of W

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmC);
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, 1);
        }
        for (int b = 0; b < C::kAccBufs; ++b) {
            mbar_init(acc_full + 8 * b, 1);
            mbar_init(acc_empty + 8 * b, 128 * NH);
        }
        mbar_fence_init();
    }
    if (warp == 1) g_tmem_alloc(tmem_slot, kXTmemCols);
    g_fence_before();
    __syncthreads();
    g_fence_after();
    uint32_t tmem_base;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(tmem_base) : "r"(tmem_slot) : "memory");
    grid_dependency_wait();

    if (warp == 0) {
        if (lane == 0) {
            int64_t kk = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int64_t mt = t / g.ntiles, nt = t % g.ntiles;
                for (int64_t ks = 0; ks < g.ksteps; ++ks, ++kk) {
                    const int s = static_cast<int>(kk % kXStages);
                    if (kk >= kXStages &&
                        !mbar_wait(empty + 8 * s, static_cast<uint32_t>(((kk / kXStages) - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    // scale tiles holding the blocks this stage's instructions
                    // use (none for a half of W past the edge of C)
                    const int64_t rem = (g.k - ks * kXBK + 63) / 64;
                    const int64_t nmma = rem < 4 ? rem : 4;
                    const uint32_t sf_bytes = MX ? static_cast<uint32_t>((nmma + 1) / 2) * 512u : 0u;
                    const bool w1 = NH == 2 && 2 * nt + 1 < wrt;
                    const uint32_t st = base + s * kXStageBytes;
                    mbar_arrive_expect_tx(full + 8 * s, kXACodeBytes + kXWCodeBytes +
                                                            (w1 ? 3u : 2u) * sf_bytes);
                    // 128 bytes of every row: 128 packed-code bytes or 64 bf16
                    const int32_t x = static_cast<int32_t>(ks * (MX ? 128 : 64));
                    tma_load_2d(st, &tmA, x, static_cast<int32_t>(mt * 128), full + 8 * s, 0);
                    tma_load_2d(st + kXACodeBytes, &tmW, x, static_cast<int32_t>(nt * kXBN),
                                full + 8 * s, 0);
                    if constexpr (MX) {
                        bulk_load(st + kXSfaOff, g.sfa + (mt * g.ncb + 2 * ks) * 512, sf_bytes,
                                  full + 8 * s);
                        bulk_load(st + kXSfwOff, g.sfw + (NH * nt * g.ncb + 2 * ks) * 512, sf_bytes,
                                  full + 8 * s);
                        if (w1)
                            bulk_load(st + kXSfwOff + 1024,
                                      g.sfw + ((2 * nt + 1) * g.ncb + 2 * ks) * 512, sf_bytes,
                                      full + 8 * s);
                    }
                }
            }
            // the last copies issued into each stage have landed before exit
            for (int64_t j = kk - 1; j >= 0 && j >= kk - kXStages; --j)
                (void)mbar_wait(full + 8 * static_cast<int>(j % kXStages),
                                static_cast<uint32_t>((j / kXStages) & 1));
        }
    } else if (warp == 1) {
        // MMA issuer: the whole warp runs the loop, so that descriptors and
        // addresses are warp-uniform values; one elected lane issues a
        // stage's scale copies (A tile, then W's halves, per scale tile at)
        // and its MMAs -- in order from one thread, the copies need no
        // commit before the MMAs that read them.  The wait for a stage's data
        // closes the previous stage (the first stage of a tile: at the top of
        // the tile).  An odd block count leaves one padding block inside the
        // last instruction: the warp first sets its scale bytes to 2^0 (lane
        // r: row r of each tile).
        int64_t kk = 0, tc = 0;
        bool ok = true;
        const bool pad_fix = MX && (g.nb & 1) != 0;
        // the issuing lane, elected once: a commit tracks only the tcgen05
        // operations of its own thread, so one lane issues everything
        const bool leader = elect_one();
        constexpr uint32_t kIdN = static_cast<uint32_t>((NH - 1) * (128 >> 3)) << 17;  // N += 128
        constexpr uint32_t id0 = x_idesc(0) + kIdN, id2 = x_idesc(2) + kIdN;
        // stages whose four K = 64 instructions all lie inside k
        const int64_t full_steps = MX ? g.k / kXBK : 0;
        auto wait_full = [&](int64_t q) {
            return __all_sync(0xffffffffu, mbar_wait(full + 8 * static_cast<int>(q % kXStages),
                                                     static_cast<uint32_t>((q / kXStages) & 1)));
        };
        for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++tc) {
            // accumulator buffer b of tile tc is free once the epilogue has
            // read tile tc - kAccBufs from it
            const int b = static_cast<int>(tc % C::kAccBufs);
            const int64_t use = tc / C::kAccBufs;
            if (use >= 1)
                ok = __all_sync(0xffffffffu,
                                mbar_wait(acc_empty + 8 * b, static_cast<uint32_t>((use - 1) & 1)));
            const uint32_t acc = tmem_base + 128 * b;
            if (ok) ok = wait_full(kk);
            for (int64_t ks = 0; ks < g.ksteps && ok; ++ks, ++kk) {
                const int s = static_cast<int>(kk % kXStages);
                const bool last = ks == g.ksteps - 1;
                const uint32_t st = base + s * kXStageBytes;
                const uint32_t sfa_s = st + kXSfaOff, sfw_s = st + kXSfwOff;
                if (pad_fix && last) {
                    const int kb = static_cast<int>(g.nb - 8 * ks);     // padding block, local index
                    const uint32_t off = static_cast<uint32_t>((kb >> 2) * 512 + 16 * lane + (kb & 3));
#pragma unroll
                    for (int grp = 0; grp < 4; ++grp) {
                        asm volatile("st.shared.u8 [%0], %1;" ::"r"(sfa_s + off + 4 * grp), "r"(127u) : "memory");
#pragma unroll
                        for (int hh = 0; hh < NH; ++hh)
                            asm volatile("st.shared.u8 [%0], %1;" ::"r"(sfw_s + 1024 * hh + off + 4 * grp),
                                         "r"(127u)
                                         : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                g_fence_after();
                // TMEM scale columns of stage s: A tile at at 4 at, W half h
                // tile at at 8 + 4 (NH at + h); one N = 128 NH instruction
                // reads the tiles of W's halves from consecutive 4-column
                // groups.  Descriptors advance in 16-byte units: +2 = the next
                // 32 bytes of codes (K = 64), +32 = the next 512-byte scale
                // tile, +64 = the next half's scale tiles of W.
                const uint32_t sft = tmem_base + kXSfCol + kXSfStride * s;
                const uint64_t da = g_desc(st), db = g_desc(st + kXACodeBytes);
                const uint64_t dsa = x_desc_noswz(sfa_s, 128), dsw = x_desc_noswz(sfw_s, 128);
                const uint32_t a0 = ks > 0 ? 1u : 0u;           // accumulate into D
                auto copies = [&](int at) {
                    x_cp_sf(sft + 4 * at, dsa + 32 * at);
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh)
                        x_cp_sf(sft + 8 + 4 * (NH * at + hh), dsw + 64 * hh + 32 * at);
                };
                bool next = true;
                if (MX && ks < full_steps) {
                    // the copies first: an MMA issued right behind a copy
                    // waits for it, and four MMAs in a row leave the pipe
                    // more work queued while the warp does its bookkeeping
                    if (leader) {
                        copies(0);
                        copies(1);
                        x_mma(acc, da, db, id0, sft, sft + 8, a0);
                        x_mma(acc, da + 2, db + 2, id2, sft, sft + 8, 1u);
                        x_mma(acc, da + 4, db + 4, id0, sft + 4, sft + 8 + 4 * NH, 1u);
                        x_mma(acc, da + 6, db + 6, id2, sft + 4, sft + 8 + 4 * NH, 1u);
                        g_commit(empty + 8 * s);
                        if (last) g_commit(acc_full + 8 * b);
                    }
                    if (!last) next = wait_full(kk + 1);
                } else {
                    if (leader && !MX) {
                        // kind::f16: four K = 16 steps of 32 bytes; zero fill past k
                        constexpr uint32_t kIdF16 = (1u << 4) | (1u << 7) | (1u << 10) |
                                                    ((static_cast<uint32_t>(kXBN) >> 3) << 17) |
                                                    ((128u >> 4) << 24);
                        for (int j = 0; j < 4; ++j)
                            g_mma_id(acc, da + 2 * j, db + 2 * j, kIdF16, (ks > 0 || j > 0) ? 1u : 0u);
                    }
                    if (leader && MX) {
                        // the last stage of a k that is not a multiple of 256
                        const int64_t rem = (g.k - ks * kXBK + 63) / 64;
                        const int nmma = rem < 4 ? static_cast<int>(rem) : 4;
                        for (int at = 0; at < (nmma + 1) / 2; ++at) {
                            copies(at);
                            for (int j = 2 * at; j < 2 * at + 2 && j < nmma; ++j)
                                x_mma(acc, da + 2 * j, db + 2 * j, (j & 1) ? id2 : id0, sft + 4 * at,
                                      sft + 8 + 4 * (NH * at), (ks > 0 || j > 0) ? 1u : 0u);
                        }
                    }
                    if (leader) {
                        g_commit(empty + 8 * s);
                        if (last) g_commit(acc_full + 8 * b);
                    }
                    if (!last) next = wait_full(kk + 1);
                }
                ok = next;
                __syncwarp();
            }
        }
        if (tc >= 1 && ok) {
            const int64_t last = tc - 1;
            (void)mbar_wait(acc_full + 8 * static_cast<int>(last % C::kAccBufs),
                            static_cast<uint32_t>((last / C::kAccBufs) & 1));
        }
        __syncwarp();
    } else {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 and the 128
        // columns of half h = (w - 2) / 4 of the tile
        const int qtr = warp & 3, h = (warp - 2) >> 2;
        const uint32_t stg = base + C::kStagingOff +
                             static_cast<uint32_t>(C::kBoxBufs * C::kBoxBytes * (warp - 2));
        int64_t tc = 0, nbox = 0;
        for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++tc) {
            const int b = static_cast<int>(tc % C::kAccBufs);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full + 8 * b,
                                                              static_cast<uint32_t>((tc / C::kAccBufs) & 1)));
            if (!ok) break;
            g_fence_after();
            uint32_t v[128];
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(qtr * 32) << 16) + 128 * (b + h);
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
                "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
                "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
                "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                  "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
                  "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
                  "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
                  "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
                  "=r"(v[31]), "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]),
                  "=r"(v[37]), "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]),
                  "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]),
                  "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]),
                  "=r"(v[55]), "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]),
                  "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
                : "r"(taddr)
                : "memory");
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
                "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
                "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
                "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
                : "=r"(v[64]), "=r"(v[65]), "=r"(v[66]), "=r"(v[67]), "=r"(v[68]), "=r"(v[69]),
                  "=r"(v[70]), "=r"(v[71]), "=r"(v[72]), "=r"(v[73]), "=r"(v[74]), "=r"(v[75]),
                  "=r"(v[76]), "=r"(v[77]), "=r"(v[78]), "=r"(v[79]), "=r"(v[80]), "=r"(v[81]),
                  "=r"(v[82]), "=r"(v[83]), "=r"(v[84]), "=r"(v[85]), "=r"(v[86]), "=r"(v[87]),
                  "=r"(v[88]), "=r"(v[89]), "=r"(v[90]), "=r"(v[91]), "=r"(v[92]), "=r"(v[93]),
                  "=r"(v[94]), "=r"(v[95]), "=r"(v[96]), "=r"(v[97]), "=r"(v[98]), "=r"(v[99]),
                  "=r"(v[100]), "=r"(v[101]), "=r"(v[102]), "=r"(v[103]), "=r"(v[104]), "=r"(v[105]),
                  "=r"(v[106]), "=r"(v[107]), "=r"(v[108]), "=r"(v[109]), "=r"(v[110]), "=r"(v[111]),
                  "=r"(v[112]), "=r"(v[113]), "=r"(v[114]), "=r"(v[115]), "=r"(v[116]), "=r"(v[117]),
                  "=r"(v[118]), "=r"(v[119]), "=r"(v[120]), "=r"(v[121]), "=r"(v[122]), "=r"(v[123]),
                  "=r"(v[124]), "=r"(v[125]), "=r"(v[126]), "=r"(v[127])
                : "r"(taddr + 64)
                : "memory");
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            g_fence_before();
            mbar_arrive(acc_empty + 8 * b);      // the accumulator may be overwritten now
            // C through shared memory: 128 / kBoxCols boxes per warp, each
            // written row = lane in the swizzle of the TMA map, then one TMA
            // store (clipped at the last row of C) while the next box is filled
            // (the TMA store writes whole 16-byte units of a row, so its map
            // covers the first n4 = 4 floor(n / 4) columns; the last n % 4
            // columns are stored directly)
            const int64_t mt = t / g.ntiles, nt = t % g.ntiles;
            const int64_t y0 = mt * 128 + 32 * qtr, x0 = nt * kXBN + 128 * h;
            const int64_t n4 = g.n & ~int64_t(3);
            constexpr int kBC = C::kBoxCols, kChunks = kBC / 4;
            if (y0 < g.m && x0 < n4) {
#pragma unroll
                for (int c = 0; c < 128 / kBC; ++c, ++nbox) {
                    if (x0 + kBC * c >= n4) break;           // boxes past column n4 of C
                    const uint32_t buf =
                        stg + static_cast<uint32_t>(C::kBoxBytes) * static_cast<uint32_t>(nbox % C::kBoxBufs);
                    if (nbox >= C::kBoxBufs) {
                        // the box's last store has read it
                        if (lane == 0) {
                            if constexpr (C::kBoxBufs == 2)
                                bulk_wait_group_read<1>();
                            else
                                bulk_wait_group_read<0>();
                        }
                        __syncwarp();
                    }
                    // 16-byte chunk q of row r sits at q ^ (r & 7) (128-byte
                    // swizzle) or q ^ ((r >> 1) & 3) (64-byte swizzle)
                    const uint32_t sw = kBC == 32 ? static_cast<uint32_t>(lane & 7)
                                                  : static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll
                    for (int q = 0; q < kChunks; ++q)
                        sts128(buf + static_cast<uint32_t>(kBC * 4 * lane) + ((q ^ sw) << 4),
                               make_uint4(v[kBC * c + 4 * q], v[kBC * c + 4 * q + 1], v[kBC * c + 4 * q + 2],
                                          v[kBC * c + 4 * q + 3]));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, static_cast<int32_t>(x0 + kBC * c), static_cast<int32_t>(y0), buf);
                        bulk_commit_group();
                    }
                    __syncwarp();
                }
            }
            if (n4 < g.n && x0 <= n4 && n4 < x0 + 128 && y0 + lane < g.m) {
                float *crow = g.c + (y0 + lane) * g.ldc + x0;
#pragma unroll
                for (int j = 0; j < 128; ++j)
                    if (x0 + j >= n4 && x0 + j < g.n) crow[j] = __uint_as_float(v[j]);
            }
        }
        if (lane == 0) bulk_wait_group_all();   // the stores have read shared memory and landed
        __syncwarp();
    }

    g_fence_before();
    __syncthreads();
    if (warp == 1) {
        g_fence_after();
        g_tmem_dealloc(tmem_base, kXTmemCols);
    }
}

struct GSlot {
    std::once_flag once[64];
    cudaError_t err[64] = {};
};

kq_status launch_dequant(const CUtensorMap &ma, const CUtensorMap &mw, const GemmArgs &g,
                         int sm_count, cudaStream_t stream)
{
    auto kern = w4a4_gemm_kernel;
    static GSlot slot;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KQ_ERR_CUDA;
    std::call_once(slot.once[dev], [&] {
        slot.err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kGSmemBytes);
    });
    if (slot.err[dev] != cudaSuccess) return KQ_ERR_CUDA;
    const int64_t tiles = g.mtiles * g.ntiles;
    if (tiles == 0) return KQ_OK;
    const int grid = static_cast<int>(std::min<int64_t>(tiles, sm_count));
    return launch_pdl(kern, grid, kGThreads, static_cast<size_t>(kGSmemBytes), stream, ma, mw, g);
}

// Sums of (c - c_ref)^2 and c_ref^2 in fp64: one partial per thread, a
// block reduction, one atomic per block and sum.
__global__ void __launch_bounds__(256) layer_error_kernel(const float *__restrict__ c, int64_t ldc,
                                                          const float *__restrict__ r, int64_t ldr,
                                                          int64_t m, int64_t n, double *out)
{
    const int64_t n4 = (n + 3) / 4, total = m * n4;
    double e2 = 0.0, r2 = 0.0;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = idx / n4, j = (idx % n4) * 4;
        const float *cp = c + i * ldc + j, *rp = r + i * ldr + j;
        if (j + 4 <= n) {
            const float4 a = ldg_nc_f4(cp), b = ldg_nc_f4(rp);
            const double d0 = static_cast<double>(a.x) - b.x, d1 = static_cast<double>(a.y) - b.y,
                         d2 = static_cast<double>(a.z) - b.z, d3 = static_cast<double>(a.w) - b.w;
            e2 += d0 * d0 + d1 * d1 + d2 * d2 + d3 * d3;
            r2 += static_cast<double>(b.x) * b.x + static_cast<double>(b.y) * b.y +
                  static_cast<double>(b.z) * b.z + static_cast<double>(b.w) * b.w;
        } else {
            for (int64_t t = 0; j + t < n; ++t) {
                const double dd = static_cast<double>(cp[t]) - rp[t];
                e2 += dd * dd;
                r2 += static_cast<double>(rp[t]) * rp[t];
            }
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        e2 += __shfl_xor_sync(0xffffffffu, e2, o);
        r2 += __shfl_xor_sync(0xffffffffu, r2, o);
    }
    __shared__ double part[2][8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        part[0][warp] = e2;
        part[1][warp] = r2;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double se = 0.0, sr = 0.0;
        for (int w = 0; w < (blockDim.x >> 5); ++w) {
            se += part[0][w];
            sr += part[1][w];
        }
        atomicAdd(out, se);
        atomicAdd(out + 1, sr);
    }
}

template <int NH, bool MX>
kq_status launch_mxf4_t(const CUtensorMap &ma, const CUtensorMap &mw, const CUtensorMap &mc,
                        const GemmArgs &g, int sm_count, cudaStream_t stream)
{
    using C = XCfg<NH, MX>;
    auto kern = w4a4_mxf4_kernel<NH, MX>;
    static GSlot slot;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KQ_ERR_CUDA;
    std::call_once(slot.once[dev], [&] {
        slot.err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
    });
    if (slot.err[dev] != cudaSuccess) return KQ_ERR_CUDA;
    const int64_t tiles = g.mtiles * g.ntiles;
    const int grid = static_cast<int>(std::min<int64_t>(tiles, sm_count));
    return launch_pdl(kern, grid, C::kThreads, static_cast<size_t>(C::kSmemBytes), stream, ma, mw, mc,
                      g);
}

kq_status launch_w4a4_mxf4(const uint8_t *qa, int64_t ldqa, const uint8_t *sfa, const uint8_t *qw,
                           int64_t ldqw, const uint8_t *sfw, int64_t m, int64_t n, int64_t k,
                           float *c, int64_t ldc, int wide_sel, cudaStream_t stream)
{
    DeviceInfo info;
    kq_status st = device_info(info);
    if (st != KQ_OK) return st;
    CUtensorMap ma, mw;
    st = make_tensor_map_2d_u8(&ma, const_cast<uint8_t *>(qa), m, k / 2, ldqa, 128, 128,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != KQ_OK) return st;
    // Tile width by a wave model fitted on GB300: a CTA's time is its tile
    // count times (K stages x the stage time + the tile's exposed epilogue),
    // in narrow-stage units -- a wide stage (twice the work) costs 1.35, the
    // narrow tile's epilogue is mostly hidden behind its second accumulator
    // (0.5), the wide tile's single accumulator exposes about 2.
    const int64_t mtiles = (m + 127) / 128, ksteps = (k + 255) / 256;
    auto cost = [&](int64_t bn, double per_stage, double per_tile) {
        const int64_t tiles = mtiles * ((n + bn - 1) / bn);
        const int64_t waves = (tiles + info.sm_count - 1) / info.sm_count;
        return static_cast<double>(waves) * (static_cast<double>(ksteps) * per_stage + per_tile);
    };
    const bool wide = wide_sel >= 0 ? wide_sel == 1 : cost(256, 1.35, 2.0) < cost(128, 1.0, 0.5);
    const int bn = wide ? 256 : 128;
    st = make_tensor_map_2d_u8(&mw, const_cast<uint8_t *>(qw), n, k / 2, ldqw, 128,
                               static_cast<uint32_t>(bn), CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != KQ_OK) return st;
    GemmArgs g;
    g.m = m;
    g.n = n;
    g.k = k;
    g.nb = k / 32;
    g.ncb = (k / 32 + 3) / 4;
    g.sfa = sfa;
    g.sfw = sfw;
    g.c = c;
    g.ldc = ldc;
    g.mtiles = (m + 127) / 128;
    g.ntiles = (n + bn - 1) / bn;
    g.ksteps = (k + 255) / 256;
    CUtensorMap mc;   // the first 4 floor(n / 4) columns (at least 4: never stored past n)
    const int64_t n4 = std::max<int64_t>(n & ~int64_t(3), 4);
    const uint32_t box_cols = static_cast<uint32_t>(wide ? XCfg<2, true>::kBoxCols : XCfg<1, true>::kBoxCols);
    st = make_tensor_map_2d_f32(&mc, c, m, n4, ldc, box_cols, 32,
                                box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    if (st != KQ_OK) return st;
    return wide ? launch_mxf4_t<2, true>(ma, mw, mc, g, info.sm_count, stream)
                : launch_mxf4_t<1, true>(ma, mw, mc, g, info.sm_count, stream);
}

}  // namespace

kq_status launch_layer_error(const float *c, int64_t ldc, const float *r, int64_t ldr, int64_t m,
                             int64_t n, double *out, cudaStream_t stream)
{
    DeviceInfo info;
    kq_status st = device_info(info);
    if (st != KQ_OK) return st;
    if (cudaMemsetAsync(out, 0, 2 * sizeof(double), stream) != cudaSuccess) return KQ_ERR_CUDA;
    if (m == 0 || n == 0) return KQ_OK;
    const int64_t work = m * ((n + 3) / 4);
    const int grid = static_cast<int>(
        std::min<int64_t>((work + 255) / 256, static_cast<int64_t>(info.sm_count) * 8));
    layer_error_kernel<<<grid, 256, 0, stream>>>(c, ldc, r, ldr, m, n, out);
    return check_launch();
}

kq_status launch_w4a4_gemm(const uint8_t *qa, int64_t ldqa, const uint8_t *sfa, const uint8_t *qw,
                           int64_t ldqw, const uint8_t *sfw, int64_t m, int64_t n, int64_t k,
                           float *c, int64_t ldc, int variant, cudaStream_t stream)
{
    if (variant == 0) return launch_w4a4_mxf4(qa, ldqa, sfa, qw, ldqw, sfw, m, n, k, c, ldc, -1, stream);
    if (variant == 2 || variant == 3)
        return launch_w4a4_mxf4(qa, ldqa, sfa, qw, ldqw, sfw, m, n, k, c, ldc, variant - 2, stream);
    DeviceInfo info;
    kq_status st = device_info(info);
    if (st != KQ_OK) return st;
    CUtensorMap ma, mw;
    st = make_tensor_map_2d_u8(&ma, const_cast<uint8_t *>(qa), m, k / 2, ldqa, 32, kGBM,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != KQ_OK) return st;
    st = make_tensor_map_2d_u8(&mw, const_cast<uint8_t *>(qw), n, k / 2, ldqw, 32, kGBN,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != KQ_OK) return st;
    GemmArgs g;
    g.m = m;
    g.n = n;
    g.k = k;
    g.nb = k / 32;
    g.ncb = (k / 32 + 3) / 4;
    g.sfa = sfa;
    g.sfw = sfw;
    g.c = c;
    g.ldc = ldc;
    g.mtiles = (m + kGBM - 1) / kGBM;
    g.ntiles = (n + kGBN - 1) / kGBN;
    g.ksteps = (k + kGBK - 1) / kGBK;
    return launch_dequant(ma, mw, g, info.sm_count, stream);
}

kq_status launch_bf16_gemm(const uint16_t *a, int64_t lda, const uint16_t *w, int64_t ldw,
                           int64_t m, int64_t n, int64_t k, float *c, int64_t ldc,
                           cudaStream_t stream)
{
    DeviceInfo info;
    kq_status st = device_info(info);
    if (st != KQ_OK) return st;
    // tile width by the same wave model as the FP4 product (K stages of 64)
    const int64_t mtiles = (m + 127) / 128, ksteps = (k + 63) / 64;
    auto cost = [&](int64_t bn, double per_stage, double per_tile) {
        const int64_t tiles = mtiles * ((n + bn - 1) / bn);
        const int64_t waves = (tiles + info.sm_count - 1) / info.sm_count;
        return static_cast<double>(waves) * (static_cast<double>(ksteps) * per_stage + per_tile);
    };
    const bool wide = cost(256, 1.35, 2.0) < cost(128, 1.0, 0.5);
    const int bn = wide ? 256 : 128;
    CUtensorMap ma, mw, mc;
    st = make_tensor_map_2d_bf16(&ma, a, m, k, lda, 64, 128);
    if (st != KQ_OK) return st;
    st = make_tensor_map_2d_bf16(&mw, w, n, k, ldw, 64, static_cast<uint32_t>(bn));
    if (st != KQ_OK) return st;
    const int64_t n4 = std::max<int64_t>(n & ~int64_t(3), 4);
    const uint32_t box_cols = static_cast<uint32_t>(wide ? XCfg<2, false>::kBoxCols : XCfg<1, false>::kBoxCols);
    st = make_tensor_map_2d_f32(&mc, c, m, n4, ldc, box_cols, 32,
                                box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    if (st != KQ_OK) return st;
    GemmArgs g;
    g.m = m;
    g.n = n;
    g.k = k;
    g.nb = 0;
    g.ncb = 0;
    g.sfa = nullptr;
    g.sfw = nullptr;
    g.c = c;
    g.ldc = ldc;
    g.mtiles = mtiles;
    g.ntiles = (n + bn - 1) / bn;
    g.ksteps = ksteps;
    return wide ? launch_mxf4_t<2, false>(ma, mw, mc, g, info.sm_count, stream)
                : launch_mxf4_t<1, false>(ma, mw, mc, g, info.sm_count, stream);
}

}  // namespace kq
