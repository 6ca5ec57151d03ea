// TMA-fed MXFP4 quantizer kernels: KroQuant butterfly, diagonal scale,
// fixed block-Hadamard and identity transforms (sm_103a).
//
// What is computed ("KroQuant: Kronecker-Structured Block Transforms for
// Efficient Post-Training Quantization of Diffusion Transformers"):
//   eq. (4)/(5): per 32-channel block j, y = a . K_j with
//   K_j = G1 (x) ... (x) G5; eq. (12): G_k acts on bit 5-k of the channel
//   index inside the block.  Applying the Kronecker product factor by factor
//   is the same linear map: for every pair of channels (i, i + 2^p) that
//   differ only in bit p = 5 - k,
//       y_i       <- y_i * G_k[0][0] + y_{i+2^p} * G_k[1][0]
//       y_{i+2^p} <- y_i * G_k[0][1] + y_{i+2^p} * G_k[1][1]
//   (row vector times G_k, K1's A_tile @ K orientation of Sec. 3.5.1).  The
//   five stages cost 10 fp32 operations per element instead of the 32 MACs
//   of the dense block; they run on packed fp32x2 FMAs.
//   Sec. 3.1 / 4.1: the block's fp32 y is then quantized to MXFP4 directly
//   (no intermediate rounding of y).
//
// Data path (one pass, [KQ] Sec. 4.4: one read, one write per tile):
//   * persistent CTAs, one producer warp + 8 consumer warps;
//   * a tile is BR rows x 128 channels (4 blocks), loaded as two 2-D TMA
//     boxes of BR x 64 bf16 with the 128-byte swizzle into a STAGES-deep
//     shared-memory ring guarded by full/empty mbarriers;
//   * each consumer thread owns one (row, block) item: it reads its 64 bytes
//     from shared memory (the swizzle makes the 4 x 16-byte reads of a
//     quarter-warp hit 8 distinct bank groups), transforms, finds amax,
//     encodes and stores 16 bytes of codes + 1 scale byte.
#include <algorithm>
#include <mutex>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;

// Per-block parameter bytes a tile stages next to its activations.
template <int T>
__host__ __device__ constexpr int param_bytes_per_block()
{
    return T == kKron ? 80 : (T == kDiag ? 128 : 0);   // 5 factors / 32 scales
}

// Shared-memory stride between the staged parameters of the tile's blocks.
// The two blocks a quarter-warp reads must not start 128 bytes apart (same
// banks): the 32 scales of the diagonal kernel sit 144 bytes apart.
template <int T>
__host__ __device__ constexpr int param_stride()
{
    return T == kDiag ? 144 : param_bytes_per_block<T>();
}

template <int T, int BR, int STAGES>
struct TileCfg {
    static constexpr int kBoxBytes = BR * 128;           // BR rows x 64 bf16
    static constexpr int kABytes = 2 * kBoxBytes;        // 128 channels
    static constexpr int kParamBytes = param_bytes_per_block<T>() > 0 ? 1024 : 0;
    static constexpr int kStageBytes = kABytes + kParamBytes;
    static constexpr int kSmemBytes = STAGES * kStageBytes + 1024 + 2 * STAGES * 8;
    static_assert(BR % 8 == 0 && BR <= 256, "box rows");
    static_assert(4 * param_stride<T>() <= kParamBytes, "parameter area");
};

__device__ __forceinline__ float2 swap2(float2 a) { return make_float2(a.y, a.x); }

// y <- y . (G (x) I) on the channel pairs that differ in bit p >= 1 (float2
// index stride 2^(p-1)).
template <int S2>
__device__ __forceinline__ void butterfly_cross(float2 (&Y)[16], float4 g)
{
    const float2 a00 = make_float2(g.x, g.x), a01 = make_float2(g.y, g.y);
    const float2 a10 = make_float2(g.z, g.z), a11 = make_float2(g.w, g.w);
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        if (t & S2) continue;
        const float2 lo = Y[t], hi = Y[t | S2];
        Y[t] = __ffma2_rn(hi, a10, __fmul2_rn(lo, a00));
        Y[t | S2] = __ffma2_rn(hi, a11, __fmul2_rn(lo, a01));
    }
}

// Bit 0: both channels of a pair sit in one float2 (x0, x1):
// (x0 g00 + x1 g10, x0 g01 + x1 g11) = (x0, x1)*(g00, g11) + (x1, x0)*(g10, g01).
__device__ __forceinline__ void butterfly_inpair(float2 (&Y)[16], float4 g)
{
    const float2 d0 = make_float2(g.x, g.w), d1 = make_float2(g.z, g.y);
#pragma unroll
    for (int t = 0; t < 16; ++t) Y[t] = __ffma2_rn(swap2(Y[t]), d1, __fmul2_rn(Y[t], d0));
}

// `prm`: shared-memory address of this block's staged parameters.
template <int T>
__device__ __forceinline__ void apply_transform(float2 (&Y)[16], uint32_t prm)
{
    if constexpr (T == kKron) {
        const float4 g1 = lds_f4(prm), g2 = lds_f4(prm + 16), g3 = lds_f4(prm + 32);
        const float4 g4 = lds_f4(prm + 48), g5 = lds_f4(prm + 64);
        butterfly_inpair(Y, g5);      // G5: bit 0
        butterfly_cross<1>(Y, g4);    // G4: bit 1
        butterfly_cross<2>(Y, g3);    // G3: bit 2
        butterfly_cross<4>(Y, g2);    // G2: bit 3
        butterfly_cross<8>(Y, g1);    // G1: bit 4
    } else if constexpr (T == kDiag) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 v = lds_f4(prm + 16 * k);
            Y[2 * k] = __fmul2_rn(Y[2 * k], make_float2(v.x, v.y));
            Y[2 * k + 1] = __fmul2_rn(Y[2 * k + 1], make_float2(v.z, v.w));
        }
    } else if constexpr (T == kHadamard) {
        // unnormalised +-1 butterflies, then one multiply by 1/sqrt(32)
        const float2 pm = make_float2(1.0f, -1.0f), mm = make_float2(-1.0f, -1.0f);
#pragma unroll
        for (int t = 0; t < 16; ++t) Y[t] = __ffma2_rn(Y[t], pm, swap2(Y[t]));
#pragma unroll
        for (int S2 = 1; S2 < 16; S2 <<= 1) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                if (t & S2) continue;
                const float2 lo = Y[t], hi = Y[t | S2];
                Y[t] = __fadd2_rn(lo, hi);
                Y[t | S2] = __ffma2_rn(hi, mm, lo);
            }
        }
        const float c = 0.17677669529663688f;  // 1/sqrt(32) rounded to fp32
        const float2 c2 = make_float2(c, c);
#pragma unroll
        for (int t = 0; t < 16; ++t) Y[t] = __fmul2_rn(Y[t], c2);
    }
}

__device__ __forceinline__ void store_scale(const QuantParams &p, int64_t row, int64_t j,
                                            uint32_t byte)
{
    if (p.sf_layout == KQ_SF_ROWMAJOR) {
        if (row < p.m) p.sf[row * p.nb + j] = static_cast<uint8_t>(byte);
    } else {
        p.sf[sf_blocked_offset(row, j, p.ncb)] = static_cast<uint8_t>(byte);
    }
}

// Marks every item this thread owns from `tile` on as failed (scale 0xFF).
template <int BR>
__device__ void fail_items(const QuantParams &p, int64_t tile, int lane, int cw)
{
    const int h = lane & 1, rlo = (lane >> 1) & 3, box = (lane >> 3) & 1, rhi = (lane >> 4) & 1;
    for (; tile < p.ntiles; tile += gridDim.x) {
        const int64_t rt = tile / p.ncol_tiles, ct = tile % p.ncol_tiles;
        const int64_t j = ct * 4 + box * 2 + h;
        if (j >= p.nb) continue;
        for (int g = cw; g < BR / 8; g += kConsumerWarps) {
            const int64_t row = rt * BR + g * 8 + rhi * 4 + rlo;
            if (row < p.m_rows) store_scale(p, row, j, 0xFFu);
        }
    }
}

template <int T, int BR, int STAGES>
__global__ void __launch_bounds__(kThreads, 2)
    quant_tma_kernel(const __grid_constant__ CUtensorMap tmA, const QuantParams p)
{
    using Cfg = TileCfg<T, BR, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;   // 128B-swizzle atoms: 1 KB
    const uint32_t bar_full = base + STAGES * Cfg::kStageBytes;
    const uint32_t bar_empty = bar_full + STAGES * 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);              // a kernel parameter: no dependency on earlier grids
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerThreads);
        }
        mbar_fence_init();
    }
    __syncthreads();
    grid_dependency_wait();

    if (warp == kConsumerWarps) {
        // ---------------- producer: one thread issues the TMA loads ----------------
        if (lane != 0) return;
        const uint64_t pol = l2_policy_evict_first();
        int64_t it = 0;
        for (TileWalk tw(static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x),
                             static_cast<int>(p.ncol_tiles));
             tw.rt < p.nrow_tiles; tw.next(), ++it) {
            const int s = static_cast<int>(it % STAGES);
            const uint32_t ph = static_cast<uint32_t>((it / STAGES) & 1);
            if (it >= STAGES && !mbar_wait(bar_empty + 8 * s, ph ^ 1u)) break;
            const int64_t rt = tw.rt, ct = tw.ct;
            const uint32_t dst = base + s * Cfg::kStageBytes;
            uint32_t pbytes = 0;
            const void *psrc = nullptr;
            if constexpr (param_bytes_per_block<T>() > 0) {
                const int64_t left = p.nb - ct * 4;
                pbytes = static_cast<uint32_t>((left < 4 ? left : 4) * param_bytes_per_block<T>());
                psrc = (T == kKron) ? static_cast<const void *>(p.factors + (p.shared_params ? 0 : ct * 4 * 20))
                                    : static_cast<const void *>(p.s + ct * 4 * 32);
            }
            mbar_arrive_expect_tx(bar_full + 8 * s, Cfg::kABytes + pbytes);
            tma_load_2d(dst, &tmA, static_cast<int32_t>(ct * 128), static_cast<int32_t>(rt * BR),
                        bar_full + 8 * s, pol);
            tma_load_2d(dst + Cfg::kBoxBytes, &tmA, static_cast<int32_t>(ct * 128 + 64),
                        static_cast<int32_t>(rt * BR), bar_full + 8 * s, pol);
            if constexpr (param_stride<T>() == param_bytes_per_block<T>()) {
                if (T == kKron && p.shared_params) {
                    // one factor set for every block: a copy of it per block slot
                    const uint32_t per = param_bytes_per_block<T>();
                    for (uint32_t off = 0; off < pbytes; off += per)
                        bulk_load(dst + Cfg::kABytes + off, psrc, per, bar_full + 8 * s);
                } else if (pbytes) {
                    bulk_load(dst + Cfg::kABytes, psrc, pbytes, bar_full + 8 * s);
                }
            } else {
                // one copy per block into its padded slot
                const uint32_t per = param_bytes_per_block<T>();
                for (uint32_t off = 0, b = 0; off < pbytes; off += per, ++b)
                    bulk_load(dst + Cfg::kABytes + b * param_stride<T>(),
                              static_cast<const uint8_t *>(psrc) + off, per, bar_full + 8 * s);
            }
        }
        // Do not leave while loads into this CTA's shared memory may be in
        // flight: wait (bounded) for the last ring's worth of them.
        for (int64_t k = (it > STAGES ? it - STAGES : 0); k < it; ++k)
            (void)mbar_wait(bar_full + 8 * static_cast<int>(k % STAGES),
                            static_cast<uint32_t>((k / STAGES) & 1));
        return;
    }

    // ---------------- consumers ----------------
    const int cw = warp;
    const int h = lane & 1, rlo = (lane >> 1) & 3, box = (lane >> 3) & 1, rhi = (lane >> 4) & 1;
    int64_t it = 0;
    for (TileWalk tw(static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x),
                             static_cast<int>(p.ncol_tiles));
             tw.rt < p.nrow_tiles; tw.next(), ++it) {
        const int s = static_cast<int>(it % STAGES);
        const uint32_t ph = static_cast<uint32_t>((it / STAGES) & 1);
        const int64_t rt = tw.rt, ct = tw.ct;
        if (!mbar_wait(bar_full + 8 * s, ph)) {
            fail_items<BR>(p, rt * p.ncol_tiles + ct, lane, cw);
            return;
        }
        const int64_t j = ct * 4 + box * 2 + h;
        const uint32_t stage = base + s * Cfg::kStageBytes + box * Cfg::kBoxBytes;
        const uint32_t prm = base + s * Cfg::kStageBytes + Cfg::kABytes +
                             (box * 2 + h) * param_stride<T>();
#pragma unroll 1
        for (int g = cw; g < BR / 8; g += kConsumerWarps) {
            const int r = g * 8 + rhi * 4 + rlo;
            const uint32_t rowaddr = stage + r * 128;
            uint4 w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = lds128(rowaddr + ((((h << 2) | k) ^ (r & 7)) << 4));
            const bool last = g + kConsumerWarps >= BR / 8;

            const int64_t row = rt * BR + r;
            if (j >= p.nb) {
                // block-column padding of the tiled scale layout
                if (p.sf_layout != KQ_SF_ROWMAJOR) store_scale(p, row, j, 0u);
                if (last) mbar_arrive(bar_empty + 8 * s);
                continue;
            }
            float2 Y[16];
            if (p.in_f16) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    Y[4 * k + 0] = make_float2(f16_lo(w[k].x), f16_hi(w[k].x));
                    Y[4 * k + 1] = make_float2(f16_lo(w[k].y), f16_hi(w[k].y));
                    Y[4 * k + 2] = make_float2(f16_lo(w[k].z), f16_hi(w[k].z));
                    Y[4 * k + 3] = make_float2(f16_lo(w[k].w), f16_hi(w[k].w));
                }
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    Y[4 * k + 0] = make_float2(bf16_lo(w[k].x), bf16_hi(w[k].x));
                    Y[4 * k + 1] = make_float2(bf16_lo(w[k].y), bf16_hi(w[k].y));
                    Y[4 * k + 2] = make_float2(bf16_lo(w[k].z), bf16_hi(w[k].z));
                    Y[4 * k + 3] = make_float2(bf16_lo(w[k].w), bf16_hi(w[k].w));
                }
            }
            apply_transform<T>(Y, prm);
            if (p.y_debug != nullptr && row < p.m) {
                float *yd = p.y_debug + row * p.d + j * 32;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    stg_f4(yd + 4 * k, make_float4(Y[2 * k].x, Y[2 * k].y, Y[2 * k + 1].x,
                                                   Y[2 * k + 1].y));
            }
            uint32_t byte;
            const uint4 codes = quantize_block(Y, byte);
            if (row < p.m) stg128_cs(p.q + row * p.ldq + j * 16, codes);
            store_scale(p, row, j, byte);
            // Release the stage only after this item's results are stored:
            // the stores consume the loaded words, so the reads are complete.
            if (last) mbar_arrive(bar_empty + 8 * s);
        }
    }
}

// ---------------------------------------------------------------------------
// launch configuration

struct KernelSlot {
    std::once_flag once[64];
    int occupancy[64] = {};
    cudaError_t err[64] = {};
};

template <int T, int BR, int STAGES>
kq_status launch_one(const CUtensorMap &map, QuantParams p, int sm_count, cudaStream_t stream)
{
    using Cfg = TileCfg<T, BR, STAGES>;
    auto kern = quant_tma_kernel<T, BR, STAGES>;
    static KernelSlot slot;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KQ_ERR_CUDA;
    std::call_once(slot.once[dev], [&] {
        slot.err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg::kSmemBytes);
        if (slot.err[dev] == cudaSuccess)
            slot.err[dev] = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &slot.occupancy[dev], kern, kThreads, Cfg::kSmemBytes);
    });
    if (slot.err[dev] != cudaSuccess || slot.occupancy[dev] < 1) return KQ_ERR_CUDA;
    p.nrow_tiles = (p.m_rows + BR - 1) / BR;
    p.ntiles = p.nrow_tiles * p.ncol_tiles;
    if (p.ntiles == 0) return KQ_OK;
    const int64_t resident = static_cast<int64_t>(slot.occupancy[dev]) * sm_count;
    const int grid = static_cast<int>(std::min<int64_t>(p.ntiles, resident));
    if (!tiles_fit_int32(p, grid)) return KQ_ERR_SHAPE;
    return launch_pdl(kern, grid, kThreads, Cfg::kSmemBytes, stream, map, p);
}

template <int T>
kq_status launch_t(const CUtensorMap &map, const QuantParams &p, int sm_count,
                   cudaStream_t stream, int br)
{
    if (br == 64) return launch_one<T, 64, 6>(map, p, sm_count, stream);
    return launch_one<T, 128, 3>(map, p, sm_count, stream);
}

}  // namespace

kq_status launch_quant_tma(Transform t, const uint16_t *A, int64_t lda, const QuantParams &p,
                           cudaStream_t stream)
{
    DeviceInfo info;
    kq_status st = device_info(info);
    if (st != KQ_OK) return st;
    // Rows per tile: the one whose last wave leaves the fewest idle rows
    // (2 resident CTAs per SM for both shapes).
    const int64_t slots = 2LL * info.sm_count;
    auto makespan = [&](int64_t br) {
        const int64_t tiles = ((p.m_rows + br - 1) / br) * p.ncol_tiles;
        return ((tiles + slots - 1) / slots) * br;
    };
    const int br = makespan(64) < makespan(128) ? 64 : 128;
    CUtensorMap map;
    st = make_tensor_map_2d_bf16(&map, A, p.m, p.d, lda, 64, static_cast<uint32_t>(br));
    if (st != KQ_OK) return st;
    switch (t) {
    case kKron: return launch_t<kKron>(map, p, info.sm_count, stream, br);
    case kDiag: return launch_t<kDiag>(map, p, info.sm_count, stream, br);
    case kHadamard: return launch_t<kHadamard>(map, p, info.sm_count, stream, br);
    default: return launch_t<kIdentity>(map, p, info.sm_count, stream, br);
    }
}

}  // namespace kq
