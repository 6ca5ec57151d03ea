// Tensor-core variant of the KroQuant block transform (mma.sync, sm_103a).
//
// "KroQuant: Kronecker-Structured Block Transforms for Efficient Post-
// Training Quantization of Diffusion Transformers", eq. (5): with
// K_j = G1 (x) K'_j, K'_j = G2 (x) G3 (x) G4 (x) G5 (16 x 16), the row
// transform y = a . K_j of a 32-channel block splits over the two 16-channel
// halves a_0, a_1 (channel bit 4, the bit G1 acts on, eq. 12):
//     Z_h = a_h . K'_j                      (two dense 16x16 products)
//     y_0 = G1[0][0] Z_0 + G1[1][0] Z_1,    y_1 = G1[0][1] Z_0 + G1[1][1] Z_1.
// The dense products run on the tensor cores (mma.sync m16n8k16, bf16
// operands, fp32 accumulate) against K'_j pre-expanded by kq_expand_blocks
// as three bf16 terms hi + mid + lo (together exact to ~2^-24 relative;
// the activations are exact in bf16); the G1 stage runs in fp32 on the
// accumulators.  Expanding only G2..G5 halves the tensor work of the dense
// 32x32 form (48 instead of 96 MACs per element) and quarters the operand
// bytes, which keeps the tensor pipe well below its mma.sync peak at HBM
// speed.
//
// Data path: the same persistent TMA ring as the butterfly kernels (tiles of
// BR rows x 128 channels, two 128B-swizzled boxes); the producer also copies
// the tile's four operand records (1552 bytes per block) into the stage with
// one bulk copy, so operand fetches ride the same pipeline.  Consumer warp w
// owns block (w & 3) of the tile for half of its rows; A fragments come from
// shared memory with ldmatrix (conflict-free under the swizzle).
//
// Operand record of block j (kq_expand_blocks, KQ_K_BF16X3):
//   bytes [0, 1536): uint32 frag[lane 0..31][12]: term t (0 hi, 1 mid, 2 lo),
//     n-tile nt (0, 1), register r (0, 1) at index (t*2 + nt)*2 + r; the
//     registers are the m16n8k16 B fragments of B_t, where
//     B_t[k][8 nt + n] = term_t(K'[k][4 (n >> 1) + 2 nt + (n & 1)]):
//     the column order makes the accumulator thread with lane % 4 == q hold
//     output channels 4q..4q+3 of each half (its G1 partners included);
//   bytes [1536, 1552): G1 as fp32 (g00, g01, g10, g11).
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int kRecordBytes = static_cast<int>(kMmaRecordBytes);
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;

template <int BR, int STAGES>
struct MmaCfg {
    static constexpr int kBoxBytes = BR * 128;
    static constexpr int kABytes = 2 * kBoxBytes;
    static constexpr int kBBytes = 7168;                 // 4 records, padded to 1 KB
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSmemBytes = STAGES * kStageBytes + 1024 + 2 * STAGES * 8;
    static_assert(BR % 32 == 0 && BR <= 256, "box rows");
    static_assert(4 * kRecordBytes <= kBBytes, "operand records");
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&a)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void store_scale_m(const QuantParams &p, int64_t row, int64_t j,
                                              uint32_t byte)
{
    if (p.sf_layout == KQ_SF_ROWMAJOR) {
        if (row < p.m) p.sf[row * p.nb + j] = static_cast<uint8_t>(byte);
    } else {
        p.sf[sf_blocked_offset(row, j, p.ncb)] = static_cast<uint8_t>(byte);
    }
}

template <int BR>
__device__ void fail_items_m(const QuantParams &p, int64_t tile, int warp, int lane)
{
    const int b = warp & 3, part = warp >> 2;
    for (; tile < p.ntiles; tile += gridDim.x) {
        const int64_t rt = tile / p.ncol_tiles, ct = tile % p.ncol_tiles;
        const int64_t j = ct * 4 + b;
        if (j >= p.nb) continue;
        for (int r = lane; r < BR / 2; r += 32) {
            const int64_t row = rt * BR + part * (BR / 2) + r;
            if (row < p.m_rows) store_scale_m(p, row, j, 0xFFu);
        }
    }
}

template <int BR, int STAGES>
__global__ void __launch_bounds__(kThreads, 2)
    quant_mma_kernel(const __grid_constant__ CUtensorMap tmA, const QuantParams p,
                     const uint8_t *__restrict__ records)
{
    using Cfg = MmaCfg<BR, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
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
            const int64_t left = p.nb - ct * 4;
            const int64_t nrec = left < 4 ? left : 4;
            const uint32_t rec_bytes = static_cast<uint32_t>(nrec * kRecordBytes);
            mbar_arrive_expect_tx(bar_full + 8 * s, Cfg::kABytes + rec_bytes);
            tma_load_2d(dst, &tmA, static_cast<int32_t>(ct * 128), static_cast<int32_t>(rt * BR),
                        bar_full + 8 * s, pol);
            tma_load_2d(dst + Cfg::kBoxBytes, &tmA, static_cast<int32_t>(ct * 128 + 64),
                        static_cast<int32_t>(rt * BR), bar_full + 8 * s, pol);
            bulk_load(dst + Cfg::kABytes, records + ct * 4 * kRecordBytes, rec_bytes,
                      bar_full + 8 * s);
        }
        for (int64_t k = (it > STAGES ? it - STAGES : 0); k < it; ++k)
            (void)mbar_wait(bar_full + 8 * static_cast<int>(k % STAGES),
                            static_cast<uint32_t>((k / STAGES) & 1));
        return;
    }

    // ---------------- consumers ----------------
    const int b = warp & 3;               // block of the tile
    const int part = warp >> 2;           // which half of the tile's rows
    const int bb = b & 1, box = b >> 1;   // block within its TMA box, the box
    const int g = lane >> 2, q = lane & 3;
    // ldmatrix lane -> (row within the 16-row group, 8-channel chunk)
    const int lm_row = ((lane >> 3) & 1) * 8 + (lane & 7);
    const int lm_kc = lane >> 4;
    int64_t it = 0;
    for (TileWalk tw(static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x),
                             static_cast<int>(p.ncol_tiles));
             tw.rt < p.nrow_tiles; tw.next(), ++it) {
        const int s = static_cast<int>(it % STAGES);
        const uint32_t ph = static_cast<uint32_t>((it / STAGES) & 1);
        const int64_t rt = tw.rt, ct = tw.ct;
        if (!mbar_wait(bar_full + 8 * s, ph)) {
            fail_items_m<BR>(p, rt * p.ncol_tiles + ct, warp, lane);
            return;
        }
        const int64_t j = ct * 4 + b;
        const uint32_t stage = base + s * Cfg::kStageBytes;
        if (j >= p.nb) {
            // block-column padding of the tiled scale layout
            if (p.sf_layout != KQ_SF_ROWMAJOR) {
                for (int r = lane; r < BR / 2; r += 32)
                    store_scale_m(p, rt * BR + part * (BR / 2) + r, j, 0u);
            }
            mbar_arrive(bar_empty + 8 * s);
            continue;
        }
        // operand record: B fragments of the three terms and G1
        const uint32_t rec = stage + Cfg::kABytes + b * kRecordBytes;
        uint32_t bf[12];
        {
            const uint4 r0 = lds128(rec + lane * 48), r1 = lds128(rec + lane * 48 + 16),
                        r2 = lds128(rec + lane * 48 + 32);
            bf[0] = r0.x; bf[1] = r0.y; bf[2] = r0.z; bf[3] = r0.w;
            bf[4] = r1.x; bf[5] = r1.y; bf[6] = r1.z; bf[7] = r1.w;
            bf[8] = r2.x; bf[9] = r2.y; bf[10] = r2.z; bf[11] = r2.w;
        }
        const uint4 g1u = lds128(rec + 1536);
        const float g00 = __uint_as_float(g1u.x), g01 = __uint_as_float(g1u.y);
        const float g10 = __uint_as_float(g1u.z), g11 = __uint_as_float(g1u.w);
        const uint32_t boxbase = stage + box * Cfg::kBoxBytes;

#pragma unroll 1
        for (int grp = 0; grp < BR / 32; ++grp) {
            const int row0 = part * (BR / 2) + grp * 16;
            // A fragments of the two 16-channel halves
            uint32_t a[2][4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = row0 + lm_row;
                const int chunk = bb * 4 + h * 2 + lm_kc;
                ldmatrix_x4(boxbase + r * 128 + ((chunk ^ (r & 7)) << 4), a[h]);
            }
            float z[2][2][4];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) z[h][nt][0] = z[h][nt][1] = z[h][nt][2] = z[h][nt][3] = 0.f;
#pragma unroll
            for (int t = 0; t < 3; ++t)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        mma_bf16(z[h][nt], a[h], bf[(t * 2 + nt) * 2], bf[(t * 2 + nt) * 2 + 1]);

            // two rows per thread: g and g + 8
#pragma unroll
            for (int rs = 0; rs < 2; ++rs) {
                float v[2][2][2];   // [output half][nt][e] -> channel 16 h + 4 q + 2 nt + e
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float z0 = z[0][nt][2 * rs + e], z1 = z[1][nt][2 * rs + e];
                        v[0][nt][e] = fmaf(z1, g10, z0 * g00);
                        v[1][nt][e] = fmaf(z1, g11, z0 * g01);
                    }
                float amax = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        amax = fmaxf(amax, fmaxf(fabsf(v[h][nt][0]), fabsf(v[h][nt][1])));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                const uint32_t byte = e8m0_byte(amax);
                const float sc = inv_scale(byte);
                const int64_t row = rt * BR + row0 + g + 8 * rs;
                if (p.y_debug != nullptr && row < p.m) {
                    float *yd = p.y_debug + row * p.d + j * 32 + 4 * q;
                    stg_f4(yd, make_float4(v[0][0][0], v[0][0][1], v[0][1][0], v[0][1][1]));
                    stg_f4(yd + 16, make_float4(v[1][0][0], v[1][0][1], v[1][1][0], v[1][1][1]));
                }
                // bytes: 2q, 2q+1 (channels 4q..4q+3) and 8+2q, 9+2q (16+4q..)
                const uint32_t w = e2m1x8(v[0][0][0] * sc, v[0][0][1] * sc, v[0][1][0] * sc,
                                          v[0][1][1] * sc, v[1][0][0] * sc, v[1][0][1] * sc,
                                          v[1][1][0] * sc, v[1][1][1] * sc);
                const uint32_t lo16 = w & 0xffffu, hi16 = w >> 16;
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, (q & 1) ? lo16 : hi16, 1);
                const uint32_t word = (q & 1) ? (recv | (hi16 << 16)) : (lo16 | (recv << 16));
                const int wi = (q & 1) ? 2 + (q >> 1) : (q >> 1);
                if (row < p.m) {
                    uint32_t *dstq = reinterpret_cast<uint32_t *>(p.q + row * p.ldq + j * 16) + wi;
                    asm volatile("st.global.cs.b32 [%0], %1;" ::"l"(dstq), "r"(word) : "memory");
                }
                if (q == 0) store_scale_m(p, row, j, byte);
            }
        }
        mbar_arrive(bar_empty + 8 * s);
    }
}

struct Slot {
    std::once_flag once[64];
    int occupancy[64] = {};
    cudaError_t err[64] = {};
};

template <int BR, int STAGES>
kq_status launch_mma(const CUtensorMap &map, QuantParams p, const uint8_t *records,
                     int sm_count, cudaStream_t stream)
{
    using Cfg = MmaCfg<BR, STAGES>;
    auto kern = quant_mma_kernel<BR, STAGES>;
    static Slot slot;
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
    return launch_pdl(kern, grid, kThreads, Cfg::kSmemBytes, stream, map, p, records);
}

// ---- operand records (kq_expand_blocks, KQ_K_BF16X3) ------------------------------

__device__ __forceinline__ double kron_tail(const float *f, int r, int c)
{
    // K'[r][c] = prod_{k=2..5} G_k[bit_{5-k}(r)][bit_{5-k}(c)], r, c in 0..15
    double x = 1.0;
#pragma unroll
    for (int k = 2; k <= 5; ++k) {
        const int bit = 5 - k;
        x *= static_cast<double>(f[(k - 1) * 4 + ((r >> bit) & 1) * 2 + ((c >> bit) & 1)]);
    }
    return x;
}

__device__ __forceinline__ uint16_t bf16_term(double x, int t)
{
    // term t of the three-term bf16 split x = hi + mid + lo
    double rem = x;
    __nv_bfloat16 v = __double2bfloat16(rem);
    for (int i = 0; i < t; ++i) {
        rem -= static_cast<double>(__bfloat162float(v));
        v = __double2bfloat16(rem);
    }
    return __bfloat16_as_ushort(v);
}

__global__ void mma_records_kernel(const float *__restrict__ factors, int64_t nb,
                                   uint8_t *__restrict__ out)
{
    const int64_t n = nb * (32 * 12 + 4);
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t j = idx / (32 * 12 + 4);
        const int w = static_cast<int>(idx % (32 * 12 + 4));
        const float *f = factors + j * 20;
        uint32_t *rec = reinterpret_cast<uint32_t *>(out + j * kRecordBytes);
        if (w >= 32 * 12) {                       // G1 entries
            rec[32 * 12 + (w - 32 * 12)] = __float_as_uint(f[w - 32 * 12]);
            continue;
        }
        const int lane = w / 12, slot = w % 12;
        const int t = slot / 4, nt = (slot / 2) & 1, reg = slot & 1;
        const int n = lane >> 2, q = lane & 3;
        const int col = 4 * (n >> 1) + 2 * nt + (n & 1);   // K' column of MMA column 8 nt + n
        const int k0 = 2 * q + 8 * reg;
        const uint16_t lo = bf16_term(kron_tail(f, k0, col), t);
        const uint16_t hi = bf16_term(kron_tail(f, k0 + 1, col), t);
        rec[w] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
}

// Records of the tcgen05 variant: per block, the dense K_j = G1 (x) K'_j
// (entries in fp64, eq. 12) as three bf16 terms, arranged as the B operands
// of the block's two K = 16 steps.  Step h (input channels 16 h .. 16 h + 15)
// occupies bytes [3072 h, 3072 h + 3072): B^T with n = 32 t + c (term t,
// output channel c) and k = input channel - 16 h, in the no-swizzle K-major
// layout -- 8 x 16-byte core matrices, core (n / 8, k / 8) at
// (n / 8) * 256 + (k / 8) * 128, row n % 8 at 16 B, element k % 8 at 2 B.
__global__ void umma_records_kernel(const float *__restrict__ factors, int64_t nb,
                                    uint8_t *__restrict__ out)
{
    constexpr int kWords = static_cast<int>(kUmmaRecordBytes / 4);   // element pairs
    const int64_t n = nb * kWords;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t j = idx / kWords;
        const int w = static_cast<int>(idx % kWords);
        const float *f = factors + j * 20;
        uint8_t *rec = out + j * kUmmaRecordBytes;
        const int h = w / 768, nn = (w / 8) % 96, kp = w % 8;
        const int t = nn / 32, c = nn % 32, k0 = 2 * kp, r0 = 16 * h + k0;
        // K_j[r][c] = G1[bit4(r)][bit4(c)] * K'_j[r % 16][c % 16]
        const double g0 = static_cast<double>(f[((r0 >> 4) & 1) * 2 + ((c >> 4) & 1)]);
        const uint16_t e0 = bf16_term(g0 * kron_tail(f, r0 & 15, c & 15), t);
        const uint16_t e1 = bf16_term(g0 * kron_tail(f, (r0 + 1) & 15, c & 15), t);
        const int off = h * 3072 + (nn >> 3) * 256 + (k0 >> 3) * 128 + (nn & 7) * 16 + (k0 & 7) * 2;
        *reinterpret_cast<uint32_t *>(rec + off) = static_cast<uint32_t>(e0) |
                                                   (static_cast<uint32_t>(e1) << 16);
    }
}

}  // namespace

kq_status launch_quant_mma(const uint16_t *A, int64_t lda, const void *K_expanded,
                           const QuantParams &p, cudaStream_t stream)
{
    DeviceInfo info;
    kq_status st = device_info(info);
    if (st != KQ_OK) return st;
    constexpr int BR = 64;
    CUtensorMap map;
    st = make_tensor_map_2d_bf16(&map, A, p.m, p.d, lda, 64, BR);
    if (st != KQ_OK) return st;
    // the mma.sync records follow the nb tcgen05 records
    return launch_mma<BR, 4>(map, p,
                             static_cast<const uint8_t *>(K_expanded) + p.nb * kUmmaRecordBytes,
                             info.sm_count, stream);
}

// K_expanded (KQ_K_BF16X3) = [nb tcgen05 records][nb mma.sync records].
kq_status launch_mma_records(const float *factors, int64_t nb, void *out, cudaStream_t stream)
{
    uint8_t *o = static_cast<uint8_t *>(out);
    const int64_t work_u = nb * (kUmmaRecordBytes / 4);
    umma_records_kernel<<<static_cast<int>(std::min<int64_t>((work_u + 255) / 256, 4096)), 256, 0,
                          stream>>>(factors, nb, o);
    const int64_t work = nb * (32 * 12 + 4);
    mma_records_kernel<<<static_cast<int>(std::min<int64_t>((work + 255) / 256, 4096)), 256, 0,
                         stream>>>(factors, nb, o + nb * kUmmaRecordBytes);
    return check_launch();
}

}  // namespace kq
