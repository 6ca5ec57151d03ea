// KroQuant quantizer with the block transform on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in TMEM), sm_103a.
//
// "KroQuant: Kronecker-Structured Block Transforms for Efficient Post-
// Training Quantization of Diffusion Transformers", eq. (5) and (12): the
// row transform y = a . K_j of a 32-channel block runs as tcgen05.mma (bf16
// operands, fp32 accumulation in TMEM) against the dense 32 x 32 K_j =
// G1 (x) G2 (x) G3 (x) G4 (x) G5, expanded once per layer by kq_expand_blocks
// (entries in fp64) as three bf16 terms hi + mid + lo (exact to about 2^-24
// relative; the activations are exact in bf16).  The three terms sit side by
// side along N: per block two M = 128, N = 96, K = 16 MMAs (one per
// 16-channel input half, accumulating) read each A slice from shared memory
// once, and the epilogue adds the three partial results.
// Alternatives measured on GB300 and dropped: one MMA per term re-reads A
// three times from shared memory; copying A into TMEM once (tcgen05.cp) and
// accumulating the terms there with 12 N = 32 MMAs per tile frees the
// epilogue but the longer tcgen05 instruction stream (about 150 cycles per
// instruction to issue) then limits the tile rate; keeping G1 out of the
// operands and applying it on the CUDA cores loads the epilogue, which
// limits this kernel; and a separate, shallower ring for the operand records
// (more activation tiles in flight) was no faster.
// The MXFP4 encoding runs on the CUDA cores after the accumulators are read
// back with tcgen05.ld (one thread = one row of a 32-channel block, all 32
// values in registers).
//
// Roles in a CTA (one CTA per SM, persistent over tiles of 128 rows x 64
// channels = 2 blocks = one 128B-swizzled TMA box):
//   warp 0      TMA producer: the A box + one bulk copy of the tile's two
//               operand records (6 KB each: the three bf16 terms of K_j in
//               the no-swizzle K-major layout) into a STAGES-deep
//               shared-memory ring;
//   warps 1-2   MMA issuers, one per accumulator buffer (2 x 192 TMEM columns,
//               allocated by warp 1): warp 1 + m takes the CTA's tiles with
//               it % 2 == m, so two tiles are in flight through the tensor
//               core; one lane issues the tile's 4 MMAs and commits them to the
//               ring's empty barrier and to the accumulator's full barrier;
//   warps 3-18  epilogue, two groups of 8 warps taking alternate tiles (and
//               accumulator buffers): warp w reads TMEM lanes 32 (w % 4)..+31
//               (rows) of one block, sums the terms and quantizes; the two
//               warps of a 32-row quarter put their 16 bytes of codes per row
//               side by side in a shared staging buffer, and one TMA store
//               writes the quarter's 32 rows x 32 bytes (a thread owns a row,
//               so direct 16-byte stores from a warp would touch 32 rows and
//               clog the memory pipe; whole 32-byte rows also halve the L2
//               write transactions of 16-byte ones).
// With DUAL, the kernel also writes the 16-bit side output A T that feeds
// the low-rank branch of eq. (11) ("KroQuant ...", App. D "Quantization":
// those activations stay in 16 bits; Sec. 3.5.1 K1 casts y to the input
// dtype): the epilogue rounds y to bf16 and writes it over the tile's
// activations in its ring stage (the MMAs have read them; same 128 x 64
// shape and 128B swizzle), and one TMA store per tile sends it to HBM.  The
// ring stage is then released by the epilogue, once that store has read it,
// instead of by the MMA commit.
// With K2 ("KroQuant ...", Sec. 3.5.1 K2 and App. B), no operand records come
// from memory: the epilogue groups write them into the ring stages from the
// raw factors (build_record_rows).  With PAIR, the CTA walks its tiles by
// pairs of row tiles of one column, which share one set of records built
// once (PairWalk).
// Every wait is bounded in time (one second, or the shorter limit of the
// verification hook); a timed-out epilogue writes the E8M0 NaN byte 0xFF as
// the scale of the blocks it could not finish (and bf16 NaNs into the side
// output).
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kMmaWarps = 2;                   // one per accumulator buffer
constexpr int kFirstEpiWarp = 1 + kMmaWarps;
constexpr int kThreadsU = (kFirstEpiWarp + kEpiWarps) * 32;
constexpr int kBR = 128;                       // rows per tile (= MMA M)
constexpr int kBlockCols = 96;                 // per block: 3 terms x 32 outputs
constexpr int kAccCols = 2 * kBlockCols;       // fp32 columns per accumulator buffer
constexpr int kTmemCols = 512;                 // 2 buffers (384 columns), power of two

template <int STAGES>
struct UCfg {
    static constexpr int kABytes = kBR * 128;                 // 128 rows x 64 bf16 = 16 KB
    static constexpr int kBOff = kABytes;                     // operand records
    static constexpr int kRecBytes = static_cast<int>(kUmmaRecordBytes);   // 3 terms of K_j
    static constexpr int kStageBytes = kABytes + 2 * kRecBytes;          // 28 KB
    // after the ring: barriers + TMEM base (1 KB), 1 KB spare, code staging
    // for the TMA stores: per pair of epilogue warps (the two blocks of one
    // 32-row quarter) 3 buffers of 32 rows x 32 B
    static constexpr int kBarOff = STAGES * kStageBytes;
    static constexpr int kStgOff = kBarOff + 2048;
    static constexpr int kStgBytes = 32 * 32;
    static constexpr int kStgBufs = 3;
    // and per pair and buffer the b = 1 warp's 32 scale bytes (tiled layout)
    static constexpr int kSfStgOff = kStgOff + (kEpiWarps / 2) * kStgBufs * kStgBytes;
    static constexpr int kSmemBytes =
        kSfStgOff + (kEpiWarps / 2) * kStgBufs * 32 + 1024;   // + alignment slack
    static_assert(kStageBytes % 1024 == 0, "stage alignment");
    // The two MMA issuers take alternate tiles and wait on the ring's full
    // barriers by phase parity.  With an even ring every stage is always
    // consumed by the same issuer, which has itself consumed the stage's
    // previous phase; with an odd ring an issuer could wait on phase k of a
    // stage whose phase k - 1 (the other issuer's tile) is still in flight,
    // and the parity test would pass on phase k - 2.
    static_assert(STAGES % 2 == 0, "each ring stage must belong to one MMA issuer");
};

// ---- tcgen05 wrappers ---------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
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

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), descriptor version 1, swizzle mode (0 none, 2 128B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle)
{
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>(lbo >> 4) << 16) | (static_cast<uint64_t>(sbo >> 4) << 32) |
           (1ull << 46) | (static_cast<uint64_t>(swizzle) << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = 96 (three 32-column terms), M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((96u >> 3) << 17) |
                            ((128u >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
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
}

// Waits until this thread's earlier tcgen05.ld results are in registers.
__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void store_scale_u(const QuantParams &p, int64_t row, int64_t j,
                                              uint32_t byte)
{
    if (p.sf_layout == KQ_SF_ROWMAJOR) {
        if (row < p.m) p.sf[row * p.nb + j] = static_cast<uint8_t>(byte);
    } else {
        p.sf[sf_blocked_offset(row, j, p.ncb)] = static_cast<uint8_t>(byte);
    }
}

// Walk over a CTA's tiles by pairs of row tiles: super tile (rtp, ct) in
// row-major order over ceil(nrow / 2) x ncol, the CTA's super tiles first,
// first + step, ...; within one, rows 2 rtp + h.  half >= 0 walks that half
// only, half < 0 both halves in turn (h = 0, then 1).  Neighbouring CTAs
// still read neighbouring columns of the same rows, as the row-major walk.
struct PairWalk {
    TileWalk sw;
    int h, rt, ct;
    bool fixed;
    __device__ __forceinline__ PairWalk(int first, int step, int ncol, int half)
        : sw(first, step, ncol), h(half < 0 ? 0 : half), rt(2 * sw.rt + h), ct(sw.ct), fixed(half >= 0)
    {
    }
    __device__ __forceinline__ void next()
    {
        if (!fixed && h == 0) {
            h = 1;
        } else {
            if (!fixed) h = 0;
            sw.next();
        }
        rt = 2 * sw.rt + h;
        ct = sw.ct;
    }
};

// K2 (the tensor-core path without expanded records in memory): eight
// entries of K_j -- rows 8 g .. 8 g + 7, column c -- as the three bf16 terms,
// written into a tile's record area in the MMA operand layout (see
// umma_records_kernel).  Entries by eq. (12), K_j[r][c] =
// prod_k G_k[bit_{5-k}(r)][bit_{5-k}(c)], as fp32 products.  Each fp32 value
// k splits exactly into three bf16 terms by truncation: hi = the top 16 bits
// of k, mid = the top 16 bits of k - hi (exact), lo = k - hi - mid (exact,
// and at most 8 significant bits, so exact in bf16).  The eight entries of a
// term form one 16-byte row of a core matrix; a warp with c = lane fills
// 4 x 128 contiguous bytes per term (no bank conflicts).
__device__ __forceinline__ void build_record_rows(uint32_t rec, const float *__restrict__ f, int c,
                                                  int g)
{
    // the ten factor entries column c needs: G_k[row][bit_{4-k}(c)], k = 0..4
    // for G1..G5 (f holds the block's raw factors, [5][2][2])
    float col[5][2];
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const int bit = (c >> (4 - k)) & 1;
        col[k][0] = __ldg(f + 4 * k + bit);
        col[k][1] = __ldg(f + 4 * k + 2 + bit);
    }
    // r = 8 g + i: bit 4 of r = g >> 1, bit 3 = g & 1, bits 2..0 = i (g is a
    // run-time value: selects, not an indexed array, keep col in registers)
    const float P = ((g >> 1) ? col[0][1] : col[0][0]) * ((g & 1) ? col[1][1] : col[1][0]);
    const float2 P2 = make_float2(P, P), c4 = make_float2(col[4][0], col[4][1]);
    uint32_t w[3][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {       // entries i = 2q, 2q + 1: bit 0 of i = G5's row
        const float s = col[2][q >> 1] * col[3][q & 1];
        const float2 kv = __fmul2_rn(P2, __fmul2_rn(make_float2(s, s), c4));
        const uint32_t b0 = __float_as_uint(kv.x), b1 = __float_as_uint(kv.y);
        const float2 hi = make_float2(__uint_as_float(b0 & 0xffff0000u), __uint_as_float(b1 & 0xffff0000u));
        const float2 r = __fadd2_rn(kv, make_float2(-hi.x, -hi.y));                 // exact
        const uint32_t m0 = __float_as_uint(r.x) & 0xffff0000u, m1 = __float_as_uint(r.y) & 0xffff0000u;
        const float2 lo = __fadd2_rn(r, make_float2(-__uint_as_float(m0), -__uint_as_float(m1)));  // exact
        // element 2q in the low half of each word
        w[0][q] = __byte_perm(b0, b1, 0x7632);
        w[1][q] = __byte_perm(m0, m1, 0x7632);
        w[2][q] = __byte_perm(__float_as_uint(lo.x), __float_as_uint(lo.y), 0x7632);
    }
    // step h = g >> 1 (input channels 16 h..), core column g & 1, row c % 8
    const uint32_t off = rec + (g >> 1) * 3072 + (g & 1) * 128 + (c & 7) * 16;
#pragma unroll
    for (int t = 0; t < 3; ++t)
        sts128(off + ((32 * t + c) >> 3) * 256, make_uint4(w[t][0], w[t][1], w[t][2], w[t][3]));
}

template <int STAGES, bool DEBUG, bool DUAL, bool K2, bool PAIR>
__global__ void __launch_bounds__(kThreadsU, 1)
    quant_umma_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmAT, const QuantParams p,
                      const uint8_t *__restrict__ records)
{
    using Cfg = UCfg<STAGES>;
    static_assert(!PAIR || (K2 && !DUAL), "tile pairs share the records K2 builds");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    const uint32_t bar = base + Cfg::kBarOff;
    const uint32_t bar_full = bar;                        // [STAGES]
    const uint32_t bar_empty = bar + 8 * STAGES;          // [STAGES]
    const uint32_t bar_acc_full = bar + 16 * STAGES;      // [2]
    const uint32_t bar_acc_empty = bar_acc_full + 16;     // [2]
    const uint32_t tmem_slot = bar_acc_empty + 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint64_t lim = p.wait_limit_ns;

    // PAIR (K2 only): the CTA walks its tiles by pairs of row tiles of one
    // column, tile it = 2 P + h; the pair shares one set of operand records,
    // built once into the ring stage of its first tile, 2 P % STAGES (an
    // even stage; the odd stages hold no records).  A pair of an odd row
    // count's last row is completed by a tile past the last row: its loads
    // fill with zeros and its stores are clipped or skipped.
    const int nrp = static_cast<int>((p.nrow_tiles + 1) / 2);
    auto valid = [&](const auto &w) {
        if constexpr (PAIR) return w.sw.rt < nrp;
        else return w.rt < p.nrow_tiles;
    };
    // this CTA's tiles (half < 0: all of them in order; else tiles it % 2 ==
    // half, in order)
    auto walker = [&](int half) {
        if constexpr (PAIR) {
            return PairWalk(static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x),
                            static_cast<int>(p.ncol_tiles), half);
        } else if (half < 0) {
            return TileWalk(static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x),
                            static_cast<int>(p.ncol_tiles));
        } else {
            return TileWalk(static_cast<int>(blockIdx.x + half * gridDim.x),
                            static_cast<int>(2 * gridDim.x), static_cast<int>(p.ncol_tiles));
        }
    };

    // The producer (thread 0) walks the CTA's tiles in order; it loads the
    // activation box and the operand records of tile `it` into ring stage
    // it % STAGES.  (Its work per tile sits on the pipeline's critical path:
    // each stage is reissued as soon as its MMAs have read it, so the time
    // from that release to the next load decides how much data is in
    // flight.  Measured on GB300: a generic tile-index fetch with an integer
    // division per tile made the FLUX FFN-down launch 13 % slower.)
    auto pw = walker(-1);
    int64_t pit = 0;
    uint64_t pol = 0;
    // verification hook: the position in this CTA's walk of the tile whose
    // loads are never issued (-1: none)
    const int64_t skip_it =
        (p.skip_tile >= 0 && p.skip_tile % gridDim.x == blockIdx.x) ? p.skip_tile / gridDim.x : -1;
    auto issue_tile = [&]() {
        const int s = static_cast<int>(pit % STAGES);
        const uint32_t dst = base + s * Cfg::kStageBytes;
        const int64_t left = p.nb - pw.ct * 2;          // < 1 on padding tiles
        // K2: the records are built in the stage by the epilogue warps
        const uint32_t rbytes = K2 ? 0u :
            static_cast<uint32_t>((left < 0 ? 0 : (left < 2 ? left : 2)) * Cfg::kRecBytes);
        mbar_arrive_expect_tx(bar_full + 8 * s, Cfg::kABytes + rbytes);
        if (pit == skip_it) {                            // the stage stays armed, never filled
            pw.next();
            ++pit;
            return;
        }
        tma_load_2d(dst, &tmA, pw.ct * 64, pw.rt * kBR, bar_full + 8 * s, pol);
        if (K2) {
        } else if (p.shared_params) {
            // one operand record for every block: a copy of it per block slot
            for (uint32_t off = 0; off + Cfg::kRecBytes <= rbytes; off += Cfg::kRecBytes)
                bulk_load(dst + Cfg::kBOff + off, records, Cfg::kRecBytes, bar_full + 8 * s);
        } else if (rbytes) {
            bulk_load(dst + Cfg::kBOff, records + static_cast<int64_t>(pw.ct) * 2 * Cfg::kRecBytes,
                      rbytes, bar_full + 8 * s);
        }
        pw.next();
        ++pit;
    };

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);              // kernel parameters: no dependency on
        tma_prefetch_desc(&tmQ);              // earlier grids
        if (DUAL) tma_prefetch_desc(&tmAT);
        for (int s = 0; s < STAGES; ++s) {
            // K2: the producer's TMA bytes and the 8 record-building warps
            // (PAIR: on the even stages only, which hold a pair's records
            // and are released by the MMAs of both its tiles)
            const bool rec = K2 && (!PAIR || s % 2 == 0);
            mbar_init(bar_full + 8 * s, rec ? 1 + kEpiWarps / 2 : 1);
            mbar_init(bar_empty + 8 * s, PAIR && s % 2 == 0 ? 2 : 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_acc_full + 8 * a, 1);        // MMA commit
            mbar_init(bar_acc_empty + 8 * a, kEpiThreads / 2);
        }
        mbar_fence_init();
        // The first tile's loads go out before the CTA-wide setup barrier
        // (TMEM allocation), so its DRAM round trip overlaps it; every other
        // thread touches the ring only after that barrier.  (Measured on
        // GB300: sending the whole first ring this early made small launches
        // slower; one tile is faster on every shape tried.)
        grid_dependency_wait();
        pol = l2_policy_evict_first();
        if (valid(pw)) issue_tile();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    uint32_t tmem_base;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(tmem_base) : "r"(tmem_slot) : "memory");
    grid_dependency_wait();

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            while (valid(pw)) {
                const int s = static_cast<int>(pit % STAGES);
                const uint32_t ph = static_cast<uint32_t>((pit / STAGES) & 1);
                if (pit >= STAGES && !mbar_wait(bar_empty + 8 * s, ph ^ 1u, lim)) break;
                issue_tile();
            }
            // The next grid may be scheduled once every CTA is this far: its
            // CTAs then take the SMs as this grid's CTAs exit, instead of
            // being launched after the last exit.  Measured on GB300 by
            // tiles per CTA: 4096 x 1152 (4) 5.15 -> 4.62 us, 4608 x 3072
            // (11) 8.57 -> 8.38 us, 4608 x 12288 (45) unchanged, but 16384 x
            // 12288 (162) +0.8 % and 65536 x 12288 (647) +3.2 %; the dual
            // kernel gained at 4 and lost 2-3 % from 45 on.
            if (p.ntiles < (DUAL ? 8 : 48) * static_cast<int64_t>(gridDim.x)) grid_dependents_launch();
            const int64_t it = pit;
            for (int64_t k = (it > STAGES ? it - STAGES : 0); k < it; ++k)
                (void)mbar_wait(bar_full + 8 * static_cast<int>(k % STAGES),
                                static_cast<uint32_t>((k / STAGES) & 1), lim);
        }
    } else if (warp < kFirstEpiWarp) {
        // ---------------- MMA issuers ----------------
        const int a = warp - 1;               // accumulator buffer; tiles with it % 2 == a
        int64_t it = a;
        bool ok = true;
        // the issuing lane, elected once (a commit tracks only the tcgen05
        // operations of its own thread)
        const bool leader = elect_one();
        for (auto tw = walker(a); valid(tw) && ok; tw.next(), it += 2) {
            const int s = static_cast<int>(it % STAGES);
            // PAIR: the second tile of a pair takes the records from the
            // first tile's stage, so it also waits for that stage's phase
            // (which cannot move on before this tile's own commit below)
            const int sr = PAIR && a == 1 ? static_cast<int>((it - 1) % STAGES) : s;
            const int64_t ct = tw.ct;
            const int64_t left = p.nb - ct * 2;
            const int nblk = static_cast<int>(left < 0 ? 0 : (left < 2 ? left : 2));
            bool w = mbar_wait(bar_full + 8 * s, static_cast<uint32_t>((it / STAGES) & 1), lim);
            if (PAIR && a == 1 && w)
                w = mbar_wait(bar_full + 8 * sr, static_cast<uint32_t>(((it - 1) / STAGES) & 1), lim);
            if (w && it >= 2)
                w = mbar_wait(bar_acc_empty + 8 * a, static_cast<uint32_t>(((it >> 1) & 1) ^ 1), lim);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            const uint32_t stage = base + s * Cfg::kStageBytes;
            const uint32_t rstage = base + sr * Cfg::kStageBytes;
            tc_fence_after();
            if (leader) {
                const uint32_t d0 = tmem_base + a * kAccCols;
                for (int b = 0; b < nblk; ++b)
                    for (int h = 0; h < 2; ++h)       // input half h: K = 16 step
                        umma_bf16(d0 + b * kBlockCols,
                                  smem_desc(stage + 64 * b + 32 * h, 16, 1024, 2),
                                  smem_desc(rstage + Cfg::kBOff + b * Cfg::kRecBytes + h * 3072,
                                            128, 256, 0),
                                  static_cast<uint32_t>(h));
                if (!DUAL)
                    umma_commit(bar_empty + 8 * s);      // ring stage free once the MMAs read it
                if (PAIR && a == 1)
                    umma_commit(bar_empty + 8 * sr);     // and the pair's records
                umma_commit(bar_acc_full + 8 * a);       // accumulators ready
            }
            __syncwarp();
        }
        // Wait (bounded) for this warp's last MMAs before TMEM is released.
        if (it >= 2)
            (void)mbar_wait(bar_acc_full + 8 * a, static_cast<uint32_t>(((it - 2) >> 1) & 1), lim);
    } else {
        // ---------------- epilogue ----------------
        const int e = warp - kFirstEpiWarp;
        const int grp = e >> 3;               // takes tiles (and buffers) with it % 2 == grp
        const int b = (e >> 2) & 1;           // block of the tile
        const int qtr = warp & 3;             // TMEM lane quarter this warp may access
        const int r = qtr * 32 + lane;        // row within the tile
        const int pair = grp * 4 + (e & 3);   // the quarter's two warps (b = 0, 1)
        int slot = 0;                         // staging buffer of this tile, mod 3
        // DUAL: one warp of the group stores the tile's side output and
        // releases the tile's ring stage as soon as that store has read it
        // (measured on GB300: deferring the release by a tile, to overlap
        // the wait, costs more in ring depth than the wait itself)
        const bool at_leader = DUAL && (e & 7) == 4 && lane == 0;
        int it = grp;
        bool ok = true;
        auto tw = walker(grp);
        // K2: the group also builds the operand records of its tiles in their
        // ring stages.  A tile's stage is free for its records once the MMAs
        // of the tile STAGES positions earlier -- the group's own tile three
        // steps back -- have completed, which the group sees when it reads
        // that tile's accumulators; so, after finishing tile it, the group
        // builds tile it + STAGES into the same stage (the first STAGES / 2
        // of its tiles before the loop).  Warp (e & 7) writes block
        // (e & 7) >> 2, rows 8 ((e & 7) & 3) .. + 7, lane = output channel.
        // Each warp then arrives on the stage's full barrier (which counts
        // the producer and these 8 warps) -- unless one of its own waits ran
        // out (the stage might then still be read), in which case the phase
        // never completes and the tile's MMAs time out in turn.
        // PAIR: the records of pair P are built once, by group P % 2, into
        // stage 2 P % STAGES, which is free once both tiles of pair P - 3
        // (the pair STAGES / 2 earlier in the same stage) have been read by
        // their MMAs: the group waits on the stage's empty barrier, which
        // counts the two MMA warps' commits.  So each group builds after every
        // other tile, half the work of the unpaired walk.
        TileWalk bwk(static_cast<int>(blockIdx.x), static_cast<int>(PAIR ? gridDim.x : 2 * gridDim.x),
                     static_cast<int>(p.ncol_tiles));   // the next tile (PAIR: pair) whose records to build
        if constexpr (!PAIR) bwk = TileWalk(static_cast<int>(blockIdx.x + grp * gridDim.x),
                                            static_cast<int>(2 * gridDim.x), static_cast<int>(p.ncol_tiles));
        const int bb = (e & 7) >> 2, bg = (e & 7) & 3;
        auto build = [&](int ct, int s, bool can) {
            const int64_t j = 2 * static_cast<int64_t>(ct) + bb;
            if (can && j < p.nb)
                build_record_rows(base + s * Cfg::kStageBytes + Cfg::kBOff + bb * Cfg::kRecBytes,
                                  p.factors + (p.shared_params ? 0 : j * 20), lane, bg);
            fence_proxy_async_smem();
            __syncwarp();
            if (can && lane == 0) mbar_arrive(bar_full + 8 * s);
        };
        // bwk's next position is the one this group builds (unpaired), or
        // the pair to build after this iteration, if the group's (PAIR)
        auto bwk_valid = [&]() {
            if constexpr (PAIR) return bwk.rt < nrp;
            else return bwk.rt < p.nrow_tiles;
        };
        if (K2 && !PAIR) {
            for (int k = 0; k < STAGES / 2 && bwk_valid(); ++k, bwk.next())
                build(bwk.ct, grp + 2 * k, true);
        }
        if (PAIR) {
            for (int P = 0; P < STAGES / 2 && bwk_valid(); ++P, bwk.next())
                if (P % 2 == grp) build(bwk.ct, (2 * P) % STAGES, true);
        }

        for (; valid(tw); tw.next(), it += 2) {
            const int a = grp;
            const int rt = tw.rt, ct = tw.ct;
            // PAIR: this iteration is pair Q = it / 2; after it the group
            // builds pair Q + 3 if that pair is its own
            const bool builds = K2 && bwk_valid() && (!PAIR || ((it / 2 + STAGES / 2) % 2) == grp);
            if (builds && lane < 2) {
                // this iteration's record build reads 80 bytes of factors:
                // fetch them into L1 now, under the tile's epilogue
                const int64_t j = 2 * static_cast<int64_t>(bwk.ct) + bb;
                if (j < p.nb) {
                    const char *f = reinterpret_cast<const char *>(
                        p.factors + (p.shared_params ? 0 : j * 20));
                    asm volatile("prefetch.global.L1 [%0];" ::"l"(f + 79 * lane));
                }
            }
            const int j = ct * 2 + b;
            const int row = rt * kBR + r;
            const uint32_t stg = base + Cfg::kStgOff + (pair * Cfg::kStgBufs + slot) * Cfg::kStgBytes;
            const uint32_t sfstg = base + Cfg::kSfStgOff + (pair * Cfg::kStgBufs + slot) * 32;
            uint32_t sbyte = 0;       // this row's scale byte for block j (0: padding block)
            bool swrite = false;
            if (ok) ok = __all_sync(0xffffffffu,
                                    mbar_wait(bar_acc_full + 8 * a, static_cast<uint32_t>((it >> 1) & 1), lim));
            uint4 codes = make_uint4(0u, 0u, 0u, 0u);
            uint4 at_w[4];            // DUAL: the row's 32 bf16 of y (bf16 NaN if not computed)
            if (DUAL) {
#pragma unroll
                for (int k = 0; k < 4; ++k) at_w[k] = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
            }
            if (ok) {
                tc_fence_after();
                float2 Y[16];
                if (j < p.nb) {
                    // columns: term hi, mid, lo (32 outputs each); y = (hi + mid) + lo
                    const uint32_t tb = tmem_base + (static_cast<uint32_t>(qtr * 32) << 16) +
                                        a * kAccCols + b * kBlockCols;
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tb, r0);
                    tmem_ld32(tb + 32, r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        Y[t] = __fadd2_rn(
                            make_float2(__uint_as_float(r0[2 * t]), __uint_as_float(r0[2 * t + 1])),
                            make_float2(__uint_as_float(r1[2 * t]), __uint_as_float(r1[2 * t + 1])));
                    tmem_ld32(tb + 64, r0);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(bar_acc_empty + 8 * a);
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        Y[t] = __fadd2_rn(Y[t], make_float2(__uint_as_float(r0[2 * t]),
                                                            __uint_as_float(r0[2 * t + 1])));
                    if (DEBUG && row < p.m) {
                        float *yd = p.y_debug + static_cast<int64_t>(row) * p.d + j * 32;
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            stg_f4(yd + 4 * k, make_float4(Y[2 * k].x, Y[2 * k].y, Y[2 * k + 1].x,
                                                           Y[2 * k + 1].y));
                    }
                    if (DUAL) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint32_t w[4];
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const __nv_bfloat162 h = __floats2bfloat162_rn(Y[4 * k + t].x, Y[4 * k + t].y);
                                w[t] = *reinterpret_cast<const uint32_t *>(&h);
                            }
                            at_w[k] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                    codes = quantize_block(Y, sbyte);
                    swrite = true;
                } else {
                    tc_fence_before();
                    mbar_arrive(bar_acc_empty + 8 * a);
                    swrite = p.sf_layout != KQ_SF_ROWMAJOR;
                }
            } else if (j < p.nb && row < p.m_rows) {
                sbyte = 0xFFu;        // E8M0 NaN: this block was not computed
                swrite = true;
            }
            // Scales.  Row-major: one byte per thread.  Tiled: blocks 2 ct and
            // 2 ct + 1 of a row are adjacent bytes, so the b = 1 warp hands its
            // byte to the b = 0 warp (through shared memory, across the pair
            // barrier below) and that warp writes both as one 16-bit store.
            const bool tiled = p.sf_layout != KQ_SF_ROWMAJOR;
            if (!tiled) {
                if (swrite) store_scale_u(p, row, j, sbyte);
            } else if (b == 1) {
                asm volatile("st.shared.u8 [%0], %1;" ::"r"(sfstg + lane), "r"(sbyte) : "memory");
            }
            // Codes -> the pair's staging buffer (32-byte rows, the 32-byte
            // swizzle of the tensor map: 16-byte chunk b ^ bit 2 of the row)
            // -> one TMA store of 32 rows x 32 bytes by the b = 0 warp.  Three
            // buffers rotate: the store that last read this one was committed
            // three tiles ago, and the b = 0 warp waited for it to finish
            // reading (below) before the pair barrier of the previous tile.
            sts128(stg + lane * 32 + ((b ^ ((lane >> 2) & 1)) << 4), codes);
            if (DUAL) {
                // side output over the tile's activations in its ring stage:
                // row r, 16-byte chunk 4 b + k at position (4 b + k) ^ (r % 8)
                // (the 128B swizzle of the activation tensor map)
                const uint32_t arow = base + static_cast<uint32_t>(it % STAGES) * Cfg::kStageBytes +
                                      static_cast<uint32_t>(r) * 128;
#pragma unroll
                for (int k = 0; k < 4; ++k) sts128(arow + (((4 * b + k) ^ (r & 7)) << 4), at_w[k]);
            }
            fence_proxy_async_smem();
            named_barrier(1 + pair, 64);
            if (tiled && b == 0 && (!PAIR || row < p.m_rows)) {     // PAIR: rows past the last tile
                uint32_t partner;
                asm volatile("ld.shared.u8 %0, [%1];" : "=r"(partner) : "r"(sfstg + lane) : "memory");
                *reinterpret_cast<uint16_t *>(p.sf + sf_blocked_offset(row, ct * 2, p.ncb)) =
                    static_cast<uint16_t>(sbyte | (partner << 8));
            }
            if (b == 0 && lane == 0) {
                if (ct * 2 < p.nb)      // padding tiles of the scale layout have no codes
                    tma_store_2d(&tmQ, ct * 32, rt * kBR + qtr * 32, stg);
                bulk_commit_group();
                bulk_wait_group_read<1>();
            }
            if (DUAL) {
                named_barrier(9 + grp, kEpiThreads / 2);   // the whole tile is in the stage
                if (at_leader) {
                    const int s = it % STAGES;
                    if (ct * 2 < p.nb)
                        tma_store_2d(&tmAT, ct * 64, rt * kBR,
                                     base + static_cast<uint32_t>(s) * Cfg::kStageBytes);
                    bulk_commit_group();
                    bulk_wait_group_read<0>();
                    mbar_arrive(bar_empty + 8 * s);
                }
            }
            slot = slot == Cfg::kStgBufs - 1 ? 0 : slot + 1;
            if (K2 && !PAIR && bwk_valid()) {
                build(bwk.ct, static_cast<int>(it % STAGES), ok);
                bwk.next();
            }
            if (PAIR && bwk_valid()) {
                if (builds) {
                    // pair Q + 3 goes into pair Q's stage once both of pair
                    // Q's tiles have been read
                    const int64_t q0 = it - grp;                 // pair Q's first tile
                    const int s2 = static_cast<int>(q0 % STAGES);
                    const bool can = __all_sync(0xffffffffu,
                        ok && mbar_wait(bar_empty + 8 * s2, static_cast<uint32_t>((q0 / STAGES) & 1), lim));
                    build(bwk.ct, s2, can);
                }
                bwk.next();
            }
        }
        if (b == 0 && lane == 0) bulk_wait_group_all();
        if (at_leader) bulk_wait_group_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---- operand records (kq_expand_blocks, KQ_K_BF16X3) ------------------------------

// K'[r][c] = prod_{k=2..5} G_k[bit_{5-k}(r)][bit_{5-k}(c)] for r, c in
// 0..15 (eq. 12 without G1), in fp64.
__device__ __forceinline__ double kron_tail(const float *f, int r, int c)
{
    double x = 1.0;
#pragma unroll
    for (int k = 2; k <= 5; ++k) {
        const int bit = 5 - k;
        x *= static_cast<double>(f[(k - 1) * 4 + ((r >> bit) & 1) * 2 + ((c >> bit) & 1)]);
    }
    return x;
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
    // one thread per block j, K = 16 step h, output channel c and input
    // channel pair kp: the entries K_j[16 h + 2 kp][c] and K_j[16 h + 2 kp + 1][c]
    // in fp64, each split into its three bf16 terms in turn (term t = the
    // remainder after terms 0 .. t-1, rounded to nearest), one word per term
    const int64_t n = nb * 512;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t j = idx >> 9;
        const int w = static_cast<int>(idx & 511);
        const int h = w >> 8, c = (w >> 3) & 31, kp = w & 7;
        const int k0 = 2 * kp, r0 = 16 * h + k0;
        const float *f = factors + j * 20;
        uint8_t *rec = out + j * kUmmaRecordBytes;
        // K_j[r][c] = G1[bit4(r)][bit4(c)] * K'_j[r % 16][c % 16]
        const double g0 = static_cast<double>(f[((r0 >> 4) & 1) * 2 + ((c >> 4) & 1)]);
        double x0 = g0 * kron_tail(f, r0 & 15, c & 15);
        double x1 = g0 * kron_tail(f, (r0 + 1) & 15, c & 15);
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            const __nv_bfloat16 v0 = __double2bfloat16(x0), v1 = __double2bfloat16(x1);
            x0 -= static_cast<double>(__bfloat162float(v0));
            x1 -= static_cast<double>(__bfloat162float(v1));
            const int nn = 32 * t + c;
            const int off = h * 3072 + (nn >> 3) * 256 + (k0 >> 3) * 128 + (nn & 7) * 16 + (k0 & 7) * 2;
            *reinterpret_cast<uint32_t *>(rec + off) =
                static_cast<uint32_t>(__bfloat16_as_ushort(v0)) |
                (static_cast<uint32_t>(__bfloat16_as_ushort(v1)) << 16);
        }
    }
}

struct USlot {
    std::once_flag once[64];
    int occupancy[64] = {};
    cudaError_t err[64] = {};
};

template <int STAGES, bool DEBUG, bool DUAL, bool K2, bool PAIR = false>
kq_status launch_umma(const CUtensorMap &map, const CUtensorMap &mapq, const CUtensorMap &mapat,
                      QuantParams p, const uint8_t *records, int sm_count, cudaStream_t stream)
{
    using Cfg = UCfg<STAGES>;
    auto kern = quant_umma_kernel<STAGES, DEBUG, DUAL, K2, PAIR>;
    constexpr int threads = kThreadsU;
    static USlot slot;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KQ_ERR_CUDA;
    std::call_once(slot.once[dev], [&] {
        slot.err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg::kSmemBytes);
        if (slot.err[dev] == cudaSuccess)
            slot.err[dev] = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &slot.occupancy[dev], kern, threads, Cfg::kSmemBytes);
    });
    if (slot.err[dev] != cudaSuccess || slot.occupancy[dev] < 1) return KQ_ERR_CUDA;
    // tiles of 64 channels (one TMA box); the tiled scale layout also needs
    // its padding block-columns (up to a multiple of 4) visited and zeroed
    p.ncol_tiles = p.sf_layout == KQ_SF_ROWMAJOR ? (p.nb + 1) / 2 : 2 * p.ncb;
    p.nrow_tiles = (p.m_rows + kBR - 1) / kBR;
    p.ntiles = p.nrow_tiles * p.ncol_tiles;
    if (p.ntiles == 0) return KQ_OK;
    // one CTA per SM: each holds 256 of the SM's 512 TMEM columns
    const int grid = static_cast<int>(std::min<int64_t>(p.ntiles, sm_count));
    if (!tiles_fit_int32(p, grid)) return KQ_ERR_SHAPE;
    return launch_pdl(kern, grid, threads, Cfg::kSmemBytes, stream, map, mapq, mapat, p,
                      records);
}

}  // namespace

kq_status launch_umma_records(const float *factors, int64_t nb, void *out, cudaStream_t stream)
{
    const int64_t work = nb * 512;
    umma_records_kernel<<<static_cast<int>(std::min<int64_t>((work + 255) / 256, 4096)), 256, 0,
                          stream>>>(factors, nb, static_cast<uint8_t *>(out));
    return check_launch();
}

kq_status launch_quant_umma(const uint16_t *A, int64_t lda, const void *K_expanded,
                            const QuantParams &p, uint16_t *at, int64_t ldat, cudaStream_t stream)
{
    DeviceInfo info;
    kq_status st = device_info(info);
    if (st != KQ_OK) return st;
    CUtensorMap map, mapq;
    st = make_tensor_map_2d_bf16(&map, A, p.m, p.d, lda, 64, kBR);
    if (st != KQ_OK) return st;
    st = make_tensor_map_2d_u8(&mapq, p.q, p.m, p.d / 2, p.ldq, 32, 32,
                               CU_TENSOR_MAP_SWIZZLE_32B);
    if (st != KQ_OK) return st;
    const uint8_t *rec = static_cast<const uint8_t *>(K_expanded);
    const int sms = info.sm_count;
    if (K_expanded == nullptr) {
        // K2: no records in memory, the kernel builds them from p.factors.
        // With at least four tiles per CTA the tiles go by pairs of one
        // column, which share their records (half the building); below
        // that, pairs would leave SMs idle.
        if (at != nullptr || p.factors == nullptr) return KQ_ERR_NULL;
        const int64_t ncol = p.sf_layout == KQ_SF_ROWMAJOR ? (p.nb + 1) / 2 : 2 * p.ncb;
        const int64_t ntiles = (p.m_rows + kBR - 1) / kBR * ncol;
        if (ntiles >= 4 * static_cast<int64_t>(sms)) {
            if (p.y_debug != nullptr)
                return launch_umma<6, true, false, true, true>(map, mapq, map, p, nullptr, sms, stream);
            return launch_umma<6, false, false, true, true>(map, mapq, map, p, nullptr, sms, stream);
        }
        if (p.y_debug != nullptr)
            return launch_umma<6, true, false, true>(map, mapq, map, p, nullptr, sms, stream);
        return launch_umma<6, false, false, true>(map, mapq, map, p, nullptr, sms, stream);
    }
    if (at == nullptr) {
        if (p.y_debug != nullptr)
            return launch_umma<6, true, false, false>(map, mapq, map, p, rec, sms, stream);
        return launch_umma<6, false, false, false>(map, mapq, map, p, rec, sms, stream);
    }
    CUtensorMap mapat;
    st = make_tensor_map_2d_bf16(&mapat, at, p.m, p.d, ldat, 64, kBR);
    if (st != KQ_OK) return st;
    if (p.y_debug != nullptr)
        return launch_umma<6, true, true, false>(map, mapq, mapat, p, rec, sms, stream);
    return launch_umma<6, false, true, false>(map, mapq, mapat, p, rec, sms, stream);
}

}  // namespace kq
