// Device-side building blocks of the KroQuant MXFP4 quantizer (sm_103a).
//
// Hand-written PTX for the Blackwell data path: mbarrier pipeline waits with
// a time limit, 2-D TMA tile loads (cp.async.bulk.tensor), the fp32 -> E2M1
// conversion (cvt.rn.satfinite.e2m1x2.f32) and packed fp32x2 arithmetic.
//
// MXFP4 rule ("KroQuant: Kronecker-Structured Block Transforms for Efficient
// Post-Training Quantization of Diffusion Transformers", Sec. 3.1 and 4.1,
// OCP MX v1.0): per 32-element block, e = floor(log2 amax) - 2 clamped to
// [-127, 127], scale byte e + 127, codes = E2M1(y / 2^e) with round to
// nearest even and saturation.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

namespace kq {

// A wait that has not completed after this many nanoseconds gives up.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Release arrive: this thread's earlier shared-memory reads of the guarded
// buffer happen before the arrival is observed.
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that may suspend the thread (up to the hint, in ns) until the
// phase completes, so that waiting threads do not keep polling the barrier.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(100000u)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if
// it has not completed within limit_ns nanoseconds.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ---- TMA ----------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of the box at element coordinates (x, y) into shared memory,
// completing `bytes` of transaction count on the barrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t x,
                                            int32_t y, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16),
// completing its bytes on the barrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// 2-D tiled store of a shared-memory box to global memory at element
// coordinates (x, y); out-of-range parts of the box are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int32_t x, int32_t y,
                                             uint32_t src)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_group_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tensor cores).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Barrier over `count` threads (whole warps) with id `id` (1..15).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// L2 policy for data read exactly once (the activations): evict first.
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- loads / stores -------------------------------------------------------------

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr)
{
    const uint4 v = lds128(addr);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                       __uint_as_float(v.w));
}

// Entry [r][c] of a 2x2 factor held as (g00, g01, g10, g11).
__device__ __forceinline__ float sel2x2(float4 g, int r, int c)
{
    return r ? (c ? g.w : g.z) : (c ? g.y : g.x);
}

__device__ __forceinline__ float4 ldg_nc_f4(const float *p)
{
    float4 v;
    asm("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p));
    return v;
}

// Streaming 16-byte store (written once, not re-read by this kernel).
__device__ __forceinline__ void stg128_cs(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void stg_f4(float *p, float4 v)
{
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

// ---- bf16 -> fp32 -------------------------------------------------------------------

// A 32-bit word holds two bf16 values, element 2t in the low half.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The same for two fp16 values (exact: every fp16 is an fp32).
__device__ __forceinline__ float f16_lo(uint32_t w)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// ---- MXFP4 epilogue -----------------------------------------------------------------

// E8M0 byte of a block from its amax (>= 0, finite): with E the biased fp32
// exponent field, floor(log2 amax) = E - 127 for normal amax, so
// e + 127 = E - 2; zero, subnormal and E <= 2 amax all clamp to byte 0
// (e = -127).  The largest finite amax gives 252 (e = 125).
__device__ __forceinline__ uint32_t e8m0_byte(float amax)
{
    const int E = static_cast<int>(__float_as_uint(amax) >> 23);
    return static_cast<uint32_t>(max(E - 2, 0));
}

// 2^-e as fp32 for scale byte b (e = b - 127): exponent field 254 - b, which
// stays in [2, 254] for b in [0, 252], so the multiply y * 2^-e is exact.
__device__ __forceinline__ float inv_scale(uint32_t byte)
{
    return __uint_as_float((254u - byte) << 23);
}

// Programmatic dependent launch: returns once the grids this one depends on
// have completed and their memory is visible (at once when there are none).
// The persistent quantizers are launched with programmatic stream
// serialization and call this after their shared-memory / TMEM setup and
// before their first global-memory access, so the launch of a quantizer
// overlaps the end of the previous kernel while every read of A and write of
// q / sf stays ordered after it.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the grids that depend on this one be scheduled once every CTA has
// called it (or exited); their grid_dependency_wait still waits for this
// grid to complete.  Measured on GB300: called from the start of a 27 us
// quantizer it slowed it by 1.2 us; the tcgen05 quantizer calls it when its
// producer has issued its last tile.
__device__ __forceinline__ void grid_dependents_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// max(a, b, c) in one instruction (3-input max.f32; a NaN input is ignored
// like fmaxf does).
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Eight fp32 values -> eight E2M1 codes packed in a word, value 0 in bits 0-3.
// cvt.rn.satfinite.e2m1x2.f32 d, a, b puts a in the high nibble of d and b in
// the low nibble.
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                           float v5, float v6, float v7)
{
    uint32_t out;
    asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n\t"
        "mov.b32 %0, {c0, c1, c2, c3};\n\t}"
        : "=r"(out)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
    return out;
}

// Quantizes one 32-element block held as 16 float2 (y[2t], y[2t+1]).
// Returns the packed codes (16 bytes) and writes the scale byte.
__device__ __forceinline__ uint4 quantize_block(const float2 (&Y)[16], uint32_t &byte_out)
{
    // four independent chains of 3-input maxima over |y|
    float m[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float2 p0 = Y[4 * c], p1 = Y[4 * c + 1], p2 = Y[4 * c + 2], p3 = Y[4 * c + 3];
        float t = fmax3(fabsf(p0.x), fabsf(p0.y), fabsf(p1.x));
        t = fmax3(t, fabsf(p1.y), fabsf(p2.x));
        t = fmax3(t, fabsf(p2.y), fabsf(p3.x));
        m[c] = fmaxf(t, fabsf(p3.y));
    }
    const float amax = fmax3(fmaxf(m[0], m[1]), m[2], m[3]);
    const uint32_t byte = e8m0_byte(amax);
    const float s = inv_scale(byte);
    const float2 s2 = make_float2(s, s);
    // scale and encode eight values at a time (keeps few values live)
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 v0 = __fmul2_rn(Y[4 * k], s2), v1 = __fmul2_rn(Y[4 * k + 1], s2);
        const float2 v2 = __fmul2_rn(Y[4 * k + 2], s2), v3 = __fmul2_rn(Y[4 * k + 3], s2);
        w[k] = e2m1x8(v0.x, v0.y, v1.x, v1.y, v2.x, v2.y, v3.x, v3.y);
    }
    byte_out = byte;
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Row-major walk over (row tile, column tile) pairs: first, first + step,
// first + 2 step, ... with tile = rt * ncol + ct, in 32-bit arithmetic (the
// launchers check that tile counts fit, see tiles_fit_int32) and without any
// division in the loop.  The walk ends when rt reaches the number of row tiles.
struct TileWalk {
    int rt, ct;
    int ncol, step_rt, step_ct;
    __device__ __forceinline__ TileWalk(int first, int step, int ncol_)
        : rt(first / ncol_), ct(first % ncol_), ncol(ncol_), step_rt(step / ncol_),
          step_ct(step % ncol_)
    {
    }
    __device__ __forceinline__ void next()
    {
        ct += step_ct;
        rt += step_rt;
        if (ct >= ncol) {
            ct -= ncol;
            ++rt;
        }
    }
};

// Byte position of a scale in the 128x4 tiled layout of block-scaled MMA.
__device__ __forceinline__ int64_t sf_blocked_offset(int64_t row, int64_t kb, int64_t ncb)
{
    const int64_t tile = (row >> 7) * ncb + (kb >> 2);
    return tile * 512 + (row & 31) * 16 + ((row & 127) >> 5) * 4 + (kb & 3);
}

}  // namespace kq
