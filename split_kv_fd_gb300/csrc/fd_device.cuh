// fd_device.cuh -- device-side building blocks for the split-KV decode
// kernels: shared-memory mbarriers, 1-D bulk (TMA) global->shared copies,
// bounded waits, and 16-byte element vectors widened to float32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include <type_traits>

namespace fd {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Upper bound on any single wait for one of a kernel's own bulk copies.  A
// 8 KB copy lands in microseconds; the bound only exists so that a kernel
// can never spin forever.  After it expires the kernel records the event in
// the device status word and stops waiting.
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;   // 1 s
constexpr unsigned WAIT_LIMIT_POLLS = 1u << 30;

// Status word bits.
constexpr unsigned STATUS_TIMEOUT = 1u;
constexpr unsigned STATUS_BAD_PAGE = 2u;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One plain arrival.
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One arrival that also announces `bytes` of incoming transaction data.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for phase `parity` of barrier `bar` by one thread on its own
// (no warp vote: for a lane that runs a role by itself while its warp's
// other lanes wait elsewhere).
__device__ __forceinline__ bool mbar_wait_bounded_thread(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    for (unsigned i = 0; i < WAIT_LIMIT_POLLS; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 63u) == 63u && global_ns() - t0 > WAIT_LIMIT_NS)
            break;
    }
    return false;
}

// Bounded wait for phase `parity` of barrier `bar`.  Every lane polls; the
// result is made warp-uniform (all lanes must have seen completion).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
        unsigned long long t0 = global_ns();
        for (unsigned i = 0; i < WAIT_LIMIT_POLLS; ++i) {
            if (mbar_try_wait(bar, parity)) {
                ok = true;
                break;
            }
            if ((i & 63u) == 63u && global_ns() - t0 > WAIT_LIMIT_NS)
                break;
        }
    }
    return __all_sync(FULL_MASK, ok);
}

// One try at phase `parity` of barrier `bar` that may suspend the thread in
// hardware for up to `hint_ns`; it resumes as soon as the phase completes.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// Bounded wait for a phase that may take long (a whole segment of
// streaming), for a warp that must not slow the warps doing the work: each
// try suspends the warp in hardware for up to `hint_ns` and resumes it as
// soon as the phase completes.
__device__ __forceinline__ bool mbar_wait_bounded_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    const unsigned long long t0 = global_ns();
    bool ok = false;
    for (unsigned i = 0; i < WAIT_LIMIT_POLLS; ++i) {
        if (mbar_try_wait_hint(bar, parity, hint_ns)) {
            ok = true;
            break;
        }
        if (global_ns() - t0 > WAIT_LIMIT_NS)
            break;
    }
    return __all_sync(FULL_MASK, ok);
}

// The same for one thread on its own (no warp vote).
__device__ __forceinline__ bool mbar_wait_bounded_sleep_thread(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    if (mbar_try_wait_hint(bar, parity, hint_ns))
        return true;
    const unsigned long long t0 = global_ns();
    for (unsigned i = 0; i < WAIT_LIMIT_POLLS; ++i) {
        if (mbar_try_wait_hint(bar, parity, hint_ns))
            return true;
        if (global_ns() - t0 > WAIT_LIMIT_NS)
            break;
    }
    return false;
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Same, with an L2 eviction-priority policy (streamed data is read once).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero):
// ex2(-inf) = +0.
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two float32 lanes of a 64-bit register pair, and the packed FMA on them
// (PTX fma.rn.f32x2: two independent round-to-nearest fp32 FMAs).
__device__ __forceinline__ uint64_t pack2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t r, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}

__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// ---------------------------------------------------------------------------
// Tensor-map (tiled) TMA and warp-level tensor-core helpers.
// ---------------------------------------------------------------------------

// 3-D tiled copy global -> shared through a tensor map, completion on `bar`.
// The innermost coordinate (x) times the element size must be a multiple of
// 16 bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int x, int y, int z,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// 4-D tiled copy global -> shared through a tensor map, completion on `bar`
// (the same rule for x).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, int x, int y, int z, int w,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

// Barrier `id` (1..15) over `count` threads (whole warps) of the block.
__device__ __forceinline__ void named_bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Hint: start fetching the global-memory line holding `ptr` into L1.
__device__ __forceinline__ void prefetch_l1(const void *ptr)
{
    asm volatile("prefetch.global.L1 [%0];" ::"l"(__cvta_generic_to_global(ptr)));
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Four 8x8 b16 matrices from shared memory (lane l gives the address of row
// l % 8 of matrix l / 8), plain or transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// The transpose of an 8x8 matrix of 16-bit elements held as an mma
// fragment (lane t holds row t/4, columns 2(t%4) and 2(t%4)+1): afterwards
// lane t holds row t/4, columns 2(t%4), 2(t%4)+1 of the transpose.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x)
{
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D = A(16x16) * B(16x8) + D, fp32 accumulate; A, B both bf16 or both f16.
// (not volatile: a pure function of registers, free to be scheduled)
template <typename T> struct Mma;
template <> struct Mma<__nv_bfloat16> {
    __device__ __forceinline__ static void run(float *d, const uint32_t *a, uint32_t b0, uint32_t b1)
    {
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // two floats -> one packed register (lower half = x), round-to-nearest-even
    __device__ __forceinline__ static uint32_t pack(float x, float y)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
        uint32_t r;
        memcpy(&r, &h, 4);
        return r;
    }
    __device__ __forceinline__ static float2 unpack(uint32_t r)
    {
        __nv_bfloat162 h;
        memcpy(&h, &r, 4);
        return __bfloat1622float2(h);
    }
};
template <> struct Mma<__half> {
    __device__ __forceinline__ static void run(float *d, const uint32_t *a, uint32_t b0, uint32_t b1)
    {
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float x, float y)
    {
        __half2 h = __floats2half2_rn(x, y);
        uint32_t r;
        memcpy(&r, &h, 4);
        return r;
    }
    __device__ __forceinline__ static float2 unpack(uint32_t r)
    {
        __half2 h;
        memcpy(&h, &r, 4);
        return __half22float2(h);
    }
};

// ---------------------------------------------------------------------------
// 16-byte vectors of the storage type, widened to float32.
// ---------------------------------------------------------------------------
template <typename T> struct Elem;

template <> struct Elem<float> {
    static constexpr int VEC = 4;
    __device__ __forceinline__ static void widen(const uint4 &u, float *f)
    {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
};

template <> struct Elem<__nv_bfloat16> {
    static constexpr int VEC = 8;
    // bf16 is the upper half of a binary32: widening is a shift / mask.
    __device__ __forceinline__ static void widen(const uint4 &u, float *f)
    {
        f[0] = __uint_as_float(u.x << 16);
        f[1] = __uint_as_float(u.x & 0xffff0000u);
        f[2] = __uint_as_float(u.y << 16);
        f[3] = __uint_as_float(u.y & 0xffff0000u);
        f[4] = __uint_as_float(u.z << 16);
        f[5] = __uint_as_float(u.z & 0xffff0000u);
        f[6] = __uint_as_float(u.w << 16);
        f[7] = __uint_as_float(u.w & 0xffff0000u);
    }
};

template <> struct Elem<__half> {
    static constexpr int VEC = 8;
    __device__ __forceinline__ static void widen(const uint4 &u, float *f)
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h;
            memcpy(&h, &w[i], 4);
            float2 p = __half22float2(h);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
};

// OCP E4M3 bytes: each pair converts exactly to f16x2 (cvt.rn.f16x2.e4m3x2,
// lower byte to the lower half), then to float32.
template <> struct Elem<__nv_fp8_e4m3> {
    static constexpr int VEC = 16;
    __device__ __forceinline__ static void widen(const uint4 &u, float *f)
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t h01, h23;
            asm("{\n\t.reg .b16 lo, hi;\n\t"
                "mov.b32 {lo, hi}, %2;\n\t"
                "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
                "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
                : "=r"(h01), "=r"(h23)
                : "r"(w[i]));
            __half2 a, b;
            memcpy(&a, &h01, 4);
            memcpy(&b, &h23, 4);
            const float2 fa = __half22float2(a), fb = __half22float2(b);
            f[4 * i] = fa.x;
            f[4 * i + 1] = fa.y;
            f[4 * i + 2] = fb.x;
            f[4 * i + 3] = fb.y;
        }
    }
};

// VEC elements of q starting at element `off`, widened to float32; q is
// float32 (q_dtype 0), float16 (1) or bfloat16 (2) and 16-byte aligned.
template <int VEC>
__device__ __forceinline__ void load_q(const void *q, int q_dtype, long long off, float *qf)
{
    if (q_dtype == 0) {
        const float4 *p4 = reinterpret_cast<const float4 *>(static_cast<const float *>(q) + off);
#pragma unroll
        for (int i = 0; i < VEC / 4; ++i) {
            const float4 x = __ldg(p4 + i);
            qf[4 * i] = x.x;
            qf[4 * i + 1] = x.y;
            qf[4 * i + 2] = x.z;
            qf[4 * i + 3] = x.w;
        }
    } else if (VEC % 8 == 0) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(q) + off);
#pragma unroll
        for (int i = 0; i < VEC / 8; ++i) {
            const uint4 u = __ldg(p + i);
            if (q_dtype == 1)
                Elem<__half>::widen(u, qf + 8 * i);
            else
                Elem<__nv_bfloat16>::widen(u, qf + 8 * i);
        }
    } else {
        const uint16_t *p = static_cast<const uint16_t *>(q) + off;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const uint16_t h = __ldg(p + i);
            qf[i] = q_dtype == 1 ? __half2float(__ushort_as_half(h))
                                 : __uint_as_float(((uint32_t)h) << 16);
        }
    }
}

// Store one float as the requested output dtype (round-to-nearest-even).
__device__ __forceinline__ void store_out(void *out, long long idx, int out_dtype, float x)
{
    if (out_dtype == 0)
        static_cast<float *>(out)[idx] = x;
    else if (out_dtype == 1)
        static_cast<__half *>(out)[idx] = __float2half_rn(x);
    else
        static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(x);
}

}  // namespace fd
