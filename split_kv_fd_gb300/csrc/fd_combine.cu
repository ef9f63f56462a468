// fd_combine.cu -- stage 2 of FlashDecoding as its own launch: merge the P
// partials of every (b, h) into out and lse.
//
//   m/l/o form ("FlashDecoding 数学推导", §2.4.2, §2.5 stage 2):
//     m_g = max_p m_p,  w_p = exp(m_p - m_g) l_p,  l_g = sum_p w_p,
//     out = sum_p w_p o_p / l_g,  lse = m_g + ln l_g.
//   LSE form ("FlashDecoding 数学推导：传统 m/l/o 方法与 LSE 方法", §2.3.4):
//     S_g = S_max + ln sum_p exp(S_p - S_max),  out = sum_p exp(S_p - S_g) o_p.
// Empty splits (l_p == 0, S_p == -inf) get weight 0 explicitly.
//
// One CTA per (b, h): the P weights are computed once into shared memory by
// the whole block, then each thread forms one output element; the partial
// rows are read coalesced along d.  The work is tiny next to stage 1 (P*(d+3)
// floats per (b, h) against 2*len*d K/V elements).
#include "fd_device.cuh"
#include "fd_internal.h"

namespace fd {

constexpr int COMBINE_THREADS = 128;

__device__ __forceinline__ float block_reduce(float x, bool is_max, float *scratch)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float y = __shfl_xor_sync(FULL_MASK, x, o);
        x = is_max ? fmaxf(x, y) : x + y;
    }
    __syncthreads();  // scratch may still be read by a previous reduction
    if (lane == 0)
        scratch[w] = x;
    __syncthreads();
    float r = scratch[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i)
        r = is_max ? fmaxf(r, scratch[i]) : r + scratch[i];
    return r;
}

template <bool LSE> __global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(const CombineParams p)
{
    extern __shared__ float wgt[];  // [P]
    __shared__ float scratch[32];
    const long long row = blockIdx.x;
    const int P = p.P, d = p.d;
    const float *key = LSE ? p.lse_part + row * P : p.m_part + row * P;
    const float *lp = LSE ? nullptr : p.l_part + row * P;

    float mx = -INFINITY;
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const bool empty = LSE ? (key[i] == -INFINITY) : !(lp[i] > 0.f);
        if (!empty)
            mx = fmaxf(mx, key[i]);
    }
    const float M = block_reduce(mx, true, scratch);

    float sum = 0.f;
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
        float e = 0.f;
        if (LSE) {
            if (key[i] != -INFINITY)
                e = expf(key[i] - M);
        } else if (lp[i] > 0.f) {
            e = expf(key[i] - M) * lp[i];
        }
        wgt[i] = e;
        sum += e;
    }
    const float L = block_reduce(sum, false, scratch);
    const bool nonempty = L > 0.f;
    const float lse_g = nonempty ? M + logf(L) : -INFINITY;

    // Both forms finish as out = sum_p e_p o_p / sum_p e_p.  For the LSE form
    // this is the page's exp(S_p - S_g) = exp(S_p - S_max) / sum evaluated
    // without first rounding S_g = S_max + ln(sum) to float32.
    __syncthreads();

    const float *o = p.o_part + row * P * d;
    for (int t = threadIdx.x; t < d; t += blockDim.x) {
        float acc = 0.f;
#pragma unroll 8
        for (int i = 0; i < P; ++i)
            acc = fmaf(wgt[i], o[(long long)i * d + t], acc);
        store_out(p.out, row * d + t, p.out_dtype, nonempty ? acc / L : 0.f);
    }
    if (threadIdx.x == 0 && p.lse)
        p.lse[row] = lse_g;
}

// (o_a, S_a) (+) (o_b, S_b) per row: the merge operator of "FlashDecoding
// 数学推导：传统 m/l/o 方法与 LSE 方法" §2.3.5, evaluated in the safe form of
// §3.2.1 stage 2: S = S_max + log1p(exp(S_min - S_max)),
// o = o_a exp(S_a - S) + o_b exp(S_b - S).  An empty side (S = -inf) leaves
// the other unchanged; two empty sides give (0, -inf).  One warp per row:
// every lane reads the row's S_a, S_b before lane 0 writes S, so the outputs
// may alias either input.
__global__ void merge_lse_kernel(const float4 *oa, const float *sa, const float4 *ob,
                                 const float *sb, int rows, int d4, float4 *out, float *sout)
{
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long r = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
         r += warps) {
        const float s1 = sa[r], s2 = sb[r];
        float w1, w2, S;
        if (s1 == -INFINITY && s2 == -INFINITY) {
            w1 = w2 = 0.f;
            S = -INFINITY;
        } else if (s2 == -INFINITY) {
            w1 = 1.f, w2 = 0.f, S = s1;
        } else if (s1 == -INFINITY) {
            w1 = 0.f, w2 = 1.f, S = s2;
        } else {
            const float smax = fmaxf(s1, s2), smin = fminf(s1, s2);
            S = smax + log1pf(expf(smin - smax));
            w1 = expf(s1 - S);
            w2 = expf(s2 - S);
        }
        for (int c = lane; c < d4; c += 32) {
            const long long i = r * d4 + c;
            const float4 a = oa[i], b = ob[i];
            out[i] = make_float4(a.x * w1 + b.x * w2, a.y * w1 + b.y * w2, a.z * w1 + b.z * w2,
                                 a.w * w1 + b.w * w2);
        }
        __syncwarp();
        if (lane == 0)
            sout[r] = S;
    }
}

cudaError_t launch_merge_lse(const float *oa, const float *sa, const float *ob, const float *sb,
                             int rows, int d, float *out, float *sout, cudaStream_t s)
{
    const int threads = 256;  // 8 rows per block
    long long blocks = ((long long)rows + 7) / 8;
    if (blocks > 65535LL * 4)
        blocks = 65535LL * 4;
    merge_lse_kernel<<<(unsigned)blocks, threads, 0, s>>>(
        reinterpret_cast<const float4 *>(oa), sa, reinterpret_cast<const float4 *>(ob), sb, rows,
        d / 4, reinterpret_cast<float4 *>(out), sout);
    return cudaGetLastError();
}

// Self-test of the bounded wait every kernel uses on its copies: one warp
// waits, with that same wait, on an mbarrier that nothing completes.  The
// wait gives up after its limit (1 s) and the kernel records a timeout in
// the status word, as a kernel whose copies never landed would; then it
// ends, and the context stays usable.
__global__ void wait_selftest_kernel(unsigned *status)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0)
        mbar_init(b, 1);
    fence_mbar_init();
    __syncthreads();
    if (!mbar_wait_bounded(b, 0) && threadIdx.x == 0)
        atomicOr(status, STATUS_TIMEOUT);
}

cudaError_t launch_wait_selftest(unsigned *status, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 32, 0, s>>>(status);
    return cudaGetLastError();
}

static cudaError_t launch_combine(const CombineParams &p, bool lse_form, cudaStream_t s)
{
    const size_t smem = (size_t)p.P * sizeof(float);
    if (lse_form) {
        auto k = combine_kernel<true>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        k<<<p.rows, COMBINE_THREADS, smem, s>>>(p);
    } else {
        auto k = combine_kernel<false>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        k<<<p.rows, COMBINE_THREADS, smem, s>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_combine_mlo(const CombineParams &p, cudaStream_t s) { return launch_combine(p, false, s); }
cudaError_t launch_combine_lse(const CombineParams &p, cudaStream_t s) { return launch_combine(p, true, s); }

}  // namespace fd
