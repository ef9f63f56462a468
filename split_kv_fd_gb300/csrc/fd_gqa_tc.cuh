// fd_gqa_tc.cuh -- grouped-query decode for large groups (MQA and GQA with
// many query heads per K/V head, "从第一性原理推导 Flash Attention" §8) on
// the fifth-generation tensor cores: tcgen05.mma with operands in shared
// memory and accumulators in tensor memory (TMEM).
//
// Per (b, K/V head) and chunk of CT = 64 tokens the work is two dense
// products over all the K/V head's query heads at once (up to 128, the MMA's
// M; more are served in slices by adjacent CTAs):
//     S [128 x CT] = Q [128 x d] . K_chunk^T      (TMEM, fp32)
//     O [128 x d] += P [128 x CT] . V_chunk       (TMEM, fp32, the whole segment)
// so every K/V byte enters shared memory once per CTA, whatever the number
// of query heads (the mma.sync kernel of fd_gqa.cuh stages a chunk once per
// 16 heads).  The online softmax between the two products runs in fp32
// registers, one thread per query head (TMEM lane = MMA row = head):
//  - S is read with tcgen05.ld; the scores past the chunk's tokens are
//    masked; P = 2^(s - m_ref) is split into a 16-bit high part and the
//    16-bit remainder, both written to shared memory (K-major, 128-byte
//    swizzle), and the two products P_hi V + P_lo V keep P.V close to fp32
//    accuracy with 16-bit operands.
//  - The rescale of the block-wise update ("FlashDecoding 数学推导" §2.4.1:
//    acc and l times exp(m_old - m_new) when the max grows) is done lazily:
//    the reference max m_ref moves only when a chunk's max exceeds it by
//    more than TAU (in base 2), and only then is the head's O row in TMEM
//    rescaled (tcgen05.ld, multiply, tcgen05.st).  In between, P may reach
//    2^TAU, which fp32 and the 16-bit high part hold exactly enough; the
//    result is the same quotient (o = acc / l with both relative to m_ref).
//
// Warp roles (192 threads, one CTA per SM):
//  - warps 0-3: softmax, one query head per thread (TMEM lanes 0-127);
//  - warp 4: the producer, K and V chunks by tensor-map TMA into a ring of
//    STAGES stages (128 KB in flight, as in the other kernels);
//  - warp 5: allocates TMEM; its lane 0 issues the MMAs.
// Two S buffers in TMEM let the MMA warp compute S for chunk c + 1 while the
// softmax threads work on chunk c; P.V of chunk c runs while they read S of
// chunk c + 1.  Every hand-off is an mbarrier (the MMA warp's through
// tcgen05.commit), and every wait is bounded: on expiry a role records
// FD_ERR_DEVICE_TIMEOUT, stops, drains what it issued and the CTA frees its
// TMEM.
//
// The decomposition, slots, arrival counters and merges are those of the
// grouped-query kernel (fd_gqa.cuh): same workspace layout, same results up
// to fp32 rounding.
#pragma once

#include "fd_gqa.cuh"
#include "fd_tc.cuh"

// Groups of at least this many query heads per K/V head run this kernel
// (16-bit K/V, contiguous cache, head dim 64 or 128).
#ifndef FD_GQA_TC_MIN_G
#define FD_GQA_TC_MIN_G 17
#endif

namespace fd {

template <typename T, int D> struct TcCfg {
    static constexpr bool F8K = false;             // (TmaProducer) 16-bit K/V by tensor maps
    static constexpr bool F8REG = false;
    static constexpr int CT = 64;                  // tokens per chunk: N of S, K of P.V
    static constexpr int M = 128;                  // query-head rows of the MMAs (TMEM lanes)
    static constexpr int MAXG = M;
    static constexpr int LINES = D / 64;           // 128-byte planes of a row
    static constexpr int ROW = D * 2;
    static constexpr int PLANE = CT * 128;         // one 64-element plane of a chunk
    static constexpr int CHUNK_BYTES = CT * ROW;   // K or V of one chunk
    static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;
    static constexpr int STAGES = (128 * 1024) / STAGE_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int QPLANE = M * 128;         // one 64-element plane of Q
    static constexpr int Q_BYTES = LINES * QPLANE;
    static constexpr int PHALF = M * CT * 2;       // P_hi (then P_lo): [M][CT] 16-bit, one plane
    static constexpr int P_BYTES = 2 * PHALF;
    static constexpr int SOFT_THREADS = 128, PROD_WARP = 4, MMA_WARP = 5, THREADS = 192;
    // mbarriers: full[STAGES], empty[STAGES], s_full[2], s_free[2], q_full, p_full, o_full, fin,
    // and the softmax warps' segment-end barrier
    static constexpr int NBAR = 2 * STAGES + 9;
    static constexpr int TMEM_O = 2 * CT;          // S buffers at columns 0 and CT, O after them
    static constexpr uint32_t TMEM_COLS = (2 * CT + D) <= 256 ? 256u : 512u;
    static constexpr float TAU = 8.f;              // lazy-rescale threshold (base 2)
    static constexpr int MERGE_PB = 64;            // pieces merged with weights in shared memory
    static_assert(D == 64 || D == 128, "head dim 64 or 128");
    static_assert(CT == 64, "P is one 128-byte plane per row");
    static_assert(RING_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0 && PHALF % 1024 == 0, "1024-byte atoms");
    // the last arriver's merge scratch lives in the Q and P buffers
    static_assert(MERGE_PB * 8 + MERGE_PB * MAXG * 4 + 2 * MAXG * 4 <= Q_BYTES + P_BYTES, "merge scratch");

    static size_t smem_bytes(int decomp, int B)
    {
        size_t s = 1024 + RING_BYTES + Q_BYTES + P_BYTES + NBAR * 8 + 16;
        if (decomp == DECOMP_BALANCED)
            s += (size_t)(B + 1) * 8 + (size_t)B * 4;
        return s;
    }
};

// A barrier of the 4 softmax warps on an mbarrier (count 4), with the
// bounded wait: a warp whose partner gave up does not hang here.  `phase`
// is the parity of the next completion; every softmax thread runs the same
// sequence of syncs.  Returns false on expiry.
struct SoftBar {
    uint32_t bar;
    uint32_t phase;
    __device__ __forceinline__ bool sync(int lane)
    {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar);
        const bool ok = mbar_wait_bounded(bar, phase);
        phase ^= 1u;
        return ok;
    }
};

// Stage 2 of a (b, virtual head) by the last piece to arrive, on the 128
// softmax threads: the m/l/o merge ("FlashDecoding 数学推导" §2.4.2) of the
// `target` workspace partials of each of its Gv query rows.  With at most
// MERGE_PB pieces the per-(piece, head) weights are formed once in `scr`
// (the free Q and P buffers); otherwise each output element walks the
// pieces itself.
template <int D, int MERGE_PB>
__device__ __forceinline__ bool tc_merge_pieces(const GqaParams &gp, const Ctx &ctx, long long bhv, int slice,
                                                int G, int Gv, long long qrow0, unsigned target, int gf,
                                                long long off, int tid, unsigned char *scr, SoftBar &sb)
{
    const SplitParams &p = gp.s;
    const int n = (int)target;
    if (n > MERGE_PB) {
        for (int idx = tid; idx < Gv * D; idx += 128) {
            const int g = idx / D, dim = idx % D;
            float M = -INFINITY;
            for (int i = 0; i < n; ++i) {
                const long long r = vh_slot(gp, ctx, bhv, (unsigned)i, gf, off, slice) * G + g;
                if (__ldcg(p.ws_ml + 2 * r + 1) > 0.f)
                    M = fmaxf(M, __ldcg(p.ws_ml + 2 * r));
            }
            float L = 0.f, O = 0.f;
            for (int i = 0; i < n; ++i) {
                const long long r = vh_slot(gp, ctx, bhv, (unsigned)i, gf, off, slice) * G + g;
                const float l = __ldcg(p.ws_ml + 2 * r + 1);
                if (l > 0.f) {
                    const float e = ex2(__ldcg(p.ws_ml + 2 * r) - M) * l;
                    L += e;
                    O = fmaf(e, __ldcg(p.ws_o + r * D + dim), O);
                }
            }
            const long long qrow = qrow0 + g;
            store_out(p.out, qrow * D + dim, p.out_dtype, L > 0.f ? O / L : 0.f);
            if (dim == 0 && p.lse)
                p.lse[qrow] = L > 0.f ? (M + log2f(L)) * LN2_F : -INFINITY;
        }
        return true;
    }
    long long *ss = reinterpret_cast<long long *>(scr);            // [n] slots
    float *wt = reinterpret_cast<float *>(scr + MERGE_PB * 8);      // [n][G] weights
    float *sM = wt + MERGE_PB * G;                                   // [G]
    float *sL = sM + G;                                              // [G]
    for (int i = tid; i < n; i += 128)
        ss[i] = vh_slot(gp, ctx, bhv, (unsigned)i, gf, off, slice);
    if (!sb.sync(tid & 31))
        return false;
    if (tid < Gv) {
        float M = -INFINITY;
        for (int i = 0; i < n; ++i) {
            const long long r = ss[i] * G + tid;
            const float l = __ldcg(p.ws_ml + 2 * r + 1);
            const float m = __ldcg(p.ws_ml + 2 * r);
            wt[i * G + tid] = l;
            if (l > 0.f)
                M = fmaxf(M, m);
        }
        float L = 0.f;
        for (int i = 0; i < n; ++i) {
            const long long r = ss[i] * G + tid;
            const float l = wt[i * G + tid];
            const float e = l > 0.f ? ex2(__ldcg(p.ws_ml + 2 * r) - M) * l : 0.f;
            wt[i * G + tid] = e;
            L += e;
        }
        sM[tid] = M;
        sL[tid] = L;
    }
    if (!sb.sync(tid & 31))
        return false;
    for (int idx = tid; idx < Gv * D; idx += 128) {
        const int g = idx / D, dim = idx % D;
        float O = 0.f;
#pragma unroll 4
        for (int i = 0; i < n; ++i) {
            const float e = wt[i * G + g];
            if (e > 0.f)
                O = fmaf(e, __ldcg(p.ws_o + (ss[i] * G + g) * D + dim), O);
        }
        const float L = sL[g];
        const long long qrow = qrow0 + g;
        store_out(p.out, qrow * D + dim, p.out_dtype, L > 0.f ? O / L : 0.f);
        if (dim == 0 && p.lse)
            p.lse[qrow] = L > 0.f ? (sM[g] + log2f(L)) * LN2_F : -INFINITY;
    }
    return true;
}

template <typename T, int D>
__global__ void __launch_bounds__(TcCfg<T, D>::THREADS, 1) gqa_tc_kernel(const __grid_constant__ GqaParams gp)
{
    using C = TcCfg<T, D>;
    constexpr int ST = C::STAGES;
    const SplitParams &p = gp.s;
    const int G = gp.G;   // query heads per slice (<= 128): row stride of the workspace
    const int slice = (int)(blockIdx.x % gp.NG);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int w = tid >> 5;
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);   // 1024-aligned
    const uint32_t ring = smem_addr(smem);
    const uint32_t qbuf = ring + C::RING_BYTES;
    const uint32_t pbuf = qbuf + C::Q_BYTES;
    unsigned char *scratch = smem + C::RING_BYTES;   // Q and P buffers, reused by the merge
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::RING_BYTES + C::Q_BYTES + C::P_BYTES);
    uint32_t *misc = reinterpret_cast<uint32_t *>(bars + C::NBAR);   // [0] TMEM base, [1] flag
    long long *cumH = reinterpret_cast<long long *>(misc + 4);
    int *lenS = reinterpret_cast<int *>(cumH + p.B + 1);
    const uint32_t bar0 = smem_addr(bars);
    auto FULL = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto EMPTY = [&](int s) { return bar0 + 8u * (uint32_t)(ST + s); };
    auto SFULL = [&](int b) { return bar0 + 8u * (uint32_t)(2 * ST + b); };
    auto SFREE = [&](int b) { return bar0 + 8u * (uint32_t)(2 * ST + 2 + b); };
    const uint32_t QFULL = bar0 + 8u * (2 * ST + 4);
    const uint32_t PFULL = bar0 + 8u * (2 * ST + 5);
    const uint32_t OFULL = bar0 + 8u * (2 * ST + 6);
    const uint32_t FIN = bar0 + 8u * (2 * ST + 7);
    const uint32_t SEGBAR = bar0 + 8u * (2 * ST + 8);

    if (tid == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(FULL(s), 1);    // the producer's arrival plus the copies' bytes
            mbar_init(EMPTY(s), 1);   // the MMA warp's commit after P.V of the stage's chunk
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(SFULL(b), 1);   // commit after S
            mbar_init(SFREE(b), 4);   // the softmax warps have read S
        }
        mbar_init(QFULL, 4);          // the softmax warps have written Q
        mbar_init(PFULL, 4);          // ... P (and zeroed V's rows past the chunk)
        mbar_init(OFULL, 1);          // commit after P.V
        mbar_init(FIN, 1);            // the MMA warp's last commit
        mbar_init(SEGBAR, 4);         // the softmax warps at a segment end
        prefetch_tmap(&gp.tmk);
        prefetch_tmap(&gp.tmv);
    }
    if (w == C::MMA_WARP) {
        tmem_alloc(smem_addr(misc), C::TMEM_COLS);
        tmem_relinquish();
    }

    Ctx ctx;
    ctx.g = (int)(blockIdx.x / gp.NG);
    ctx.G = p.grid / gp.NG;
    ctx.cumH = cumH;
    ctx.lenS = lenS;
    ctx.T = 0;
    ctx.Geff = 0;
    ctx.beg = ctx.end = 0;
    if (p.decomp == DECOMP_BALANCED) {
        balanced_setup<C::THREADS, C::THREADS / 32>(p, ctx, cumH, lenS);
        // (b, K/V head) of length 0 are touched by no CTA: write their Gq rows here
        for (long long bh = (long long)blockIdx.x * C::THREADS + tid; bh < (long long)p.B * p.H;
             bh += (long long)gridDim.x * C::THREADS) {
            if (lenS[bh / p.H] == 0) {
                const long long q0 = vh_qrow0(gp, (int)(bh / p.H), (int)(bh % p.H) * gp.NG);
                for (int g = 0; g < gp.Gq; ++g) {
                    for (int i = 0; i < D; ++i)
                        store_out(p.out, (q0 + g) * D + i, p.out_dtype, 0.f);
                    if (p.lse)
                        p.lse[q0 + g] = -INFINITY;
                }
            }
        }
    }
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    bool dead = false;

    if (w == C::PROD_WARP) {
        // ------------------------------------------------------------ producer
        TmaProducer<C, false> prod;
        prod.start(gp, ctx, 0, 1);
        int issued = 0;
#pragma unroll 1
        for (;;) {
            const int s = issued % ST;
            if (issued >= ST && !mbar_wait_bounded(EMPTY(s), ((issued / ST) - 1) & 1)) {
                dead = true;
                break;
            }
            if (!prod.issue(gp, ctx, ring + (uint32_t)(s * C::STAGE_BYTES), FULL(s), lane))
                break;
            ++issued;
        }
        // no copy may be in flight when the CTA ends: the last fill of each stage
        for (int i = max(0, issued - ST); i < issued; ++i)
            mbar_wait_bounded(FULL(i % ST), (i / ST) & 1);
    } else if (w == C::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr int BF = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
            constexpr uint32_t ID_S = idesc_f16(BF, 0, 0, C::M, C::CT);   // Q K-major, K K-major
            constexpr uint32_t ID_O = idesc_f16(BF, 0, 1, C::M, D);       // P K-major, V MN-major
            long long i = 0;   // chunks of this CTA so far
            int k = 0;         // non-empty segments so far
            // S of chunk j (global index) into S buffer j % 2
            auto issue_s = [&](long long j) -> bool {
                const int s = (int)(j % ST);
                if (!mbar_wait_bounded_thread(FULL(s), (uint32_t)((j / ST) & 1)))
                    return false;
                if (j >= 2 && !mbar_wait_bounded_thread(SFREE((int)(j & 1)), (uint32_t)(((j >> 1) - 1) & 1)))
                    return false;
                tc_fence_after();
                const uint32_t kb = ring + (uint32_t)(s * C::STAGE_BYTES);
                const uint32_t ds = tmem + (uint32_t)((j & 1) * C::CT);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t col = (uint32_t)((ks & 3) * 32);   // 16 elements = 32 bytes per k-step
                    const uint64_t a = smem_desc_sw128(qbuf + (uint32_t)((ks >> 2) * C::QPLANE) + col, 16, 1024);
                    const uint64_t b = smem_desc_sw128(kb + (uint32_t)((ks >> 2) * C::PLANE) + col, 16, 1024);
                    tc_mma_ss(ds, a, b, ID_S, ks > 0 ? 1u : 0u);
                }
                tc_commit(SFULL((int)(j & 1)));
                return true;
            };
            Seg cs;
            seg_first(p, ctx, cs);
#pragma unroll 1
            while (cs.valid && !dead) {
                const long long n = seg_chunks<C::CT>(cs);
                if (n > 0) {
                    if (!mbar_wait_bounded_thread(QFULL, (uint32_t)(k & 1))) {
                        dead = true;
                        break;
                    }
                    ++k;
                    tc_fence_after();
                    if (!issue_s(i)) {
                        dead = true;
                        break;
                    }
#pragma unroll 1
                    for (long long c = 0; c < n; ++c, ++i) {
                        if (c + 1 < n && !issue_s(i + 1)) {
                            dead = true;
                            break;
                        }
                        if (!mbar_wait_bounded_thread(PFULL, (uint32_t)(i & 1))) {
                            dead = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t vb = ring + (uint32_t)((i % ST) * C::STAGE_BYTES + C::CHUNK_BYTES);
#pragma unroll
                        for (int ks = 0; ks < C::CT / 16; ++ks) {
#pragma unroll
                            for (int hl = 0; hl < 2; ++hl) {
                                const uint64_t a =
                                    smem_desc_sw128(pbuf + (uint32_t)(hl * C::PHALF + ks * 32), 16, 1024);
                                const uint64_t b =
                                    smem_desc_sw128(vb + (uint32_t)(ks * 2048), (uint32_t)C::PLANE, 1024);
                                tc_mma_ss(tmem + C::TMEM_O, a, b, ID_O, (c > 0 || ks > 0 || hl > 0) ? 1u : 0u);
                            }
                        }
                        tc_commit(OFULL);
                        tc_commit(EMPTY((int)(i % ST)));
                    }
                }
                seg_next(p, ctx, cs);
            }
            // every MMA this thread issued has completed before TMEM is freed
            tc_commit(FIN);
            if (!mbar_wait_bounded_thread(FIN, 0))
                dead = true;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int row = tid;   // query head within the slice = TMEM lane
        const uint32_t tl = tmem + ((uint32_t)(w * 32) << 16);
        SoftBar sb{SEGBAR, 0u};
        long long i = 0;
        Seg cs;
        seg_first(p, ctx, cs);
#pragma unroll 1
        while (cs.valid && !dead) {
            const long long n = seg_chunks<C::CT>(cs);
            const int vh = cs.h * gp.NG + slice;
            const long long bhv = (long long)cs.b * p.H * gp.NG + vh;
            const int gv = vh_count(gp, vh);
            const long long qrow0 = vh_qrow0(gp, cs.b, vh);
            const bool live = row < gv;
            float m_ref = -INFINITY, l = 0.f;
            if (n > 0) {
                // this head's q row into the Q buffer (K-major, 128-byte swizzle)
                {
                    const uint4 *qs = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.q) +
                                                                      (qrow0 + row) * D);
#pragma unroll
                    for (int pl = 0; pl < C::LINES; ++pl)
#pragma unroll
                        for (int c16 = 0; c16 < 8; ++c16) {
                            const uint4 v = live ? __ldg(qs + pl * 8 + c16) : make_uint4(0, 0, 0, 0);
                            const uint32_t a = qbuf + (uint32_t)(pl * C::QPLANE + row * 128 +
                                                                 ((c16 ^ (row & 7)) << 4));
                            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x),
                                         "r"(v.y), "r"(v.z), "r"(v.w)
                                         : "memory");
                        }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(QFULL);
#pragma unroll 1
                for (long long c = 0; c < n; ++c, ++i) {
                    if (!mbar_wait_bounded(SFULL((int)(i & 1)), (uint32_t)((i >> 1) & 1))) {
                        dead = true;
                        break;
                    }
                    tc_fence_after();
                    float s0[32], s1[32];   // the head's scores of the chunk's 64 tokens
                    tmem_ld32(tl + (uint32_t)((i & 1) * C::CT), s0);
                    tmem_ld32(tl + (uint32_t)((i & 1) * C::CT + 32), s1);
                    tmem_wait_ld();
                    auto S = [&](int j) -> float & { return j < 32 ? s0[j] : s1[j - 32]; };
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(SFREE((int)(i & 1)));
                    int t, ntok;
                    chunk_coords<C::CT>(cs, c, t, ntok);
                    float mc = -INFINITY;
#pragma unroll
                    for (int j = 0; j < C::CT; ++j) {
                        S(j) = j < ntok ? S(j) * p.scale_log2 : -INFINITY;
                        mc = fmaxf(mc, S(j));
                    }
                    // P.V of the previous chunk is done: its P buffer is free and O is final
                    if (c > 0) {
                        if (!mbar_wait_bounded(OFULL, (uint32_t)((i - 1) & 1))) {
                            dead = true;
                            break;
                        }
                        tc_fence_after();
                    }
                    // lazy rescale: the reference max moves only when the
                    // chunk's max exceeds it by more than TAU
                    const bool grow = mc > m_ref + C::TAU;
                    float a = 1.f;
                    if (grow) {
                        a = ex2(m_ref - mc);   // 0 on the first chunk
                        l *= a;
                        m_ref = mc;
                    }
                    // the O rows in TMEM: the tcgen05 loads and stores are
                    // warp-wide, so the whole warp runs them when any of its
                    // heads grew (a = 1 for the others)
                    if (c > 0 && __any_sync(FULL_MASK, grow)) {
#pragma unroll 1
                        for (int q4 = 0; q4 < D / 32; ++q4) {
                            float o[32];
                            tmem_ld32(tl + (uint32_t)(C::TMEM_O + 32 * q4), o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] *= a;
                            tmem_st32(tl + (uint32_t)(C::TMEM_O + 32 * q4), o);
                        }
                        tmem_wait_st();
                    }
                    // P = 2^(s - m_ref), high part and remainder, into the P buffer
                    float ls = 0.f;
#pragma unroll
                    for (int c16 = 0; c16 < 8; ++c16) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = c16 * 8 + 2 * e;
                            const float p0 = live ? ex2(S(j) - m_ref) : 0.f;
                            const float p1 = live ? ex2(S(j + 1) - m_ref) : 0.f;
                            ls += p0 + p1;
                            hi[e] = Mma<T>::pack(p0, p1);
                            const float2 u = Mma<T>::unpack(hi[e]);
                            lo[e] = Mma<T>::pack(p0 - u.x, p1 - u.y);
                        }
                        const uint32_t off = (uint32_t)(row * 128 + ((c16 ^ (row & 7)) << 4));
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(pbuf + off), "r"(hi[0]),
                                     "r"(hi[1]), "r"(hi[2]), "r"(hi[3])
                                     : "memory");
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(pbuf + C::PHALF + off),
                                     "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3])
                                     : "memory");
                    }
                    l += ls;
                    // V's rows past the chunk's tokens may hold padding (NaN * 0 is NaN)
                    if (ntok < C::CT) {
                        const uint32_t vb = ring + (uint32_t)((i % ST) * C::STAGE_BYTES + C::CHUNK_BYTES);
                        const int pieces = (C::CT - ntok) * C::LINES * 8;
                        for (int x = tid; x < pieces; x += 128) {
                            const int r = ntok + x / (C::LINES * 8);
                            const int rem = x % (C::LINES * 8);
                            const uint32_t a = vb + (uint32_t)((rem >> 3) * C::PLANE + r * 128 + (rem & 7) * 16);
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(PFULL);
                }
                if (dead)
                    break;
                if (!mbar_wait_bounded(OFULL, (uint32_t)((i - 1) & 1))) {
                    dead = true;
                    break;
                }
                tc_fence_after();
            }

            // ---- segment end: this head's (o, m, l) ----
            const int len = (p.decomp == DECOMP_BALANCED) ? lenS[cs.b] : clamp_len(p, cs.b);
            bool complete;
            long long slot;
            if (p.decomp == DECOMP_SPLITS) {
                complete = (p.P == 1);
                slot = bhv * p.P + cs.p;
            } else {
                complete = (cs.t0 == 0 && cs.t1 == len);
                slot = 2LL * blockIdx.x + (cs.k == 0 ? 0 : 1);
            }
            const bool nonempty = l > 0.f;
            const float inv = nonempty ? 1.f / l : 0.f;
            const long long qrow = qrow0 + row;
            const long long r = slot * G + row;
#pragma unroll 1
            for (int q4 = 0; q4 < D / 32; ++q4) {
                float o[32];
                if (n > 0) {
                    tmem_ld32(tl + (uint32_t)(C::TMEM_O + 32 * q4), o);
                    tmem_wait_ld();
                }
                if (live) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float x = (n > 0 && nonempty) ? o[e] * inv : 0.f;
                        if (complete)
                            store_out(p.out, qrow * D + 32 * q4 + e, p.out_dtype, x);
                        else
                            p.ws_o[r * D + 32 * q4 + e] = x;
                    }
                }
            }
            tc_fence_before();
            if (live) {
                if (complete) {
                    if (p.lse)
                        p.lse[qrow] = nonempty ? (m_ref + log2f(l)) * LN2_F : -INFINITY;
                } else {
                    p.ws_ml[2 * r] = nonempty ? m_ref : -INFINITY;
                    p.ws_ml[2 * r + 1] = l;
                }
            }
            if (!complete) {
                unsigned target;
                int gf = 0;
                long long off = 0;
                if (p.decomp == DECOMP_SPLITS) {
                    target = (unsigned)p.P;
                } else {
                    off = ctx.cumH[cs.b] + (long long)cs.h * len;
                    gf = bal_owner(off, ctx.T, ctx.Geff);
                    const int gl = bal_owner(off + len - 1, ctx.T, ctx.Geff);
                    target = (unsigned)(gl - gf + 1);
                }
                // the barrier orders every thread's partial before thread 0's
                // fence and arrival
                if (!sb.sync(lane)) {
                    dead = true;
                    break;
                }
                if (tid == 0) {
                    __threadfence();
                    const unsigned old = atomicInc(p.ws_cnt + bhv, target - 1);
                    misc[1] = (old == target - 1) ? 1u : 0u;
                }
                if (!sb.sync(lane)) {
                    dead = true;
                    break;
                }
                if (misc[1]) {
                    __threadfence();
                    if (!tc_merge_pieces<D, C::MERGE_PB>(gp, ctx, bhv, slice, G, gv, qrow0, target, gf, off,
                                                         tid, scratch, sb)) {
                        dead = true;
                        break;
                    }
                }
                if (!sb.sync(lane)) {   // the flag and the scratch are reused
                    dead = true;
                    break;
                }
            }
            seg_next(p, ctx, cs);
        }
    }

    if (dead && lane == 0)
        atomicOr(p.status, STATUS_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (w == C::MMA_WARP)
        tmem_dealloc(tmem, C::TMEM_COLS);
}

template <typename T, int D> static cudaError_t launch_gqa_tc_t(const GqaParams &gp, cudaStream_t s)
{
    using C = TcCfg<T, D>;
    const size_t smem = C::smem_bytes(gp.s.decomp, gp.s.B);
    auto kern = gqa_tc_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kern<<<gp.s.grid, C::THREADS, smem, s>>>(gp);
    return cudaGetLastError();
}

}  // namespace fd
