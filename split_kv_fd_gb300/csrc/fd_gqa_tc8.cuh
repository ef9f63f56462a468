// fd_gqa_tc8.cuh -- grouped-query decode over an E4M3 KV cache ("从第一性原理推导
// Flash Attention" §6.2 FP8 storage, §8 GQA) with both products on the
// fifth-generation tensor cores in FP8 (tcgen05.mma kind::f8f6f4), straight
// from the staged cache bytes: no K or V byte is converted.
//
// Per (b, K/V head) and chunk of CT = 128 tokens, for a slice of up to 8
// query heads:
//     S^T [128 tokens x 32] = K_chunk [128 x d] . Qp^T     (K and Qp in shared memory)
//     O^T [d x 32]         += V_chunk^T [d x 128] . Pp^T   (V MN-major, Pp^T in shared memory)
// The 32 columns are the heads' parts: q and P are not E4M3 values, so each
// is split into three E4M3 parts of decreasing weight (column 8p + h holds
// part p of head h; p = 0, 1, 2 weigh 1, 2^-4, 2^-8):
//     x = x0 + 2^-4 x1 + 2^-8 x2,   x0 = e4m3(x), x1 = e4m3(16 (x - x0)), ...
// Each part takes the rounding error of the one before it times 16, so the
// three keep about 12 significant bits (one E4M3 has 4), as much as the f16
// rounding of q in the mma.sync kernel; the products of E4M3 values are
// exact and summed in fp32.  q of head h is first brought to amax in
// [128, 256) by a power of two 2^e_h (exact), undone in its score scale.
//
// The online softmax runs one thread per token (TMEM lane = S^T row):
//  - the three part columns of each head are summed with their weights and
//    scaled to base-2 scores x;
//  - the running max ("FlashDecoding 数学推导" §2.4.1) is lazy and shared by
//    the 128 tokens of a softmax group: each chunk the group's warps vote
//    whether any score exceeds its head's reference max m by more than TAU;
//    only then do they reduce the chunk's max per head, move m and rescale
//    the head's l and O^T columns (TMEM; every warp its 32 lanes of d);
//  - P = 2^(x - m + 6) <= 256 (within E4M3's 448), split into its parts and
//    written, one byte per (part, head), as the rows of Pp^T; l sums P per
//    thread and is reduced over the group at the segment end.
//
// Warp roles (384 threads, one CTA per SM): warps 0-3 and 4-7 are two
// softmax groups taking the chunks in pairs, in turn, each with its own O^T
// and (m, l); warps 8 and 9 the K and V producers (one 128-byte swizzled
// tensor-map box of 128 rows per copy; K and V have rings of their own, a K
// buffer being free once S^T is done, a V buffer once P.V is); warp 10
// allocates TMEM and issues S^T as soon as a chunk's K has landed; warp 11
// issues P.V.  The two groups' states are merged at each segment end
// ("FlashDecoding 数学推导" §2.4.2).  Every hand-off is an mbarrier and every
// wait is bounded (FD_ERR_DEVICE_TIMEOUT on expiry).
//
// The decomposition, slices (of at most 8 heads), workspace layout,
// arrival counters and merges are those of the E4M3 mma.sync kernel
// (fd_gqa.cuh).
#pragma once

#include "fd_gqa_tc.cuh"

namespace fd {

template <int D> struct Tc8Cfg {
    static constexpr bool F8K = true;              // (TmaProducer) E4M3 rows, one swizzled box per operand
    static constexpr bool F8REG = true;
    static constexpr int CT = 128;                 // tokens per chunk: M of S^T, K of P.V
    static constexpr int M = 128;
    static constexpr int MAXG = 8;                 // query heads per slice
    static constexpr int NC = 32;                  // columns: 3 parts x 8 heads, padded
    static constexpr int ROW = D;                  // bytes per token row
    static constexpr int LINES = 1;
    static constexpr int CHUNK_BYTES = CT * ROW;   // K or V of one chunk
    static constexpr int QP_BYTES = NC * D;        // q parts: NC rows of d bytes (two buffers, by segment)
    static constexpr int NWG = 2;                  // softmax groups (4 warps each), pairs of chunks in turn
    static constexpr int NPB = 2 * NWG;            // Pp^T buffers (chunk j in j % NPB)
    static constexpr int PT_BYTES = NC * CT;       // one Pp^T: NC rows of CT bytes
    static constexpr int NSB = 12;                 // S^T buffers in TMEM (chunk j in j % NSB)
    static constexpr int TMEM_O = NSB * NC;        // then the groups' O^T, two sets (by segment)
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int MERGE_PB = 64;
    static constexpr int SCR_BYTES = MERGE_PB * 8 + 2 * MAXG * 4;
    // per group: vote flags [2][4], chunk maxima [4][8]; per segment parity:
    // l sums [NWG][4][8] and m [NWG][8], and the heads' score scales [8]
    static constexpr int SEGX = NWG * 4 * 8 + NWG * 8;
    static constexpr int XCH_FLOATS = NWG * 2 * 4 + NWG * 4 * 8 + 2 * SEGX + 2 * 8;
    static constexpr int XCH_BYTES = (XCH_FLOATS * 4 + 15) / 16 * 16;
    // warps 0 .. 4 NWG - 1: the softmax groups; then four epilogue warps,
    // the K and V producers, the S^T issuer (it allocates TMEM) and the P.V
    // issuer
    static constexpr int WG_THREADS = 128, EPI_WARP = 4 * NWG, KPROD_WARP = EPI_WARP + 4;
    static constexpr int VPROD_WARP = KPROD_WARP + 1;
    static constexpr int S_WARP = KPROD_WARP + 2, PV_WARP = KPROD_WARP + 3;
    static constexpr int THREADS = 32 * (4 * NWG + 8);
    // mbarriers: full/empty of the K and V buffers, s_full[NSB],
    // s_free[NSB], p_full[NPB], pv_done[NPB], fin (2), epi, wg[NWG], and by
    // segment parity q_full, seg_done, o_free
    // every wait suspends the waiting thread in hardware (woken when the
    // phase completes) rather than polling, so that waiting warps leave the
    // issue slots to the working ones
    static constexpr uint32_t SLEEP_NS = 100000;
    static constexpr float TAU = 2.f;              // lazy-rescale threshold (base 2)
    static constexpr float PEXP = 8.f - TAU;       // P is taken times 2^PEXP: at most 2^8
    // K and V have rings of their own: a K buffer is free again once S^T of
    // its chunk is done, a V buffer only once P.V is, after the softmax of
    // (up to two pairs of) chunks; so V gets what is left of 227 KB beside
    // KST K buffers and the rest, the prefix sums of up to BALANCED_MAX_B
    // sequences included (two barriers per buffer)
    static constexpr int KST = 4;
    static constexpr int NBAR_FIXED = 2 * KST + 2 * NSB + 2 * NPB + 3 + NWG + 6;
    static constexpr int FIXED = 1024 + KST * CHUNK_BYTES + 2 * QP_BYTES + NPB * PT_BYTES + SCR_BYTES + XCH_BYTES +
                                 NBAR_FIXED * 8 + 16 + (BALANCED_MAX_B + 1) * 8 + BALANCED_MAX_B * 4;
    static constexpr int VST = (227 * 1024 - FIXED) / (CHUNK_BYTES + 16);
    static constexpr int RING_BYTES = (KST + VST) * CHUNK_BYTES;   // K buffers, then V buffers
    static constexpr int NBAR = 2 * VST + NBAR_FIXED;
    static_assert(D == 128, "head dim 128");
    static_assert(VST >= 4, "ring depth");
    static_assert(1024 + RING_BYTES + 2 * QP_BYTES + NPB * PT_BYTES + SCR_BYTES + XCH_BYTES + NBAR * 8 + 16 +
                          (BALANCED_MAX_B + 1) * 8 + BALANCED_MAX_B * 4 <= 227 * 1024,
                  "shared memory");
    static_assert(TMEM_O + 2 * NWG * NC <= (int)TMEM_COLS, "TMEM columns");
    static_assert(RING_BYTES % 1024 == 0 && QP_BYTES % 1024 == 0 && PT_BYTES % 1024 == 0, "1024-byte atoms");

    static size_t smem_bytes(int decomp, int B)
    {
        size_t s = 1024 + RING_BYTES + 2 * QP_BYTES + NPB * PT_BYTES + SCR_BYTES + XCH_BYTES + NBAR * 8 + 16;
        if (decomp == DECOMP_BALANCED)
            s += (size_t)(B + 1) * 8 + (size_t)B * 4;
        return s;
    }
};

// Two floats as an E4M3 pair (round to nearest even, saturating to +-448):
// a in the low byte, b in the high byte.
__device__ __forceinline__ uint32_t e4m3x2_rn(float a, float b)
{
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(b), "f"(a));
    return (uint32_t)h;
}

// An E4M3 pair (low byte first) back to two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t v)
{
    uint32_t f;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f) : "h"((uint16_t)v));
    __half2 h;
    memcpy(&h, &f, 4);
    return __half22float2(h);
}

// The three E4M3 parts (weights 1, 2^-4, 2^-8) of a pair of values, as
// three E4M3 pairs.
__device__ __forceinline__ void e4m3_parts2(float a, float b, uint32_t &p0, uint32_t &p1, uint32_t &p2)
{
    p0 = e4m3x2_rn(a, b);
    const float2 f0 = e4m3x2_to_f2(p0);
    const float ra = (a - f0.x) * 16.f, rb = (b - f0.y) * 16.f;
    p1 = e4m3x2_rn(ra, rb);
    const float2 f1 = e4m3x2_to_f2(p1);
    p2 = e4m3x2_rn((ra - f1.x) * 16.f, (rb - f1.y) * 16.f);
}

// Byte k of row n in a K-major operand of 128-byte rows written with the
// 128-byte swizzle (rows 1024-byte aligned in groups of 8).
__device__ __forceinline__ uint32_t sw128_byte(int n, int k)
{
    return (uint32_t)(n * 128 + (((k >> 4) ^ (n & 7)) << 4) + (k & 15));
}

__device__ __forceinline__ void st_u8(uint32_t a, uint32_t v)
{
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// One copy of the chunk at a producer cursor: the 128-byte swizzled box of
// its CT rows from `map` (K or V) into `dst`, completing on `bar`; then the
// cursor moves on.  Rows past the block's end read as zeros.
template <typename C>
__device__ __forceinline__ void tc8_issue(TmaProducer<C, false> &pr, const GqaParams &gp, const Ctx &ctx,
                                          const CUtensorMap *map, uint32_t dst, uint32_t bar)
{
    const SplitParams &p = gp.s;
    int y, blk;
    if (p.paged) {
        y = pr.t % p.page_size;
        blk = (int)(TmaProducer<C, false>::checked_page(p, pr.pg) * p.H + pr.s.h);
    } else {
        y = pr.t;
        blk = pr.s.b * p.H + pr.s.h;
    }
    mbar_arrive_expect_tx(bar, C::CHUNK_BYTES);
    tma_load_3d(dst, map, 0, y, blk, bar);
    pr.c += pr.stride;
    pr.locate(gp, ctx);
}

// The q parts of segment qs's slice of heads (K-major, 128-byte swizzle,
// row 8p + h for part p of head h; rows of heads past the slice stay zero)
// into the buffer at qb, and the heads' base-2 score scales into fh[8], on
// 128 threads (tid): 16 per head, 8 head dimensions each.  Each head's q is
// first brought to amax in [128, 256) by a power of two 2^e, and its score
// scale carries 2^-e.
template <int D>
__device__ __forceinline__ void tc8_prep_q(const GqaParams &gp, const Seg &qs, int slice, uint32_t qb, float *fh,
                                           int tid)
{
    const SplitParams &p = gp.s;
    const int vh = qs.h * gp.NG + slice;
    const int gv = vh_count(gp, vh);
    const long long qrow0 = vh_qrow0(gp, qs.b, vh);
    const int h = tid >> 4, sub = tid & 15;
    const bool live = h < gv;
    float qv[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = live ? q_pair_f32(p.q, p.q_dtype, (qrow0 + h) * D + sub * 8 + 2 * i) : make_float2(0.f, 0.f);
        qv[2 * i] = f.x;
        qv[2 * i + 1] = f.y;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        amax = fmaxf(amax, fabsf(qv[i]));
#pragma unroll
    for (int o = 1; o < 16; o <<= 1)
        amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, o));
    const int eb = (int)((__float_as_uint(amax) >> 23) & 0xff);
    // amax in [2^(eb-127), 2^(eb-126)): times 2^(134-eb); zero, subnormal,
    // infinite or NaN amax: unscaled
    const int e = (eb >= 8 && eb <= 254) ? 134 - eb : 0;
    const float up = pow2i(e);
    uint32_t pr[3][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        e4m3_parts2(qv[2 * i] * up, qv[2 * i + 1] * up, pr[0][i], pr[1][i], pr[2][i]);
#pragma unroll
    for (int pp = 0; pp < 3; ++pp) {
        const uint32_t lo = pr[pp][0] | (pr[pp][1] << 16), hi = pr[pp][2] | (pr[pp][3] << 16);
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(qb + sw128_byte(pp * 8 + h, sub * 8)), "r"(lo),
                     "r"(hi)
                     : "memory");
    }
    if (sub == 0)
        fh[h] = p.scale_log2 * __ldg(gp.k_scale + qs.b * p.H + qs.h) * pow2i(-e);
    fence_proxy_async_smem();
}

// A segment's result, on the epilogue warps ("FlashDecoding 数学推导"
// §2.4.2): the groups' states per head (l summed over each group's warps at
// lsum[g][4][8], its reference max at mseg[g][8]) merged into this thread's
// output of every head, oh[h] (thread `row` = TMEM lane of O^T = head
// dimension; the groups' O^T at columns ocols + g NC), and each head's
// base-2 max Mh and sum Lh.
template <int D>
__device__ __forceinline__ void tc8_seg_merge(const float *lsum, const float *mseg, float vsc, uint32_t ocols,
                                              float (&oh)[8], float (&Mh)[8], float (&Lh)[8])
{
    using C = Tc8Cfg<D>;
    constexpr int NWG = C::NWG;
    float lg[NWG][8];
#pragma unroll
    for (int g = 0; g < NWG; ++g)
#pragma unroll
        for (int h = 0; h < 8; ++h)
            lg[g][h] = lsum[g * 32 + h] + lsum[g * 32 + 8 + h] + lsum[g * 32 + 16 + h] + lsum[g * 32 + 24 + h];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        float M = -INFINITY;
#pragma unroll
        for (int g = 0; g < NWG; ++g)
            if (lg[g][h] > 0.f)
                M = fmaxf(M, mseg[g * 8 + h]);
        float L = 0.f;
#pragma unroll
        for (int g = 0; g < NWG; ++g)
            if (lg[g][h] > 0.f)
                L += ex2(mseg[g * 8 + h] - M) * lg[g][h];
        Mh[h] = M;
        Lh[h] = L;
        oh[h] = 0.f;
    }
    // each group's O^T (one TMEM load per group), weighted into oh
#pragma unroll 1
    for (int g = 0; g < NWG; ++g) {
        bool need = false;
        float f[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            f[h] = (lg[g][h] > 0.f && Lh[h] > 0.f) ? ex2(mseg[g * 8 + h] - Mh[h]) / Lh[h] * vsc : 0.f;
            need = need || f[h] != 0.f;
        }
        if (!need)   // the same for every thread: the values come from shared memory
            continue;
        float o[32];
        tmem_ld32(ocols + (uint32_t)(g * C::NC), o);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 8; ++h)
            if (f[h] != 0.f)
                oh[h] += f[h] * (o[h] + 0.0625f * o[8 + h] + 0.00390625f * o[16 + h]);
    }
#pragma unroll
    for (int h = 0; h < 8; ++h)
        Lh[h] *= pow2i(-(int)C::PEXP);   // P was taken times 2^PEXP
}

// Warms the lines (and their address translations) that the epilogue of
// segment cs will write, on 128 threads: its out rows, or its workspace
// rows and (m, l); called while the segment streams.
template <int D>
__device__ __forceinline__ void tc8_prefetch_dest(const GqaParams &gp, const Ctx &ctx, const Seg &cs, int slice,
                                                  int tid)
{
    const SplitParams &p = gp.s;
    const int vh = cs.h * gp.NG + slice;
    const long long bhv = (long long)cs.b * p.H * gp.NG + vh;
    const int gv = vh_count(gp, vh);
    const int len = (p.decomp == DECOMP_BALANCED) ? ctx.lenS[cs.b] : clamp_len(p, cs.b);
    bool complete;
    long long slot;
    tc_seg_dest(p, cs, bhv, len, complete, slot);
    const char *a;
    if (complete) {
        const int es = p.out_dtype == 0 ? 4 : 2;
        a = static_cast<const char *>(p.out) + vh_qrow0(gp, cs.b, vh) * D * es + tid * 128;
        if (tid * 128 < gv * D * es)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    } else {
        const long long r0 = slot * gp.G;
        a = reinterpret_cast<const char *>(p.ws_o + r0 * D) + tid * 128;
        if (tid * 128 < gv * D * 4)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
        if (tid == 0)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p.ws_ml + 2 * r0));
    }
}

// The rest of a segment's epilogue (tid 0..127 = head dimension): out/lse
// for a whole (b, h), or a workspace partial and, for the last piece to
// arrive, the merge of the pieces.  Its global-memory round trips (the
// arrival counter, the pieces' partials) overlap the next segments'
// streaming.  Returns false if a barrier wait expired.
template <int D>
__device__ __forceinline__ bool tc8_epilogue(const GqaParams &gp, const Ctx ctx, const Seg cs, int slice,
                                          const float (&oh)[8], const float (&Mh)[8], const float (&Lh)[8], int lane,
                                          int tid, uint32_t *misc, unsigned char *scratch, WarpBar &wb)
{
    using C = Tc8Cfg<D>;
    const SplitParams &p = gp.s;
    const int G = gp.G;
    const int vh = cs.h * gp.NG + slice;
    const long long bhv = (long long)cs.b * p.H * gp.NG + vh;
    const int gv = vh_count(gp, vh);
    const long long qrow0 = vh_qrow0(gp, cs.b, vh);
    const int len = (p.decomp == DECOMP_BALANCED) ? ctx.lenS[cs.b] : clamp_len(p, cs.b);
    bool complete;
    long long slot;
    tc_seg_dest(p, cs, bhv, len, complete, slot);
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        if (h < gv) {
            if (complete)
                store_out(p.out, (qrow0 + h) * D + tid, p.out_dtype, oh[h]);
            else
                p.ws_o[(slot * G + h) * D + tid] = oh[h];
        }
    }
    if (tid < gv) {
        float M = Mh[0], L = Lh[0];
#pragma unroll
        for (int h = 1; h < 8; ++h)
            if (tid == h) {
                M = Mh[h];
                L = Lh[h];
            }
        const bool nonempty = L > 0.f;
        if (complete) {
            if (p.lse)
                p.lse[qrow0 + tid] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
        } else {
            const long long r = slot * G + tid;
            p.ws_ml[2 * r] = nonempty ? M : -INFINITY;
            p.ws_ml[2 * r + 1] = L;
        }
    }
    if (!complete)
        return tc_arrive_merge<D, C::MERGE_PB, 128>(gp, ctx, cs, slice, gv, qrow0, bhv, len, lane, tid, misc, scratch, wb);
    return true;
}

template <int D>
__global__ void __launch_bounds__(Tc8Cfg<D>::THREADS, 1) gqa_tc8_kernel(const __grid_constant__ GqaParams gp)
{
    using C = Tc8Cfg<D>;
    constexpr int KST = C::KST, VST = C::VST;
    constexpr int NC = C::NC;
    const SplitParams &p = gp.s;
    const int slice = (int)(blockIdx.x % gp.NG);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int w = tid >> 5;
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);   // 1024-aligned
    const uint32_t ring = smem_addr(smem);
    const uint32_t qbuf = ring + C::RING_BYTES;   // two q-part buffers
    const uint32_t pbuf = qbuf + 2 * C::QP_BYTES;
    unsigned char *scratch = smem + C::RING_BYTES + 2 * C::QP_BYTES + C::NPB * C::PT_BYTES;
    float *xch = reinterpret_cast<float *>(scratch + C::SCR_BYTES);
    constexpr int NWG = C::NWG;
    int *flg = reinterpret_cast<int *>(xch);      // [NWG groups][2][4 warps]
    float *red = xch + NWG * 8;                   // [NWG groups][4 warps][8 heads]
    float *segx = red + NWG * 32;                 // [2 parities][l sums [NWG][4][8], m [NWG][8]]
    float *fhs = segx + 2 * C::SEGX;              // [2][8] score scales of the segment's heads
    uint64_t *bars = reinterpret_cast<uint64_t *>(scratch + C::SCR_BYTES + C::XCH_BYTES);
    uint32_t *misc = reinterpret_cast<uint32_t *>(bars + C::NBAR);   // [0] TMEM base, [1] flag
    long long *cumH = reinterpret_cast<long long *>(misc + 4);
    int *lenS = reinterpret_cast<int *>(cumH + p.B + 1);
    const uint32_t bar0 = smem_addr(bars);
    auto FULLK = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto EMPTYK = [&](int s) { return bar0 + 8u * (uint32_t)(KST + s); };
    auto FULLV = [&](int s) { return bar0 + 8u * (uint32_t)(2 * KST + s); };
    auto EMPTYV = [&](int s) { return bar0 + 8u * (uint32_t)(2 * KST + VST + s); };
    constexpr int NSB = C::NSB, NPB = C::NPB;
    constexpr int BS = 2 * KST + 2 * VST;
    auto SFULL = [&](int b) { return bar0 + 8u * (uint32_t)(BS + b); };
    auto SFREE = [&](int b) { return bar0 + 8u * (uint32_t)(BS + NSB + b); };
    constexpr int B0 = BS + 2 * NSB;
    // P of chunk j is handed over on p_full[j % NPB]: a group arrives there
    // again (chunk j + NPB) only after P.V of chunk j is done, which is after
    // the MMA warp saw the arrival, so no phase is missed
    auto PFULL = [&](int b) { return bar0 + 8u * (uint32_t)(B0 + b); };
    auto PVD = [&](int b) { return bar0 + 8u * (uint32_t)(B0 + NPB + b); };
    constexpr int B1 = B0 + 2 * NPB;
    const uint32_t FINS = bar0 + 8u * B1;
    const uint32_t FINP = bar0 + 8u * (B1 + 1);
    const uint32_t WG0BAR = bar0 + 8u * (B1 + 2);
    auto WGBAR = [&](int g) { return bar0 + 8u * (uint32_t)(B1 + 3 + g); };
    constexpr int B2 = B1 + 3 + NWG;   // then five pairs, by segment parity
    auto QFULL = [&](int i) { return bar0 + 8u * (uint32_t)(B2 + i); };
    auto SEGDONE = [&](int i) { return bar0 + 8u * (uint32_t)(B2 + 2 + i); };
    auto OFREE = [&](int i) { return bar0 + 8u * (uint32_t)(B2 + 4 + i); };
    static_assert(B2 + 6 == C::NBAR, "barrier count");

    if (tid == 0) {
        for (int s = 0; s < KST; ++s) {
            mbar_init(FULLK(s), 1);    // the producer's arrival plus the copy's bytes
            mbar_init(EMPTYK(s), 1);   // commit after S^T of the buffer's chunk
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(FULLV(s), 1);
            mbar_init(EMPTYV(s), 1);   // commit after P.V of the buffer's chunk
        }
        for (int b = 0; b < NSB; ++b) {
            mbar_init(SFULL(b), 1);   // commit after S^T
            mbar_init(SFREE(b), 4);   // the owning group's warps have read S^T
        }
        for (int b = 0; b < NPB; ++b) {
            mbar_init(PFULL(b), 4);   // the owning group's warps: Pp^T written, V's tail rows zeroed, O^T rescaled
            mbar_init(PVD(b), 1);     // commit after P.V of the buffer's chunk
        }
        mbar_init(FINS, 1);           // the MMA issuers' last commits
        mbar_init(FINP, 1);
        mbar_init(WG0BAR, 4);         // the epilogue warps (arrival and merge)
        for (int i = 0; i < 2; ++i) {
            // by parity of the non-empty segments: the epilogue warps have
            // written a q buffer and its score scales
            mbar_init(QFULL(i), 4);
            // by parity of all segments: every softmax warp has left its
            // (m, l) and its group's final O^T; the epilogue has read them
            mbar_init(SEGDONE(i), 4 * NWG);
            mbar_init(OFREE(i), 4);
        }
        for (int g = 0; g < NWG; ++g)
            mbar_init(WGBAR(g), 4);   // each group's vote and max exchange
        prefetch_tmap(&gp.tmk);
        prefetch_tmap(&gp.tmv);
    }
    // the q-part rows past 3 x 8 stay zero
    for (int i = tid; i < 2 * C::QP_BYTES / 16; i += C::THREADS)
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(qbuf + 16u * (uint32_t)i), "r"(0u) : "memory");
    if (w == C::S_WARP) {
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
    fence_proxy_async_smem();
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    bool dead = false;

    if (w == C::KPROD_WARP || w == C::VPROD_WARP) {
        // ------------------------------------------------------------ producers
        // one warp per ring (lane 0): K refills a buffer once S^T of its
        // chunk is done, V once P.V is
        if (lane == 0) {
            const bool isk = w == C::KPROD_WARP;
            const int nb = isk ? KST : VST;
            const uint32_t base = ring + (uint32_t)(isk ? 0 : KST * C::CHUNK_BYTES);
            TmaProducer<C, false> pr;
            pr.start(gp, ctx, 0, 1);
            int issued = 0;
#pragma unroll 1
            while (pr.have) {
                const int b = issued % nb;
                if (issued >= nb &&
                    !mbar_wait_bounded_sleep_thread(isk ? EMPTYK(b) : EMPTYV(b), (uint32_t)(((issued / nb) - 1) & 1), C::SLEEP_NS)) {
                    dead = true;
                    break;
                }
                tc8_issue<C>(pr, gp, ctx, isk ? &gp.tmk : &gp.tmv, base + (uint32_t)(b * C::CHUNK_BYTES),
                             isk ? FULLK(b) : FULLV(b));
                ++issued;
            }
            // no copy may be in flight when the CTA ends: the last fill of each buffer
            for (int i = max(0, issued - nb); i < issued; ++i)
                mbar_wait_bounded_sleep_thread(isk ? FULLK(i % nb) : FULLV(i % nb), (uint32_t)((i / nb) & 1), C::SLEEP_NS);
        }
        __syncwarp();
    } else if (w == C::S_WARP) {
        // ------------------------------------------------------------ S^T issuer
        // S^T of each chunk as soon as its K has landed, its S buffer is free
        // and (first chunk of a segment) the segment's q parts are written
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_f16(0, 0, 0, C::M, NC);   // K K-major, q parts K-major
            long long js = 0;
            int kq = 0;
            Seg ss;
            seg_first(p, ctx, ss);
#pragma unroll 1
            while (ss.valid && !dead) {
                const long long n = seg_chunks<C::CT>(ss);
                const int qp = kq & 1;   // this segment's q buffer (non-empty segments alternate)
                const uint32_t qb = qbuf + (uint32_t)(qp * C::QP_BYTES);
                if (n > 0) {
                    if (!mbar_wait_bounded_sleep_thread(QFULL(qp), (uint32_t)((kq >> 1) & 1), C::SLEEP_NS)) {
                        dead = true;
                        break;
                    }
                    ++kq;
                    tc_fence_after();
                }
#pragma unroll 1
                for (long long c = 0; c < n; ++c, ++js) {
                    const int st = (int)(js % KST), sb = (int)(js % NSB);
                    if (!mbar_wait_bounded_sleep_thread(FULLK(st), (uint32_t)((js / KST) & 1), C::SLEEP_NS) ||
                        (js >= NSB && !mbar_wait_bounded_sleep_thread(SFREE(sb), (uint32_t)(((js / NSB) - 1) & 1), C::SLEEP_NS))) {
                        dead = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kb = ring + (uint32_t)(st * C::CHUNK_BYTES);
#pragma unroll
                    for (int ks = 0; ks < D / 32; ++ks) {
                        // 32 E4M3 values = 32 bytes of each 128-byte row
                        const uint64_t a = smem_desc_sw128(kb + (uint32_t)(ks * 32), 16, 1024);
                        const uint64_t b = smem_desc_sw128(qb + (uint32_t)(ks * 32), 16, 1024);
                        tc_mma_f8_ss(tmem + (uint32_t)(sb * NC), a, b, ID_S, ks > 0 ? 1u : 0u);
                    }
                    tc_commit(SFULL(sb));
                    tc_commit(EMPTYK(st));
                }
                seg_next(p, ctx, ss);
            }
            // every MMA this thread issued has completed before TMEM is freed
            tc_commit(FINS);
            if (!mbar_wait_bounded_sleep_thread(FINS, 0, C::SLEEP_NS))
                dead = true;
        }
        __syncwarp();
    } else if (w == C::PV_WARP) {
        // ------------------------------------------------------------ P.V issuer
        if (lane == 0) {
            constexpr uint32_t ID_O = idesc_f16(0, 1, 0, D, NC);      // V^T MN-major, Pp^T K-major
            long long jp = 0, pp0 = 0;   // chunks, and pairs before the segment
            int ks_ = 0;                 // segments so far: their O^T sets alternate
            Seg sp;
            seg_first(p, ctx, sp);
#pragma unroll 1
            while (sp.valid && !dead) {
                const long long n = seg_chunks<C::CT>(sp);
                const uint32_t oset = (uint32_t)(C::TMEM_O + (ks_ & 1) * NWG * NC);
                // the set was read by the epilogue for segment ks_ - 2
                if (n > 0 && ks_ >= 2 &&
                    !mbar_wait_bounded_sleep_thread(OFREE(ks_ & 1), (uint32_t)(((ks_ >> 1) - 1) & 1), C::SLEEP_NS)) {
                    dead = true;
                    break;
                }
#pragma unroll 1
                for (long long c = 0; c < n; ++c, ++jp) {
                    if (!mbar_wait_bounded_sleep_thread(PFULL((int)(jp % NPB)), (uint32_t)((jp / NPB) & 1), C::SLEEP_NS) ||
                        !mbar_wait_bounded_sleep_thread(FULLV((int)(jp % VST)), (uint32_t)((jp / VST) & 1), C::SLEEP_NS)) {
                        dead = true;
                        break;
                    }
                    tc_fence_after();
                    // the pair's group; its first chunk of the segment overwrites O^T
                    const int g = (int)((pp0 + c / 2) % NWG);
                    const bool first = c < 2 * NWG && (c & 1) == 0;
                    const uint32_t vb = ring + (uint32_t)((KST + jp % VST) * C::CHUNK_BYTES);
                    const uint32_t pb = pbuf + (uint32_t)((jp % NPB) * C::PT_BYTES);
#pragma unroll
                    for (int ks = 0; ks < C::CT / 32; ++ks) {
                        // 32 tokens: four 8-row groups of V (1024 bytes apart),
                        // 32 bytes of each Pp^T row
                        const uint64_t a = smem_desc_sw128(vb + (uint32_t)(ks * 4096), 16, 1024);
                        const uint64_t b = smem_desc_sw128(pb + (uint32_t)(ks * 32), 16, 1024);
                        tc_mma_f8_ss(tmem + oset + (uint32_t)(g * NC), a, b, ID_O, (!first || ks > 0) ? 1u : 0u);
                    }
                    tc_commit(EMPTYV((int)(jp % VST)));
                    tc_commit(PVD((int)(jp % NPB)));
                }
                pp0 += (n + 1) / 2;
                ++ks_;
                seg_next(p, ctx, sp);
            }
            tc_commit(FINP);
            if (!mbar_wait_bounded_sleep_thread(FINP, 0, C::SLEEP_NS))
                dead = true;
        }
        __syncwarp();
    } else if (w >= C::EPI_WARP) {
        // ------------------------------------------------------------ epilogue
        // each segment's state (the softmax warps' (m, l), the groups' O^T)
        // merged, released, and written to out/lse or the workspace, with
        // the arrival and, for the last piece, the merge of the pieces
        const int etid = tid - 32 * C::EPI_WARP;
        const uint32_t etl = tmem + ((uint32_t)((w & 3) * 32) << 16);   // this warp's TMEM lanes
        WarpBar wb{WG0BAR, 0u, 0u};   // busy warps: no sleep between their syncs
        // the q parts of the non-empty segments, two ahead: the first two
        // now, each further one as soon as the segment two before it is done
        Seg qs;
        seg_first(p, ctx, qs);
        int kqp = 0;
        auto prep_next = [&]() {
            while (qs.valid && seg_chunks<C::CT>(qs) == 0)
                seg_next(p, ctx, qs);
            if (!qs.valid)
                return;
            tc8_prep_q<D>(gp, qs, slice, qbuf + (uint32_t)((kqp & 1) * C::QP_BYTES), fhs + (kqp & 1) * 8, etid);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(QFULL(kqp & 1));
            ++kqp;
            seg_next(p, ctx, qs);
        };
        prep_next();
        prep_next();
        int k = 0;
        Seg cs;
        seg_first(p, ctx, cs);
#pragma unroll 1
        while (cs.valid && !dead) {
            const long long n = seg_chunks<C::CT>(cs);
            const float vsc = __ldg(gp.v_scale + cs.b * p.H + cs.h);   // V's dequantisation scale
            tc8_prefetch_dest<D>(gp, ctx, cs, slice, etid);
            const float *sx = segx + (k & 1) * C::SEGX;
            if (!mbar_wait_bounded_sleep(SEGDONE(k & 1), (uint32_t)((k >> 1) & 1), C::SLEEP_NS)) {
                dead = true;
                break;
            }
            tc_fence_after();
            float oh[8], Mh[8], Lh[8];
            tc8_seg_merge<D>(sx, sx + NWG * 32, vsc, etl + (uint32_t)(C::TMEM_O + (k & 1) * NWG * NC), oh, Mh, Lh);
            // the (m, l) and the O^T set are free for segment k + 2
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(OFREE(k & 1));
            // this segment's q buffer is free (its S^T are done, its score
            // scales read): the next q parts into it
            if (n > 0)
                prep_next();
            if (!tc8_epilogue<D>(gp, ctx, cs, slice, oh, Mh, Lh, lane, etid, misc, scratch, wb)) {
                dead = true;
                break;
            }
            ++k;
            seg_next(p, ctx, cs);
        }
    } else {
        // ------------------------------------------------------------ softmax groups
        const int wg = w >> 2;             // softmax group
        const int wq = w & 3;              // warp within the group
        const int row = tid & 127;         // token of the chunk (S^T) = head dim (O^T) = TMEM lane
        const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16);
        WarpBar gb{WGBAR(wg), 0u, C::SLEEP_NS};
        long long nw = 0;   // chunks this group has handed to P.V
        long long j0 = 0;   // the CTA's chunk index of the segment's first chunk
        long long p0 = 0;   // pairs of chunks before the segment
        int k = 0;          // segments so far
        int kq = 0;         // non-empty segments so far
        Seg cs;
        seg_first(p, ctx, cs);
#pragma unroll 1
        while (cs.valid && !dead) {
            const long long n = seg_chunks<C::CT>(cs);
            const int vh = cs.h * gp.NG + slice;
            const int gv = vh_count(gp, vh);
            const long long qrow0 = vh_qrow0(gp, cs.b, vh);
            // this group's O^T in the segment's set (segments alternate)
            const uint32_t ocol = (uint32_t)(C::TMEM_O + ((k & 1) * NWG + wg) * NC);
            const int qp = kq & 1;   // the q buffer of a non-empty segment
            float m[8], l[8], fh[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                m[h] = -INFINITY;
                l[h] = 0.f;
            }
            if (n > 0) {
                if (!mbar_wait_bounded_sleep(QFULL(qp), (uint32_t)((kq >> 1) & 1), C::SLEEP_NS)) {
                    dead = true;
                    break;
                }
                ++kq;
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    fh[h] = fhs[qp * 8 + h];
            }
            bool had = false;
            long long jprev = 0;
            const long long npairs = (n + 1) / 2;
            // the segment's chunks in pairs (2i, 2i + 1), pair i to group
            // (pairs before the segment + i) % NWG; both chunks share one vote
#pragma unroll 1
            for (long long pi = (long long)(((wg - (int)(p0 % NWG)) % NWG + NWG) % NWG); pi < npairs; pi += NWG) {
                const long long c0 = 2 * pi;
                const bool two = c0 + 1 < n;
                const long long j = j0 + c0;
                const int b0 = (int)(j % NSB), b1 = (int)((j + 1) % NSB);
                if (!mbar_wait_bounded_sleep(SFULL(b0), (uint32_t)((j / NSB) & 1), C::SLEEP_NS) ||
                    (two && !mbar_wait_bounded_sleep(SFULL(b1), (uint32_t)(((j + 1) / NSB) & 1), C::SLEEP_NS))) {
                    dead = true;
                    break;
                }
                tc_fence_after();
                float sv0[32], sv1[32];
                tmem_ld32(tl + (uint32_t)(b0 * NC), sv0);
                if (two)
                    tmem_ld32(tl + (uint32_t)(b1 * NC), sv1);
                int t, ntok0, ntok1 = 0;
                chunk_coords<C::CT>(cs, c0, t, ntok0);
                if (two)
                    chunk_coords<C::CT>(cs, c0 + 1, t, ntok1);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(SFREE(b0));
                    if (two)
                        mbar_arrive(SFREE(b1));
                }
                // base-2 scores of this thread's token in each chunk; -inf
                // past the chunk's tokens (and for a missing second chunk)
                const bool valid0 = row < ntok0, valid1 = row < ntok1;
                float x0[8], x1[8];
                bool f = false;
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const float s0 = fmaf(0.00390625f, sv0[16 + h], fmaf(0.0625f, sv0[8 + h], sv0[h]));
                    const float s1 = fmaf(0.00390625f, sv1[16 + h], fmaf(0.0625f, sv1[8 + h], sv1[h]));
                    x0[h] = valid0 ? s0 * fh[h] : -INFINITY;
                    x1[h] = valid1 ? s1 * fh[h] : -INFINITY;
                    f = f || fmaxf(x0[h], x1[h]) > m[h] + C::TAU;
                }
                // the group's vote: does any head's max move?
                int *fl = flg + (wg * 2 + (int)(nw & 1)) * 4;
                const bool wf = __any_sync(FULL_MASK, f);
                if (lane == 0)
                    fl[wq] = wf ? 1 : 0;
                if (!gb.sync(lane)) {
                    dead = true;
                    break;
                }
                if (fl[0] | fl[1] | fl[2] | fl[3]) {
                    float mx[8];
#pragma unroll
                    for (int h = 0; h < 8; ++h)
                        mx[h] = fmaxf(x0[h], x1[h]);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                        for (int h = 0; h < 8; ++h)
                            mx[h] = fmaxf(mx[h], __shfl_xor_sync(FULL_MASK, mx[h], o));
                    float *rd = red + wg * 32;
                    if (lane == 0)
#pragma unroll
                        for (int h = 0; h < 8; ++h)
                            rd[wq * 8 + h] = mx[h];
                    if (!gb.sync(lane)) {
                        dead = true;
                        break;
                    }
                    float al[8];
                    bool grow = false;
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const float cm = fmaxf(fmaxf(rd[h], rd[8 + h]), fmaxf(rd[16 + h], rd[24 + h]));
                        const bool g = cm > m[h] + C::TAU;
                        al[h] = g ? ex2(m[h] - cm) : 1.f;   // 0 on the group's first pair
                        m[h] = g ? cm : m[h];
                        l[h] *= al[h];
                        grow = grow || g;
                    }
                    // the group's O^T columns of the heads that moved, once
                    // its previous P.V is done (every warp its 32 lanes)
                    if (had && grow) {
                        if (!mbar_wait_bounded_sleep(PVD((int)(jprev % NPB)), (uint32_t)((jprev / NPB) & 1), C::SLEEP_NS)) {
                            dead = true;
                            break;
                        }
                        tc_fence_after();
                        float o[32];
                        tmem_ld32(tl + ocol, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] *= al[e & 7];
                        tmem_st32(tl + ocol, o);
                        tmem_wait_st();
                    }
                }
                // the Pp^T buffers of the pair are free once P.V of chunk
                // j + 1 - NPB (or j - NPB) is done: P.V completes in order
                const long long jw = j + (two ? 1 : 0) - NPB;
                if (jw >= 0 && !mbar_wait_bounded_sleep(PVD((int)(jw % NPB)), (uint32_t)((jw / NPB) & 1), C::SLEEP_NS)) {
                    dead = true;
                    break;
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (q == 1 && !two)
                        break;
                    const long long jq = j + q;
                    const uint32_t pb = pbuf + (uint32_t)((jq % NPB) * C::PT_BYTES);
#pragma unroll
                    for (int hp = 0; hp < 4; ++hp) {
                        const float xa = q ? x1[2 * hp] : x0[2 * hp], xb = q ? x1[2 * hp + 1] : x0[2 * hp + 1];
                        const float y0 = ex2(xa - m[2 * hp] + C::PEXP);
                        const float y1 = ex2(xb - m[2 * hp + 1] + C::PEXP);
                        l[2 * hp] += y0;
                        l[2 * hp + 1] += y1;
                        uint32_t q0, q1, q2;
                        e4m3_parts2(y0, y1, q0, q1, q2);
                        st_u8(pb + sw128_byte(2 * hp, row), q0);
                        st_u8(pb + sw128_byte(2 * hp + 1, row), q0 >> 8);
                        st_u8(pb + sw128_byte(8 + 2 * hp, row), q1);
                        st_u8(pb + sw128_byte(8 + 2 * hp + 1, row), q1 >> 8);
                        st_u8(pb + sw128_byte(16 + 2 * hp, row), q2);
                        st_u8(pb + sw128_byte(16 + 2 * hp + 1, row), q2 >> 8);
                    }
                    // V's rows past the chunk's tokens may hold padding (NaN * 0 is
                    // NaN): zeroed once V's copy has landed (its buffer is not
                    // refilled before P.V of the chunk)
                    const int ntq = q ? ntok1 : ntok0;
                    if (ntq < C::CT &&
                        !mbar_wait_bounded_sleep(FULLV((int)(jq % VST)), (uint32_t)((jq / VST) & 1), C::SLEEP_NS)) {
                        dead = true;
                        break;
                    }
                    if (!(q ? valid1 : valid0)) {
                        const uint32_t va = ring + (uint32_t)((KST + jq % VST) * C::CHUNK_BYTES + row * 128);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(va + 16u * (uint32_t)i),
                                         "r"(0u)
                                         : "memory");
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(PFULL((int)(j % NPB)));
                    if (two)
                        mbar_arrive(PFULL((int)((j + 1) % NPB)));
                }
                ++nw;
                had = true;
                jprev = j + (two ? 1 : 0);
            }
            if (dead)
                break;
            if (had) {
                // the group's last P.V: its O^T is final
                if (!mbar_wait_bounded_sleep(PVD((int)(jprev % NPB)), (uint32_t)((jprev / NPB) & 1), C::SLEEP_NS)) {
                    dead = true;
                    break;
                }
                tc_fence_after();
            }
            j0 += n;
            p0 += (n + 1) / 2;

            // ---- segment end: each warp's l per head over its 32 tokens and
            // its group's m, for the epilogue warps (the buffer of segment
            // k - 2 once they have read it), which merge the groups' states
            // while the softmax groups go on ----
            if (k >= 2 && !mbar_wait_bounded_sleep(OFREE(k & 1), (uint32_t)(((k >> 1) - 1) & 1), C::SLEEP_NS)) {
                dead = true;
                break;
            }
            float *sx = segx + (k & 1) * C::SEGX;   // l sums [NWG][4][8], then m [NWG][8]
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                float v = had ? l[h] : 0.f;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    v += __shfl_xor_sync(FULL_MASK, v, o);
                if (lane == 0)
                    sx[(wg * 4 + wq) * 8 + h] = v;
                if (wq == 0 && lane == 0)
                    sx[NWG * 32 + wg * 8 + h] = had ? m[h] : -INFINITY;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(SEGDONE(k & 1));
            ++k;
            seg_next(p, ctx, cs);
        }
    }

    if (dead && lane == 0)
        atomicOr(p.status, STATUS_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (w == C::S_WARP)
        tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D> static cudaError_t launch_gqa_tc8_t(const GqaParams &gp, cudaStream_t s)
{
    using C = Tc8Cfg<D>;
    const size_t smem = C::smem_bytes(gp.s.decomp, gp.s.B);
    auto kern = gqa_tc8_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kern<<<gp.s.grid, C::THREADS, smem, s>>>(gp);
    return cudaGetLastError();
}

}  // namespace fd
