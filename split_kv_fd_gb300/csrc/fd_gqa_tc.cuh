// fd_gqa_tc.cuh -- grouped-query decode for large groups (MQA and GQA with
// many query heads per K/V head, "从第一性原理推导 Flash Attention" §8) on
// the fifth-generation tensor cores: tcgen05.mma with accumulators in tensor
// memory (TMEM).
//
// Per (b, K/V head) and chunk of CT = 64 tokens the work is two dense
// products over all the K/V head's query heads at once (up to 128, the MMA's
// M; more are served in slices by adjacent CTAs):
//     S [128 x CT] = Q [128 x d] . K_chunk^T     (Q and K in shared memory)
//     O [128 x d] += P [128 x CT] . V_chunk      (P in TMEM, V in shared memory)
// so every K/V byte enters shared memory once per CTA, whatever the number
// of query heads (the mma.sync kernel of fd_gqa.cuh stages a chunk once per
// 16 heads).  The online softmax between the two products runs in fp32
// registers, one thread per query head (TMEM lane = MMA row = head):
//  - S is read with tcgen05.ld; the scores past the chunk's tokens are
//    masked; P = 2^(s - m_ref) is split into a 16-bit high part and the
//    16-bit remainder, both written back into the chunk's S columns of TMEM
//    (tcgen05.st), and the two products P_hi V + P_lo V keep P.V close to
//    fp32 accuracy with 16-bit operands.
//  - The rescale of the block-wise update ("FlashDecoding 数学推导" §2.4.1:
//    acc and l times exp(m_old - m_new) when the max grows) is done lazily:
//    the reference max m_ref moves only when a chunk's max exceeds it by
//    more than TAU (in base 2), and only then are the head's O row in TMEM
//    and l rescaled.  In between, P may reach 2^TAU, which fp32 and the
//    16-bit high part hold exactly enough; the quotient o = acc / l is the
//    same.
//
// Warp roles (384 threads, one CTA per SM):
//  - warps 0-3 and 4-7: two softmax warpgroups taking the chunks in turn
//    (chunk j of the CTA goes to group j % 2), each with its own O
//    accumulator and (m_ref, l) per head; at a segment end both merge the
//    two states ("FlashDecoding 数学推导" §2.4.2), each for half of the
//    columns, and write the result;
//  - warps 8 and 9: the K and V producers (lane 0 each), chunks by
//    tensor-map TMA into rings of their own: a K buffer is refilled once S
//    of its chunk is done, a V buffer once P.V is;
//  - warp 10: allocates TMEM; its lane 0 issues S = Q K^T, up to NSB chunks
//    ahead of P.V;
//  - warp 11: lane 0 issues P.V and frees the chunk's V and S buffers by
//    its commits.
// TMEM holds NSB S/P buffers (chunk j in buffer j % NSB) and the two O
// accumulators.  The copies take ~3 us to land at full load, so the two
// rings take the shared memory left beside Q (160 KB at d = 128); after
// the CTA's last segment the idle rings stage the pieces of a last
// arriver's merge.  Every hand-off is an mbarrier (the MMA warps' through
// tcgen05.commit), and every wait is bounded: on expiry a role records
// FD_ERR_DEVICE_TIMEOUT, stops, drains what it issued, and the CTA frees its
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
    // K and V have rings of their own: a K buffer is free once S of its
    // chunk is done, a V buffer only once P.V is; together they take the
    // shared memory left beside Q, the merge scratch and the barriers
    static constexpr int RING_BUFS = ((D == 128 ? 160 : 192) * 1024) / CHUNK_BYTES;
    static constexpr int KST = RING_BUFS / 3 > 4 ? RING_BUFS / 3 : 4;
    static constexpr int VST = RING_BUFS - KST;
    static constexpr int RING_BYTES = RING_BUFS * CHUNK_BYTES;   // K buffers, then V buffers
    static constexpr int QPLANE = M * 128;         // one 64-element plane of Q
    static constexpr int Q_BYTES = LINES * QPLANE;
    static constexpr int MERGE_PB = 64;            // pieces per batch of the last arriver's merge
    static constexpr int SCR_BYTES = MERGE_PB * 8 + 2 * MAXG * 4;   // their slots, then M and L per head
    static constexpr int XCH_BYTES = 2 * 2 * M * 2 * 4;   // both groups' (m_ref, l) per head, two segments
    // warps 0-7: the two softmax groups; 8, 9: the K and V producers; 10:
    // the S issuer (it allocates TMEM); 11: the P.V issuer
    static constexpr int WG_THREADS = 128, KPROD_WARP = 8, VPROD_WARP = 9, S_WARP = 10, PV_WARP = 11;
    static constexpr int THREADS = 384;
    // TMEM: NSB S/P buffers of CT columns (chunk j in buffer j % NSB), then
    // the two groups' O accumulators
    static constexpr int NSB = 4;
    static constexpr int TMEM_O = NSB * CT;
    static constexpr uint32_t TMEM_COLS = 512;
    // mbarriers: full/empty of the K and V buffers, s_full[NSB],
    // s_free[NSB], p_full[NSB], o_full[2][2], q_full, fin (2), seg (both
    // groups), the two of a merge staged in the ring
    static constexpr int NBAR = 2 * RING_BUFS + 3 * NSB + 10;
    static constexpr float TAU = 8.f;              // lazy-rescale threshold (base 2)
    // every wait suspends the waiting thread in hardware (woken when the
    // phase completes) rather than polling
    static constexpr uint32_t SLEEP_NS = 100000;
    static_assert(D == 64 || D == 128, "head dim 64 or 128");
    static_assert(CT == 64, "an S buffer holds P_hi and P_lo in its 64 columns");
    static_assert(TMEM_O + 2 * D <= (int)TMEM_COLS, "TMEM columns");
    static_assert(RING_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0 && CHUNK_BYTES % 1024 == 0, "1024-byte atoms");
    static_assert(VST >= 4, "ring depth");

    static size_t smem_bytes(int decomp, int B)
    {
        size_t s = 1024 + RING_BYTES + Q_BYTES + SCR_BYTES + XCH_BYTES + NBAR * 8 + 16;
        if (decomp == DECOMP_BALANCED)
            s += (size_t)(B + 1) * 8 + (size_t)B * 4;
        return s;
    }
};

// A barrier of `warps` warps on an mbarrier initialised with that count,
// with the bounded wait: a warp whose partner gave up does not hang here.
// `phase` is the parity of the next completion; the warps run the same
// sequence of syncs.  Returns false on expiry.
struct WarpBar {
    uint32_t bar;
    uint32_t phase;
    uint32_t hint_ns = 0;   // > 0: the waiting warps are suspended in hardware meanwhile
    __device__ __forceinline__ bool sync(int lane)
    {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar);
        const bool ok = hint_ns ? mbar_wait_bounded_sleep(bar, phase, hint_ns) : mbar_wait_bounded(bar, phase);
        phase ^= 1u;
        return ok;
    }
};

// Eight consecutive outputs from index idx (a multiple of 8) in out_dtype,
// 16-byte stores for 16-bit outputs.
__device__ __forceinline__ void store_out8(void *out, long long idx, int out_dtype, const float *x)
{
    if (out_dtype == 0) {
        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(out) + idx);
        o[0] = make_float4(x[0], x[1], x[2], x[3]);
        o[1] = make_float4(x[4], x[5], x[6], x[7]);
        return;
    }
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = out_dtype == 1 ? Mma<__half>::pack(x[2 * i], x[2 * i + 1])
                              : Mma<__nv_bfloat16>::pack(x[2 * i], x[2 * i + 1]);
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + idx) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Four consecutive outputs from index idx (a multiple of 4).
__device__ __forceinline__ void store_out4(void *out, long long idx, int out_dtype, float4 x)
{
    if (out_dtype == 0) {
        *reinterpret_cast<float4 *>(static_cast<float *>(out) + idx) = x;
        return;
    }
    const uint32_t a = out_dtype == 1 ? Mma<__half>::pack(x.x, x.y) : Mma<__nv_bfloat16>::pack(x.x, x.y);
    const uint32_t b = out_dtype == 1 ? Mma<__half>::pack(x.z, x.w) : Mma<__nv_bfloat16>::pack(x.z, x.w);
    *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + idx) = make_uint2(a, b);
}

// One batch of the last arriver's merge, on NT threads: the m/l/o merge
// ("FlashDecoding 数学推导" §2.4.2) of the n <= MERGE_PB workspace partials
// whose slots are in ss[0..n-1], for each of the Gv query rows.  Each thread
// takes four elements of a head at a time and the pieces' partials and
// (m, l) together, many loads in flight, with a running max and sum for its
// head: acc and L scaled by exp2(M_old - M_new) when the max grows, so one
// round trip to memory serves the batch (the merge sits on the CTA's
// critical path).  The result goes to out/lse, or, when `into` >= 0, back
// into the workspace slot `into` as a normalised partial (o, m, l) that a
// later batch merges (each head's (m, l) through sM, sL, written once every
// thread has read the slot's).  Returns false if a barrier wait expired.
template <int D, int NT>
__device__ __forceinline__ bool tc_merge_batch(const SplitParams &p, int G, int Gv, long long qrow0, const long long *ss,
                                               int n, long long into, float *sM, float *sL, int tid, WarpBar &wb)
{
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml);   // (m, l) per workspace row
    constexpr int GB = 2, PB = 8;   // groups of 4 elements, pieces per round
    const int ngrp = Gv * D / 4;
    for (int base = 0; base < ngrp; base += NT * GB) {
        float4 acc[GB];
        int gg[GB], dd[GB];
        float Mr[GB], Lr[GB];
#pragma unroll
        for (int e = 0; e < GB; ++e) {
            acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            const int grp = min(base + e * NT + tid, ngrp - 1);
            gg[e] = grp * 4 / D;
            dd[e] = grp * 4 % D;
            Mr[e] = -INFINITY;
            Lr[e] = 0.f;
        }
        for (int i0 = 0; i0 < n; i0 += PB) {
            float4 v[GB][PB];
            float2 w[GB][PB];
#pragma unroll
            for (int u = 0; u < PB; ++u) {
                const long long s0 = ss[min(i0 + u, n - 1)] * G;
#pragma unroll
                for (int e = 0; e < GB; ++e) {
                    v[e][u] = __ldcg(reinterpret_cast<const float4 *>(p.ws_o + (s0 + gg[e]) * D + dd[e]));
                    w[e][u] = __ldcg(ml + s0 + gg[e]);
                }
            }
#pragma unroll
            for (int u = 0; u < PB; ++u) {
#pragma unroll
                for (int e = 0; e < GB; ++e) {
                    if (i0 + u < n && w[e][u].y > 0.f) {
                        const float mn = fmaxf(Mr[e], w[e][u].x);
                        const float a = ex2(Mr[e] - mn);   // 0 for the first piece
                        const float b = ex2(w[e][u].x - mn) * w[e][u].y;
                        acc[e].x = fmaf(b, v[e][u].x, acc[e].x * a);
                        acc[e].y = fmaf(b, v[e][u].y, acc[e].y * a);
                        acc[e].z = fmaf(b, v[e][u].z, acc[e].z * a);
                        acc[e].w = fmaf(b, v[e][u].w, acc[e].w * a);
                        Lr[e] = fmaf(Lr[e], a, b);
                        Mr[e] = mn;
                    }
                }
            }
        }
#pragma unroll
        for (int e = 0; e < GB; ++e) {
            const int grp = base + e * NT + tid;
            const bool mine = grp < ngrp;
            const int g = gg[e], dim = dd[e];
            const float L = Lr[e];
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const float4 o = make_float4(acc[e].x * inv, acc[e].y * inv, acc[e].z * inv, acc[e].w * inv);
            if (mine) {
                if (into >= 0) {
                    // this thread alone reads and writes these four elements
                    *reinterpret_cast<float4 *>(p.ws_o + (into * G + g) * D + dim) = o;
                } else {
                    const long long qrow = qrow0 + g;
                    store_out4(p.out, qrow * D + dim, p.out_dtype, o);
                    if (dim == 0 && p.lse)
                        p.lse[qrow] = L > 0.f ? (Mr[e] + log2f(L)) * LN2_F : -INFINITY;
                }
            }
            if (mine && dim == 0 && into >= 0) {
                sM[g] = Mr[e];
                sL[g] = L;
            }
        }
    }
    if (into < 0)
        return true;
    // every read of the batch's (m, l) is done before the slot's are replaced
    if (!wb.sync(tid & 31))
        return false;
    if (tid < Gv) {
        const long long r = into * G + tid;
        p.ws_ml[2 * r] = sL[tid] > 0.f ? sM[tid] : -INFINITY;
        p.ws_ml[2 * r + 1] = sL[tid];
    }
    return wb.sync(tid & 31);
}

// Shared memory a merge may stage the pieces in: the CTA's K/V ring once its
// last segment is done (no copy in flight, no MMA reading it), with two
// mbarriers of its own.  p == nullptr: none (the merge reads the pieces
// from global memory).
struct MergeStage {
    unsigned char *p = nullptr;
    uint32_t a = 0;       // shared-space address of p
    int bytes = 0;
    uint32_t mb[2] = {0u, 0u};
};

// The same batch as tc_merge_batch, with the pieces' o rows staged in
// shared memory: first the weights, one thread per head (each piece's
// 2^(m_i - M) l_i / L, M the max over the pieces that hold tokens, L the sum
// of 2^(m_i - M) l_i: the merge of "FlashDecoding 数学推导" §2.4.2 with the
// normalisation folded in), while bulk copies bring a block of HB heads of
// every piece into one of two buffers; then each block is summed while the
// next one lands.  Every load of the batch is in flight at once, where the
// loop of tc_merge_batch waits for a round trip per 256 groups of 4
// elements.  The results differ from tc_merge_batch's only in the order of
// the fp32 operations.  `mph` holds the two mbarriers' phases.  Returns
// false if a wait expired.
template <int D, int NT>
__device__ __forceinline__ bool tc_merge_staged(const SplitParams &p, int G, int Gv, long long qrow0,
                                                const long long *ss, int n, long long into, int tid, WarpBar &wb,
                                                const MergeStage &st, uint32_t &mph)
{
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml);
    float2 *wml = reinterpret_cast<float2 *>(st.p);   // [n][Gv]: (m, l), then (weight, -)
    const int wml_bytes = (n * Gv * 8 + 127) & ~127;
    const int buf_bytes = ((st.bytes - wml_bytes) / 2) & ~127;
    const int head_bytes = n * D * 4;                  // one head of every piece
    int hb = min(Gv, buf_bytes / head_bytes);
    const int nblk = (Gv + hb - 1) / hb;
    hb = (Gv + nblk - 1) / nblk;                       // blocks of even size
    auto issue = [&](int blk) {
        const int h0 = blk * hb, nh = min(hb, Gv - h0);
        const uint32_t bytes = (uint32_t)(nh * D * 4), bar = st.mb[blk & 1];
        const uint32_t dst = st.a + (uint32_t)(wml_bytes + (blk & 1) * buf_bytes);
        mbar_arrive_expect_tx(bar, bytes * (uint32_t)n);
        for (int i = 0; i < n; ++i)
            bulk_g2s(dst + (uint32_t)i * bytes, p.ws_o + (ss[i] * G + h0) * D, bytes, bar);
    };
    if (tid == 0) {
        fence_proxy_async_global();   // the pieces' writers' stores, acquired by the arrival
        issue(0);
        if (nblk > 1)
            issue(1);
    }
    if (tid < Gv) {
        float M = -INFINITY;
        for (int i0 = 0; i0 < n; i0 += 8) {
            float2 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[u] = __ldcg(ml + ss[min(i0 + u, n - 1)] * G + tid);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (i0 + u < n) {
                    if (v[u].y > 0.f)
                        M = fmaxf(M, v[u].x);
                    wml[(i0 + u) * Gv + tid] = v[u];
                }
        }
        float L = 0.f;
        for (int i = 0; i < n; ++i) {
            const float2 v = wml[i * Gv + tid];
            const float wgt = v.y > 0.f ? ex2(v.x - M) * v.y : 0.f;
            wml[i * Gv + tid].x = wgt;
            L += wgt;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int i = 0; i < n; ++i)
            wml[i * Gv + tid].x *= inv;
        if (into >= 0) {
            // this thread alone read the slot's (m, l) for this head
            const long long r = into * G + tid;
            p.ws_ml[2 * r] = L > 0.f ? M : -INFINITY;
            p.ws_ml[2 * r + 1] = L;
        } else if (p.lse) {
            p.lse[qrow0 + tid] = L > 0.f ? (M + log2f(L)) * LN2_F : -INFINITY;
        }
    }
    if (!wb.sync(tid & 31))
        return false;
#pragma unroll 1
    for (int blk = 0; blk < nblk; ++blk) {
        const int h0 = blk * hb, nh = min(hb, Gv - h0);
        const uint32_t par = (mph >> (blk & 1)) & 1u;
        mph ^= 1u << (blk & 1);
        if (!mbar_wait_bounded(st.mb[blk & 1], par))
            return false;
        const float *buf = reinterpret_cast<const float *>(st.p + wml_bytes + (blk & 1) * buf_bytes);
        const int ngrp = nh * D / 4;
        for (int grp = tid; grp < ngrp; grp += NT) {
            const int g = h0 + grp * 4 / D, dim = grp * 4 % D;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int i = 0; i < n; ++i) {
                const float wgt = wml[i * Gv + g].x;
                const float4 v = *reinterpret_cast<const float4 *>(buf + i * nh * D + grp * 4);
                acc.x = fmaf(wgt, v.x, acc.x);
                acc.y = fmaf(wgt, v.y, acc.y);
                acc.z = fmaf(wgt, v.z, acc.z);
                acc.w = fmaf(wgt, v.w, acc.w);
            }
            if (into >= 0)
                *reinterpret_cast<float4 *>(p.ws_o + (into * G + g) * D + dim) = acc;
            else
                store_out4(p.out, (qrow0 + g) * D + dim, p.out_dtype, acc);
        }
        if (blk + 2 < nblk) {
            // every thread is done with the buffer before it is refilled
            if (!wb.sync(tid & 31))
                return false;
            if (tid == 0)
                issue(blk + 2);
        }
    }
    if (into < 0)
        return true;
    // the next batch copies this slot back in through the async proxy, which
    // reads L2: the stores must have reached it (a barrier orders them only
    // within the CTA)
    __threadfence();
    fence_proxy_async_global();
    return wb.sync(tid & 31);
}

// Stage 2 of a (b, virtual head) by the last piece to arrive, on the NT
// threads of barrier `wb`: the merge of its `target` workspace partials, in
// batches of at most MERGE_PB pieces; each batch but the last leaves its
// result in its last piece's slot, which starts the next batch.  Staged in
// shared memory when `st` gives the idle ring.  Returns false if a barrier
// wait expired.
template <int D, int MERGE_PB, int NT>
__device__ __forceinline__ bool tc_merge_pieces(const GqaParams &gp, const Ctx &ctx, long long bhv, int slice,
                                                int G, int Gv, long long qrow0, unsigned target, int gf,
                                                long long off, int tid, unsigned char *scr, WarpBar &wb,
                                                const MergeStage &st)
{
    const SplitParams &p = gp.s;
    long long *ss = reinterpret_cast<long long *>(scr);            // [MERGE_PB] slots
    float *sM = reinterpret_cast<float *>(scr + MERGE_PB * 8);      // [G]
    float *sL = sM + G;                                              // [G]
    const int n = (int)target;
    int first = 0;
    uint32_t mph = 0;   // the staging mbarriers' phases (a CTA stages one merge, at its last segment)
    for (;;) {
        const int cnt = min(n - first, MERGE_PB);
        for (int i = tid; i < cnt; i += NT)
            ss[i] = vh_slot(gp, ctx, bhv, (unsigned)(first + i), gf, off, slice);
        if (!wb.sync(tid & 31))
            return false;
        const bool last = first + cnt == n;
        // staged when the ring is idle and a block of one head of every
        // piece fits beside the weights
        const int wml_bytes = (cnt * Gv * 8 + 127) & ~127;
        const bool staged = st.p != nullptr && ((st.bytes - wml_bytes) / 2 & ~127) >= cnt * D * 4;
        const long long into = last ? -1 : ss[cnt - 1];
        if (!(staged ? tc_merge_staged<D, NT>(p, G, Gv, qrow0, ss, cnt, into, tid, wb, st, mph)
                     : tc_merge_batch<D, NT>(p, G, Gv, qrow0, ss, cnt, into, sM, sL, tid, wb)))
            return false;
        if (last)
            return true;
        first += cnt - 1;   // the batch's result, in its last slot, opens the next batch
    }
}

// Where a segment's result goes: `complete` when the segment is its whole
// (b, virtual head), then to out/lse; else to workspace slot `slot`.
__device__ __forceinline__ void tc_seg_dest(const SplitParams &p, const Seg &cs, long long bhv, int len, bool &complete,
                                            long long &slot)
{
    if (p.decomp == DECOMP_SPLITS) {
        complete = (p.P == 1);
        slot = bhv * p.P + cs.p;
    } else {
        complete = seg_whole(p, cs, len);
        slot = 2LL * blockIdx.x + (cs.k == 0 ? 0 : 1);
    }
}

// After a segment's partial is in the workspace, on the NT threads that
// wrote it (barrier `wb`): the arrival on the (b, virtual head)'s counter
// and, for the last piece to arrive, the merge of the pieces.  Returns
// false if a barrier wait expired.
template <int D, int MERGE_PB, int NT>
__device__ __forceinline__ bool tc_arrive_merge(const GqaParams &gp, const Ctx ctx, const Seg cs, int slice, int gv,
                                             long long qrow0, long long bhv, int len, int lane, int tid,
                                             uint32_t *misc, unsigned char *scratch, WarpBar &wb,
                                             const MergeStage st = MergeStage())
{
    const SplitParams &p = gp.s;
    unsigned target;
    int gf = 0;
    long long off = 0;
    if (p.decomp == DECOMP_SPLITS) {
        target = (unsigned)p.P;
    } else {
        off = bal_offset(p, ctx, cs.b, cs.h, len);
        gf = bal_owner(off, ctx.T, ctx.Geff);
        const int gl = bal_owner(off + bal_span(p, len) - 1, ctx.T, ctx.Geff);
        target = (unsigned)(gl - gf + 1);
    }
    // the barrier orders every thread's partial before thread 0's fence and
    // arrival
    if (!wb.sync(lane))
        return false;
    if (tid == 0) {
        __threadfence();
        const unsigned old = atomicInc(p.ws_cnt + bhv, target - 1);
        misc[1] = (old == target - 1) ? 1u : 0u;
    }
    if (!wb.sync(lane))
        return false;
    if (misc[1]) {
        __threadfence();
        if (!tc_merge_pieces<D, MERGE_PB, NT>(gp, ctx, bhv, slice, gp.G, gv, qrow0, target, gf, off, tid, scratch,
                                              wb, st))
            return false;
    }
    return wb.sync(lane);   // the flag and the scratch are reused
}

// Segment end on both softmax groups (256 threads, barrier `sb`): merges
// the two groups' (m_ref, l, O) per head ("FlashDecoding 数学推导" §2.4.2),
// group g reading and writing columns [g d/2, (g+1) d/2) of both O
// accumulators, then writes out/lse for a whole (b, h), or a workspace
// partial and, for the last piece to arrive, runs the merge of the pieces
// on all 256 threads.  (m0, l0) and (m1, l1) are the groups' states
// (l = 0: the group had no chunk).  Returns false if a barrier wait expired.
template <typename C, int D>
__device__ __forceinline__ bool tc_segment_end(const GqaParams &gp, const Ctx ctx, const Seg cs, int slice, int G, int gv,
                                            long long qrow0, long long bhv, float m0, float l0, float m1, float l1,
                                            int wg, int row, int lane, int tid, uint32_t tl, uint32_t *misc,
                                            unsigned char *scratch, WarpBar &sb, const MergeStage &st)
{
    const SplitParams &p = gp.s;
    const bool live = row < gv;
    const float M = fmaxf(l0 > 0.f ? m0 : -INFINITY, l1 > 0.f ? m1 : -INFINITY);
    const float a0 = l0 > 0.f ? ex2(m0 - M) : 0.f;
    const float a1 = l1 > 0.f ? ex2(m1 - M) : 0.f;
    const float L = a0 * l0 + a1 * l1;
    const bool nonempty = L > 0.f;
    const float f0 = nonempty ? a0 / L : 0.f, f1 = nonempty ? a1 / L : 0.f;
    // warps w and w + 4 hold the same rows: the same votes
    const bool need0 = __any_sync(FULL_MASK, l0 > 0.f), need1 = __any_sync(FULL_MASK, l1 > 0.f);
    const int len = (p.decomp == DECOMP_BALANCED) ? ctx.lenS[cs.b] : clamp_len(p, cs.b);
    bool complete;
    long long slot;
    tc_seg_dest(p, cs, bhv, len, complete, slot);
    const long long qrow = qrow0 + row;
    const long long r = slot * G + row;
    constexpr int QH = D / 32;   // 16-column slices per group
#pragma unroll 1
    for (int q = wg * QH; q < (wg + 1) * QH; ++q) {
        float o0[16], o1[16];
        if (need0)
            tmem_ld16(tl + (uint32_t)(C::TMEM_O + 16 * q), o0);
        if (need1)
            tmem_ld16(tl + (uint32_t)(C::TMEM_O + D + 16 * q), o1);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e)
            o0[e] = (need0 ? f0 * o0[e] : 0.f) + (need1 ? f1 * o1[e] : 0.f);
        if (live) {
            if (complete) {
                store_out8(p.out, qrow * D + 16 * q, p.out_dtype, o0);
                store_out8(p.out, qrow * D + 16 * q + 8, p.out_dtype, o0 + 8);
            } else {
                float4 *dst = reinterpret_cast<float4 *>(p.ws_o + r * D + 16 * q);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_float4(o0[4 * e], o0[4 * e + 1], o0[4 * e + 2], o0[4 * e + 3]);
            }
        }
    }
    tc_fence_before();
    if (live && wg == 0) {
        if (complete) {
            if (p.lse)
                p.lse[qrow] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
        } else {
            p.ws_ml[2 * r] = nonempty ? M : -INFINITY;
            p.ws_ml[2 * r + 1] = L;
        }
    }
    if (!complete) {
        fence_proxy_async_global();   // the last arriver may bulk-copy this partial
        return tc_arrive_merge<D, C::MERGE_PB, 2 * C::WG_THREADS>(gp, ctx, cs, slice, gv, qrow0, bhv, len, lane, tid,
                                                                  misc, scratch, sb, st);
    }
    return true;
}

template <typename T, int D>
__global__ void __launch_bounds__(TcCfg<T, D>::THREADS, 1) gqa_tc_kernel(const __grid_constant__ GqaParams gp)
{
    using C = TcCfg<T, D>;
    constexpr int KST = C::KST, VST = C::VST;
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
    unsigned char *scratch = smem + C::RING_BYTES + C::Q_BYTES;   // the last arriver's merge
    float *xch = reinterpret_cast<float *>(scratch + C::SCR_BYTES);   // [2][2][M][2]
    uint64_t *bars = reinterpret_cast<uint64_t *>(scratch + C::SCR_BYTES + C::XCH_BYTES);
    uint32_t *misc = reinterpret_cast<uint32_t *>(bars + C::NBAR);   // [0] TMEM base, [1] flag
    long long *cumH = reinterpret_cast<long long *>(misc + 4);
    int *lenS = reinterpret_cast<int *>(cumH + p.B + 1);
    const uint32_t bar0 = smem_addr(bars);
    auto FULLK = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto EMPTYK = [&](int s) { return bar0 + 8u * (uint32_t)(KST + s); };
    auto FULLV = [&](int s) { return bar0 + 8u * (uint32_t)(2 * KST + s); };
    auto EMPTYV = [&](int s) { return bar0 + 8u * (uint32_t)(2 * KST + VST + s); };
    constexpr int NSB = C::NSB;
    constexpr int BS = 2 * (KST + VST);
    auto SFULL = [&](int b) { return bar0 + 8u * (uint32_t)(BS + b); };
    auto SFREE = [&](int b) { return bar0 + 8u * (uint32_t)(BS + NSB + b); };
    // P of chunk j is handed over on p_full[j % NSB]: a group arrives there
    // again (chunk j + NSB) only after S of that chunk, which waits for P.V
    // of chunk j, so no phase is missed
    auto PFULL = [&](int b) { return bar0 + 8u * (uint32_t)(BS + 2 * NSB + b); };
    constexpr int B0 = BS + 3 * NSB;
    // P.V of chunk j (group j % 2) commits o_full[j % 2][(j / 2) % 2]: a
    // barrier per group and parity of the group's chunk count, so that one
    // phase there is chunk j and the one before it chunk j - 4, which S of
    // chunk j waited for (P.V completes in order); a wait for a chunk's P.V
    // is then never two phases away from the barrier's
    auto OFULL = [&](int g, int b) { return bar0 + 8u * (uint32_t)(B0 + 2 * g + b); };
    auto OFULL_J = [&](long long j) { return OFULL((int)(j & 1), (int)((j >> 1) & 1)); };
    const uint32_t QFULL = bar0 + 8u * (B0 + 4);
    const uint32_t FINS = bar0 + 8u * (B0 + 5);
    const uint32_t FINP = bar0 + 8u * (B0 + 6);
    const uint32_t SEGBAR = bar0 + 8u * (B0 + 7);
    const uint32_t MRG0 = bar0 + 8u * (B0 + 8), MRG1 = bar0 + 8u * (B0 + 9);
    static_assert(B0 + 10 == C::NBAR, "barrier count");

    if (tid == 0) {
        for (int s = 0; s < KST; ++s) {
            mbar_init(FULLK(s), 1);   // the producer's arrival plus the copy's bytes
            mbar_init(EMPTYK(s), 1);  // commit after S of the buffer's chunk
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(FULLV(s), 1);
            mbar_init(EMPTYV(s), 1);  // commit after P.V of the buffer's chunk
        }
        for (int b = 0; b < NSB; ++b) {
            mbar_init(SFULL(b), 1);   // commit after S
            mbar_init(SFREE(b), 1);   // commit after P.V of the buffer's chunk
            mbar_init(PFULL(b), 4);   // the owning group's warps: P in TMEM, V's tail rows zeroed
        }
        for (int g = 0; g < 4; ++g)
            mbar_init(OFULL(g >> 1, g & 1), 1);   // commit after P.V of the group's chunk
        mbar_init(QFULL, 8);          // both groups have written their halves of Q
        mbar_init(FINS, 1);           // the MMA issuers' last commits
        mbar_init(FINP, 1);
        mbar_init(SEGBAR, 8);         // both groups: segment ends, arrivals, merges
        mbar_init(MRG0, 1);           // a merge's bulk copies into the idle ring
        mbar_init(MRG1, 1);
        prefetch_tmap(&gp.tmk);
        prefetch_tmap(&gp.tmv);
    }
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
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    bool dead = false;

    if (w == C::KPROD_WARP || w == C::VPROD_WARP) {
        // ------------------------------------------------------------ producers
        // one warp per ring (lane 0): K refills a buffer once S of its chunk
        // is done, V once P.V is
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
                if (issued >= nb && !mbar_wait_bounded_sleep_thread(isk ? EMPTYK(b) : EMPTYV(b),
                                                                    (uint32_t)(((issued / nb) - 1) & 1), C::SLEEP_NS)) {
                    dead = true;
                    break;
                }
                // one box of the chunk's CT rows, every plane; rows past the
                // block's end read as zeros
                const int y = pr.t, blk = pr.s.b * p.H + pr.s.h;
                const uint32_t bar = isk ? FULLK(b) : FULLV(b);
                mbar_arrive_expect_tx(bar, C::CHUNK_BYTES);
                tma_load_4d(base + (uint32_t)(b * C::CHUNK_BYTES), isk ? &gp.tmk : &gp.tmv, 0, y, blk, 0, bar);
                pr.c += pr.stride;
                pr.locate(gp, ctx);
                ++issued;
            }
            // no copy may be in flight when the CTA ends: the last fill of each buffer
            for (int i = max(0, issued - nb); i < issued; ++i)
                mbar_wait_bounded_sleep_thread(isk ? FULLK(i % nb) : FULLV(i % nb), (uint32_t)((i / nb) & 1),
                                               C::SLEEP_NS);
        }
        __syncwarp();
    } else if (w == C::S_WARP) {
        // ------------------------------------------------------------ S issuer
        // S of each chunk as soon as its K has landed and its S/P buffer is
        // free (P.V of chunk j - NSB done); the first S of a segment once
        // both groups have written the segment's Q
        if (lane == 0) {
            constexpr int BF = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
            constexpr uint32_t ID_S = idesc_f16(BF, 0, 0, C::M, C::CT);   // Q K-major, K K-major
            long long j = 0;   // chunks of this CTA so far
            int k = 0;         // non-empty segments so far
            Seg cs;
            seg_first(p, ctx, cs);
#pragma unroll 1
            while (cs.valid && !dead) {
                const long long n = seg_chunks<C::CT>(cs);
                if (n > 0) {
                    if (!mbar_wait_bounded_sleep_thread(QFULL, (uint32_t)(k & 1), C::SLEEP_NS)) {
                        dead = true;
                        break;
                    }
                    ++k;
                    tc_fence_after();
                }
#pragma unroll 1
                for (long long c = 0; c < n; ++c, ++j) {
                    const int st = (int)(j % KST), sb = (int)(j % NSB);
                    if (!mbar_wait_bounded_sleep_thread(FULLK(st), (uint32_t)((j / KST) & 1), C::SLEEP_NS) ||
                        (j >= NSB &&
                         !mbar_wait_bounded_sleep_thread(SFREE(sb), (uint32_t)(((j / NSB) - 1) & 1), C::SLEEP_NS))) {
                        dead = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kb = ring + (uint32_t)(st * C::CHUNK_BYTES);
                    const uint32_t ds = tmem + (uint32_t)(sb * C::CT);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        // 16 elements = 32 bytes of each 128-byte row of plane ks / 4
                        const uint32_t col = (uint32_t)((ks & 3) * 32);
                        const uint64_t a = smem_desc_sw128(qbuf + (uint32_t)((ks >> 2) * C::QPLANE) + col, 16, 1024);
                        const uint64_t b = smem_desc_sw128(kb + (uint32_t)((ks >> 2) * C::PLANE) + col, 16, 1024);
                        tc_mma_ss(ds, a, b, ID_S, ks > 0 ? 1u : 0u);
                    }
                    tc_commit(SFULL(sb));
                    tc_commit(EMPTYK(st));
                }
                seg_next(p, ctx, cs);
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
            constexpr int BF = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
            constexpr uint32_t ID_O = idesc_f16(BF, 0, 1, C::M, D);       // P (TMEM) K-major, V MN-major
            long long j = 0;
            Seg cs;
            seg_first(p, ctx, cs);
#pragma unroll 1
            while (cs.valid && !dead) {
                const long long n = seg_chunks<C::CT>(cs);
#pragma unroll 1
                for (long long c = 0; c < n; ++c, ++j) {
                    const int sb = (int)(j % NSB), vs = (int)(j % VST);
                    if (!mbar_wait_bounded_sleep_thread(PFULL(sb), (uint32_t)((j / NSB) & 1), C::SLEEP_NS) ||
                        !mbar_wait_bounded_sleep_thread(FULLV(vs), (uint32_t)((j / VST) & 1), C::SLEEP_NS)) {
                        dead = true;
                        break;
                    }
                    tc_fence_after();
                    const int g = (int)(j & 1);
                    const uint32_t vb = ring + (uint32_t)((KST + vs) * C::CHUNK_BYTES);
                    const uint32_t pa = tmem + (uint32_t)(sb * C::CT);
#pragma unroll
                    for (int ks = 0; ks < C::CT / 16; ++ks) {
#pragma unroll
                        for (int hl = 0; hl < 2; ++hl) {
                            // P_hi in columns 0-31 of the buffer, P_lo in 32-63; 8 columns per k-step
                            const uint64_t b = smem_desc_sw128(vb + (uint32_t)(ks * 2048), (uint32_t)C::PLANE, 1024);
                            tc_mma_ts(tmem + (uint32_t)(C::TMEM_O + g * D), pa + (uint32_t)(hl * 32 + ks * 8), b,
                                      ID_O, (c >= 2 || ks > 0 || hl > 0) ? 1u : 0u);
                        }
                    }
                    tc_commit(OFULL_J(j));
                    tc_commit(EMPTYV(vs));
                    tc_commit(SFREE(sb));
                }
                seg_next(p, ctx, cs);
            }
            tc_commit(FINP);
            if (!mbar_wait_bounded_sleep_thread(FINP, 0, C::SLEEP_NS))
                dead = true;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax groups
        const int wg = w >> 2;             // softmax group
        const int row = tid & 127;         // query head within the slice = TMEM lane
        const uint32_t tl = tmem + ((uint32_t)((w & 3) * 32) << 16);
        const uint32_t ocol = (uint32_t)(C::TMEM_O + wg * D);
        WarpBar sb{SEGBAR, 0u, C::SLEEP_NS};
        long long jl = -1;  // the CTA's chunk index of the last chunk this group handed to P.V
        long long j0 = 0;   // the CTA's chunk index of the segment's first chunk
        int k = 0;          // segments so far
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
                // the query rows into the Q buffer (K-major, 128-byte swizzle),
                // group g the 16-byte pieces 4g..4g+3 of each 128-byte line;
                // zero for heads past the slice's
                const uint4 *qs = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.q) +
                                                                  (qrow0 + row) * D);
#pragma unroll
                for (int pl = 0; pl < C::LINES; ++pl)
#pragma unroll
                    for (int c16 = 4 * wg; c16 < 4 * wg + 4; ++c16) {
                        const uint4 v = live ? __ldg(qs + pl * 8 + c16) : make_uint4(0, 0, 0, 0);
                        const uint32_t a =
                            qbuf + (uint32_t)(pl * C::QPLANE + row * 128 + ((c16 ^ (row & 7)) << 4));
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y),
                                     "r"(v.z), "r"(v.w)
                                     : "memory");
                    }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(QFULL);
            }
            bool had = false;
#pragma unroll 1
            for (long long c = (long long)(wg ^ (int)(j0 & 1)); c < n; c += 2) {
                const long long j = j0 + c;
                const int b = (int)(j % NSB);
                if (!mbar_wait_bounded_sleep(SFULL(b), (uint32_t)((j / NSB) & 1), C::SLEEP_NS)) {
                    dead = true;
                    break;
                }
                tc_fence_after();
                // the head's 64 scores in one TMEM round trip
                float s0[32], s1[32];
                tmem_ld32(tl + (uint32_t)(b * C::CT), s0);
                tmem_ld32(tl + (uint32_t)(b * C::CT + 32), s1);
                int t, ntok;
                chunk_coords<C::CT>(cs, c, t, ntok);
                tmem_wait_ld();
                auto S = [&](int i) -> float & { return i < 32 ? s0[i] : s1[i - 32]; };
                // the tokens past the chunk's (a partial chunk only) become -inf
                if (ntok < C::CT) {
#pragma unroll
                    for (int i = 0; i < C::CT; ++i)
                        S(i) = i < ntok ? S(i) : -INFINITY;
                }
                // the chunk's max of the base-2 scores s * sc: the max of the
                // raw scores times sc (sc > 0, the normal case), else the min
                const float sc = p.scale_log2;
                float mc;
                if (sc > 0.f) {
                    float x = S(0);
#pragma unroll
                    for (int i = 1; i < C::CT; ++i)
                        x = fmaxf(x, S(i));
                    mc = x * sc;
                } else {
                    mc = -INFINITY;
#pragma unroll
                    for (int i = 0; i < C::CT; ++i)
                        mc = fmaxf(mc, S(i) * sc);
                }
                // lazy rescale: the reference max moves only when the
                // chunk's max exceeds it by more than TAU
                const bool grow = mc > m_ref + C::TAU;
                float a = 1.f;
                if (grow) {
                    a = ex2(m_ref - mc);   // 0 on the group's first chunk
                    l *= a;
                    m_ref = mc;
                }
                // the O rows in TMEM: the tcgen05 loads and stores are
                // warp-wide, so the whole warp runs them when any of its
                // heads grew (a = 1 for the others)
                if (had && __any_sync(FULL_MASK, grow)) {
                    // once the group's previous P.V (chunk jl = j - 2) is done
                    if (!mbar_wait_bounded_sleep(OFULL_J(jl), (uint32_t)((jl >> 2) & 1), C::SLEEP_NS)) {
                        dead = true;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int q = 0; q < D / 16; ++q) {
                        float o[16];
                        tmem_ld16(tl + ocol + (uint32_t)(16 * q), o);
                        tmem_wait_ld();
                        uint32_t u[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            u[e] = __float_as_uint(o[e] * a);
                        tmem_st16u(tl + ocol + (uint32_t)(16 * q), u);
                    }
                }
                // P = 2^(s sc - m_ref): the 16-bit high part and its
                // remainder, packed pairs, into the chunk's S columns (P_hi
                // in 0-31, P_lo in 32-63; the scores are all in registers).
                // Heads past the slice's (zero q rows) get P = 1 and are
                // never written out.
                const uint64_t sc2 = pack2(sc, sc), nm2 = pack2(-m_ref, -m_ref), one2 = pack2(1.f, 1.f);
                uint64_t ls2 = pack2(0.f, 0.f);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t ph[16], plo[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int tk = 32 * h + 2 * i;
                        float x0, x1;
                        unpack2(fma2(pack2(S(tk), S(tk + 1)), sc2, nm2), x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        ls2 = fma2(pack2(p0, p1), one2, ls2);
                        ph[i] = Mma<T>::pack(p0, p1);
                        const float2 u = Mma<T>::unpack(ph[i]);
                        plo[i] = Mma<T>::pack(p0 - u.x, p1 - u.y);
                    }
                    tmem_st16u(tl + (uint32_t)(b * C::CT + 16 * h), ph);
                    tmem_st16u(tl + (uint32_t)(b * C::CT + 32 + 16 * h), plo);
                }
                float lsa, lsb;
                unpack2(ls2, lsa, lsb);
                l += lsa + lsb;
                // V's rows past the chunk's tokens may hold padding (NaN * 0 is
                // NaN): zeroed once V's copy has landed (its buffer is not
                // refilled before P.V of the chunk)
                if (ntok < C::CT) {
                    if (!mbar_wait_bounded_sleep(FULLV((int)(j % VST)), (uint32_t)((j / VST) & 1), C::SLEEP_NS)) {
                        dead = true;
                        break;
                    }
                    const uint32_t vb = ring + (uint32_t)((KST + j % VST) * C::CHUNK_BYTES);
                    const int pieces = (C::CT - ntok) * C::LINES * 8;
                    for (int x = row; x < pieces; x += 128) {
                        const int r = ntok + x / (C::LINES * 8);
                        const int rem = x % (C::LINES * 8);
                        const uint32_t va = vb + (uint32_t)((rem >> 3) * C::PLANE + r * 128 + (rem & 7) * 16);
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(va), "r"(0u) : "memory");
                    }
                    fence_proxy_async_smem();
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(PFULL((int)(j % NSB)));
                jl = j;
                had = true;
            }
            if (dead)
                break;
            if (had) {
                // the group's last P.V: its O is final
                if (!mbar_wait_bounded_sleep(OFULL_J(jl), (uint32_t)((jl >> 2) & 1), C::SLEEP_NS)) {
                    dead = true;
                    break;
                }
                tc_fence_after();
            }
            j0 += n;

            // ---- segment end: the groups swap their (m_ref, l) and share the work ----
            float *xk = xch + (k & 1) * 2 * C::M * 2;   // [group][row][2]
            xk[(wg * C::M + row) * 2] = had ? m_ref : -INFINITY;
            xk[(wg * C::M + row) * 2 + 1] = had ? l : 0.f;
            ++k;
            tc_fence_before();
            if (!sb.sync(lane)) {
                dead = true;
                break;
            }
            tc_fence_after();
            Seg nx = cs;
            seg_next(p, ctx, nx);
            // after the CTA's last segment no copy is in flight into the
            // ring and no MMA reads it: a merge may stage its pieces there
            MergeStage st;
            if (!nx.valid) {
                st.p = smem;
                st.a = ring;
                st.bytes = C::RING_BYTES;
                st.mb[0] = MRG0;
                st.mb[1] = MRG1;
            }
            // its syncs spin: both groups are in it, nothing else to run
            WarpBar se{SEGBAR, sb.phase, 0u};
            const bool ok = tc_segment_end<C, D>(gp, ctx, cs, slice, G, gv, qrow0, bhv, xk[2 * row], xk[2 * row + 1],
                                                 xk[(C::M + row) * 2], xk[(C::M + row) * 2 + 1], wg, row, lane, tid,
                                                 tl, misc, scratch, se, st);
            sb.phase = se.phase;
            if (!ok) {
                dead = true;
                break;
            }
            cs = nx;
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
