// fd_gqa.cuh -- grouped-query split-KV decode (MQA / GQA): Hq = G * Hkv query
// heads, each group of G consecutive query heads sharing one K/V head
// ("从第一性原理推导 Flash Attention" §8).  Per (b, kv head) the work is a
// small dense contraction: scores S[G x T] = Q[G x d] K[T x d]^T and
// O[G x d] = P[G x T] V[T x d] over each chunk of T tokens, so it runs on the
// tensor cores (mma.sync m16n8k16, fp32 accumulate; G padded to 16 rows).
// The K/V bytes are still read exactly once and the path stays HBM-bound:
// at G = 8 it needs ~8 flop per byte, far below the tensor rate.
//
// Same decomposition, rings and merges as the split kernel (fd_split.cuh);
// what differs:
//  - K/V chunks arrive through tensor-map TMA (cp.async.bulk.tensor.3d) with
//    the 128-byte swizzle, so ldmatrix reads them without bank conflicts.
//    A row of d elements is viewed as d/64 lines of 128 bytes: the map is
//    [64 elements, d/64 lines, rows], box [64, d/64, CT rows].
//  - P is split into a bf16/f16 high part and the low part of its residual
//    (P = P_hi + P_lo), so P.V keeps close to fp32 accuracy with 16-bit MMA
//    operands.
//  - A stage's rows past the chunk's last valid token are zeroed in shared
//    memory before P.V (those rows may hold padding).
#pragma once

#include <cuda.h>

#include "fd_split.cuh"

namespace fd {

#ifndef FD_GQA_STAGES
#define FD_GQA_STAGES 2
#endif

template <typename T, int D> struct GqaCfg {
    static constexpr int ROW = D * 2;              // bytes per token row (16-bit types)
    static constexpr int LINES = D / 64;           // 128-byte lines per row
    static constexpr int WARPS = 8;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int GW = 2;                   // warps sharing one ring
    static constexpr int GROUPS = WARPS / GW;
    static constexpr int STAGES = FD_GQA_STAGES;
    static constexpr int WT = 16;                  // tokens per warp per chunk (one PV k-step)
    static constexpr int CT = GW * WT;             // tokens per chunk
    static constexpr int CHUNK_BYTES = CT * ROW;   // one of K or V
    static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;
    static constexpr int RING_BYTES = GROUPS * STAGES * STAGE_BYTES;
    static constexpr int BAR_BYTES = GROUPS * STAGES * 2 * 8;
    static constexpr int KSTEPS = D / 16;          // k-steps of Q.K^T
    static constexpr int NT = D / 8;               // 8-wide n-tiles of O
    static constexpr int MAXG = 16;
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(CHUNK_BYTES % 1024 == 0, "stages stay 1024-byte aligned for the swizzle");

    // dynamic shared memory: 1024 of alignment slack, ring, barriers, the
    // warps' (o, m, l) for the merge, a flag, and the balanced prefix sums
    static size_t smem_bytes(int decomp, int B, int G)
    {
        size_t s = 1024 + RING_BYTES + BAR_BYTES + (size_t)WARPS * G * (D + 2) * 4 + 16;
        if (decomp == DECOMP_BALANCED)
            s += (size_t)(B + 1) * 8 + (size_t)B * 4;
        return s;
    }
};

struct GqaParams {  // CUtensorMap carries its own 64-byte (or wider) alignment
    CUtensorMap tmk;   // K as [64, d/64, B*Hkv*N] 16-bit elements, 128B swizzle
    CUtensorMap tmv;   // V likewise
    SplitParams s;     // s.H = Hkv; s.q is [B, Hkv*G, d]; outputs [B, Hkv*G, ...]
    int G;             // query heads per K/V head, 2..16
};

cudaError_t launch_gqa(int dtype, int d, const GqaParams &gp, cudaStream_t s);

// Byte offset of 16-byte chunk c of row r in a stage laid out by the 128B
// swizzle (stage base 1024-aligned): line = r*LINES + c/8, and the chunk's
// position within its 128-byte line is (c % 8) XOR (line % 8).
template <int LINES>
__device__ __forceinline__ uint32_t swz(int r, int c)
{
    const int line = r * LINES + (c >> 3);
    return (uint32_t)(line * 128 + (((c & 7) ^ (line & 7)) << 4));
}

// The group's producer: the chunk walk of the split kernel's producer, with
// each chunk fetched as one K box and one V box through the tensor maps.
template <typename C> struct TmaProducer {
    Seg s;
    long long base;
    long long c;
    bool have;
    int t, ntok;

    __device__ __forceinline__ void locate(const SplitParams &p, const Ctx &ctx)
    {
        while (s.valid && c >= base + seg_chunks<C::CT>(s)) {
            base += seg_chunks<C::CT>(s);
            seg_next(p, ctx, s);
        }
        have = s.valid;
        if (have)
            chunk_coords<C::CT>(s, c - base, t, ntok);
    }

    __device__ __forceinline__ void start(const SplitParams &p, const Ctx &ctx, int first)
    {
        seg_first(p, ctx, s);
        base = 0;
        c = first;
        locate(p, ctx);
    }

    // Copies the full CT-row boxes (rows past the tensor end read as zeros).
    __device__ __forceinline__ bool issue(const GqaParams &gp, const Ctx &ctx, uint32_t kdst,
                                          uint32_t bar, int lane)
    {
        if (!have)
            return false;
        if (lane == 0) {
            const SplitParams &p = gp.s;
            const int row = (int)(((long long)s.b * p.H + s.h) * p.N + t);
            mbar_arrive_expect_tx(bar, 2 * C::CHUNK_BYTES);
            tma_load_3d(kdst, &gp.tmk, 0, 0, row, bar);
            tma_load_3d(kdst + C::CHUNK_BYTES, &gp.tmv, 0, 0, row, bar);
        }
        c += C::GROUPS;
        locate(gp.s, ctx);
        return true;
    }
};

// Per-warp softmax state for the 16 (padded) query rows: this thread holds
// rows r0 = lane/4 and r1 = r0 + 8, and columns 2*(lane%4)+{0,1} of every
// 8-wide tile of O (the mma accumulator layout).
template <typename C> struct GqaState {
    float o[C::NT][4];
    float m0, m1;   // running max (base 2)
    float l0, l1;   // this thread's share of the running sums
};

// One warp's WT rows of a chunk (rows row0 .. row0+WT-1 of the stage, the
// first `nvalid` of them real tokens): S = Q K^T on the tensor cores, the
// block-wise online-softmax update in fp32, then O += (P_hi + P_lo) V.
template <typename T, typename C>
__device__ __forceinline__ void gqa_chunk(uint32_t kstage, uint32_t vstage, int row0, int nvalid,
                                          const uint32_t (*qa)[4], float scale_log2, int lane,
                                          GqaState<C> &st)
{
    // scores for 2 tiles of 8 tokens; even and odd k-steps accumulate
    // separately so the dependent MMA chains are half as long
    float sc[2][4], sx[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
        sx[j][0] = sx[j][1] = sx[j][2] = sx[j][3] = 0.f;
    }
#pragma unroll
    for (int s2 = 0; s2 < C::KSTEPS / 2; ++s2) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int tok = row0 + 8 * j + (lane & 7);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kstage + swz<C::LINES>(tok, 4 * s2 + (lane >> 3)), b0, b1, b2, b3);
            Mma<T>::run(sc[j], qa[2 * s2], b0, b1);
            Mma<T>::run(sx[j], qa[2 * s2 + 1], b2, b3);
        }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            sc[j][e] += sx[j][e];
    }
    // base-2 scale and the mask of rows past the last valid token
    const int colb = 2 * (lane & 3);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int tok = 8 * j + colb + (e & 1);
            sc[j][e] = tok < nvalid ? sc[j][e] * scale_log2 : -INFINITY;
        }
    }
    // row maxima over the chunk's 16 tokens (a row lives in a quad of lanes)
    float x0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
    float x1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(FULL_MASK, x0, o));
        x1 = fmaxf(x1, __shfl_xor_sync(FULL_MASK, x1, o));
    }
    const float mn0 = fmaxf(st.m0, x0), mn1 = fmaxf(st.m1, x1);  // finite: nvalid >= 1
    const float a0 = ex2(st.m0 - mn0), a1 = ex2(st.m1 - mn1);
    st.m0 = mn0;
    st.m1 = mn1;
    float pr[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        pr[j][0] = ex2(sc[j][0] - mn0);
        pr[j][1] = ex2(sc[j][1] - mn0);
        pr[j][2] = ex2(sc[j][2] - mn1);
        pr[j][3] = ex2(sc[j][3] - mn1);
    }
    st.l0 = st.l0 * a0 + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
    st.l1 = st.l1 * a1 + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
#pragma unroll
    for (int n = 0; n < C::NT; ++n) {
        st.o[n][0] *= a0;
        st.o[n][1] *= a0;
        st.o[n][2] *= a1;
        st.o[n][3] *= a1;
    }
    // P as the A operand of P.V: P = P_hi + P_lo, both 16-bit
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = i >> 1, e = (i & 1) * 2;  // (tile j, rows r0 | r1)
        ph[i] = Mma<T>::pack(pr[j][e], pr[j][e + 1]);
        const float2 h = Mma<T>::unpack(ph[i]);
        pl[i] = Mma<T>::pack(pr[j][e] - h.x, pr[j][e + 1] - h.y);
    }
    // O += P V over this warp's 16 rows: V tiles through ldmatrix.trans
    const int vtok = row0 + 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
    for (int n2 = 0; n2 < C::NT / 2; ++n2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vstage + swz<C::LINES>(vtok, 2 * n2 + (lane >> 4)), b0, b1, b2, b3);
        Mma<T>::run(st.o[2 * n2], ph, b0, b1);
        Mma<T>::run(st.o[2 * n2], pl, b0, b1);
        Mma<T>::run(st.o[2 * n2 + 1], ph, b2, b3);
        Mma<T>::run(st.o[2 * n2 + 1], pl, b2, b3);
    }
}

}  // namespace fd
