// fd_gqa.cuh -- grouped-query split-KV decode (MQA / GQA): Hq = G * Hkv query
// heads, each group of G consecutive query heads sharing one K/V head
// ("从第一性原理推导 Flash Attention" §8).  Per (b, kv head) the work is a
// small dense contraction: scores S[G x T] = Q[G x d] K[T x d]^T and
// O[G x d] = P[G x T] V[T x d] over each chunk of T tokens, so it runs on the
// tensor cores (mma.sync m16n8k16, fp32 accumulate).  The K/V bytes are still
// read exactly once and the path stays HBM-bound: at G = 8 it needs ~8 flop
// per byte, far below the tensor rate.
//
// The products are taken transposed, S^T = K Q^T and O^T = V^T P^T, so the
// 16-row side of the MMA is tokens (for S^T) or head dimensions (for O^T)
// and the 8-column side holds the query heads: a group of up to 8 heads (16
// with two column tiles) wastes no MMA rows, and the accumulators are half
// the size of the untransposed form's.  The score accumulator of S^T holds
// P^T in the layout of an 8x8 transpose of the B operand of O^T = V^T P^T,
// so P reaches the second product through movmatrix, without shared memory.
//
// Same decomposition, rings and merges as the split kernel (fd_split.cuh);
// what differs:
//  - K/V chunks arrive through tensor-map TMA (cp.async.bulk.tensor.4d) with
//    the 128-byte swizzle.  A stage holds a chunk as d/64 planes, plane j
//    being elements [64j, 64j + 64) of the CT rows, 128 bytes per row: the
//    map views K (or V) as [64 elements, N rows, B*Hkv blocks, d/64 planes]
//    (strides d*2, N*d*2 and 128 bytes) and one box [64, CT, 1, d/64]
//    fetches a whole chunk of one (b, K/V head) block.  With
//    128-byte rows the swizzle gives any 8 consecutive rows of a column 8
//    different bank groups, so the ldmatrix reads are free of bank conflicts
//    (rows of d = 128 kept whole, 256 bytes, would repeat the pattern every 4
//    rows: 2-way conflicts).  One copy per chunk and operand keeps the TMA
//    instruction count low: issuing a copy costs the issuing thread ~70 ns.
//  - P is split into a bf16/f16 high part and the low part of its residual
//    (P = P_hi + P_lo), so P.V keeps close to fp32 accuracy with 16-bit MMA
//    operands.
//  - A stage's rows outside the chunk's valid tokens are zeroed in shared
//    memory before P.V (those rows may hold padding or other rows).
//  - More than 16 query heads per K/V head (8 at d = 256; MQA) are served
//    in slices run by adjacent CTAs over the same token range (see Slices).
#pragma once

#include <cuda.h>

#include "fd_split.cuh"

namespace fd {

#ifndef FD_GQA_STAGES
#define FD_GQA_STAGES 2
#endif
#ifndef FD_GQA_GW
#define FD_GQA_GW 2
#endif

// Head dim 256: 4 warps, so that two stages per group still make 128 KB in
// flight (a 32-token chunk of K and V is then 32 KB), and G <= 8 (one column
// tile: O^T alone takes 64 accumulator registers per thread).
//
// F8: K/V stored as E4M3 bytes (d = 64, 128 or 256).  The ring stages the
// bytes as they are in memory (rows of d bytes; at d = 64 and 256 fetched by
// 1-D bulk copies, a page at a time when a chunk spans two 16-token pages),
// three stages per group at d = 64 and 256, four at d = 128; each warp
// converts its 16 rows to f16, exactly, into its own area (the 16-row layout
// of stage_row with P16, K then V), frees the stage and runs the f16
// products there.  A slice then holds at most 8 query heads, so that the
// ring, the areas and the merge buffer fit in one CTA's shared memory (at
// d = 256: 96 KB of ring, 64 KB of areas, 33 KB of merge buffer).
template <typename T, int D, bool F8 = false> struct GqaCfg {
    static constexpr bool F8K = F8;
    // F8 at d = 128: K's fragments come straight from the staged bytes (a
    // 128-byte swizzled tensor-map box per chunk) and only V goes through
    // the f16 area; at d = 64 both do
    static constexpr bool F8REG = F8 && D == 128;
    static constexpr int ROW = F8 ? D : D * 2;     // bytes per token row in the ring
    static constexpr int LINES = D / 64;           // 128-byte lines per 16-bit row
    static constexpr int WARPS = D == 256 ? 4 : 8;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int GW = FD_GQA_GW;           // warps sharing one ring
    static constexpr int GROUPS = WARPS / GW;
    static constexpr int STAGES = F8 ? (D == 128 ? 4 : 3) : FD_GQA_STAGES;
    static constexpr int WT = 16;                  // tokens per warp per chunk (one PV k-step)
    static constexpr int CT = GW * WT;             // tokens per chunk
    static constexpr int CHUNK_BYTES = CT * ROW;   // one of K or V
    static constexpr int PLANE = CT * 128;         // one 64-element plane of a 16-bit chunk
    static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;
    static constexpr int RING_BYTES = GROUPS * STAGES * STAGE_BYTES;
    // per warp: 16 f16 rows of V (F8REG), or of K and V
    static constexpr int AREA_BYTES = F8 ? (D == 128 ? 1 : 2) * LINES * 16 * 128 : 0;
    static constexpr int AREAS = WARPS * AREA_BYTES;
    static constexpr int BAR_BYTES = GROUPS * STAGES * 2 * 8;
    static constexpr int KSTEPS = D / 16;          // k-steps of S^T = K Q^T
    static constexpr int MT = D / 16;              // 16-row tiles of O^T
    static constexpr int MAXG = (D == 256 || F8) ? 8 : 16;   // F8: the areas leave room for 8 heads' merge
    static_assert(D == 64 || D == 128 || D == 256, "head dim");
    static_assert(PLANE % 1024 == 0, "planes stay 1024-byte aligned for the swizzle");
    static_assert(RING_BYTES % 1024 == 0 && AREA_BYTES % 1024 == 0, "areas stay 1024-byte aligned");

    // dynamic shared memory: 1024 of alignment slack, ring, the F8 areas,
    // barriers, the warps' (o, m, l) for the merge, a flag, and the balanced
    // prefix sums
    static size_t smem_bytes(int decomp, int B, int G)
    {
        size_t s = 1024 + RING_BYTES + AREAS + BAR_BYTES + (size_t)WARPS * G * (D + 2) * 4 + 16;
        if (decomp == DECOMP_BALANCED)
            s += (size_t)(B + 1) * 8 + (size_t)B * 4;
        return s;
    }
};

struct GqaParams {  // CUtensorMap carries its own 64-byte (or wider) alignment
    CUtensorMap tmk;   // K as [64, n, blocks, d/64] 16-bit elements (n = N token rows of each of
                       // blocks = B*Hkv (b, K/V head) blocks; paged: n = page_size, blocks =
                       // num_pages*Hkv), boxes [64, CT, 1, d/64], 128B swizzle.  E4M3 at d = 128:
                       // [128 bytes, n, blocks], boxes [128, CT, 1].  Every coordinate stays
                       // below 2^31 whatever the cache's total row count.
    CUtensorMap tmv;   // V likewise
    SplitParams s;     // s.H = Hkv; s.q is [B, Hkv*Gq, d]; outputs [B, Hkv*Gq, ...]
    int G;             // query heads per slice (the last slice of a K/V head may have fewer), <= MAXG
    int NG;            // slices per K/V head: ceil(Gq / MAXG); s.grid is a multiple of NG
    int Gq;            // query heads per K/V head
    int pages16;       // paged with 16-token pages: boxes [64, 16, d/64], the P16 stage layout
    const float *k_scale;   // F8: [B*Hkv] dequantisation scales of K and V
    const float *v_scale;
};

cudaError_t launch_gqa(int dtype, int d, const GqaParams &gp, cudaStream_t s);
cudaError_t launch_gqa_bf16(int d, const GqaParams &gp, cudaStream_t s);
cudaError_t launch_gqa_f8(int d, const GqaParams &gp, cudaStream_t s);   // E4M3 K/V, f16 products
cudaError_t launch_gqa_tc(int dtype, int d, const GqaParams &gp, cudaStream_t s);   // tcgen05, large groups
cudaError_t launch_gqa_tc8(int d, const GqaParams &gp, cudaStream_t s);   // tcgen05 FP8 products, E4M3 K/V

// Byte offset of 16-byte column c of row r in a stage of 64-element planes
// written by the 128B swizzle (stage base 1024-aligned): plane c/8, and
// within the plane's 128-byte row r, position (c % 8) XOR (r % 8).
template <int PLANE>
__device__ __forceinline__ uint32_t swz(int r, int c)
{
    return (uint32_t)((c >> 3) * PLANE + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Stage layouts.  The default one is d/64 planes of CT rows (one box per
// chunk and operand).  With 16-token pages (P16) each 16-row half of the
// stage is its own block of d/64 planes of 16 rows, so one box per page and
// operand fills a half; a warp's 16 rows are one half either way, and every
// plane starts on a 1024-byte boundary, so the swizzle phase of row r is
// r % 8 in both.
template <typename C, bool P16> __device__ __forceinline__ uint32_t stage_row(int r, int plane)
{
    if constexpr (P16)
        return (uint32_t)((r >> 4) * (C::LINES * 2048) + plane * 2048 + (r & 15) * 128);
    else
        return (uint32_t)(plane * C::PLANE + r * 128);
}

template <typename C, bool P16> __device__ __forceinline__ uint32_t stage_off(int r, int c)
{
    return stage_row<C, P16>(r, c >> 3) + (uint32_t)((((c & 7) ^ (r & 7)) << 4));
}

// Slices.  Query heads h*Gq .. h*Gq + Gq-1 of K/V head h are served as NG
// slices of at most G each (virtual head v = h*NG + j holds query heads
// h*Gq + j*G + 0..), so that a warp's accumulators stay in registers
// whatever Gq is.  The decomposition runs over the K/V heads with
// grid / NG ranges: CTA i takes range i / NG for slice i % NG, so the NG
// CTAs of a range stream the same K/V rows side by side and all but the
// first read them from L2.  Each virtual head has its own query rows,
// arrival counter and workspace slots.
__device__ __forceinline__ int vh_count(const GqaParams &gp, int v)
{
    return min(gp.G, gp.Gq - (v % gp.NG) * gp.G);
}
// first query row of virtual head v of sequence b in q, out and lse
__device__ __forceinline__ long long vh_qrow0(const GqaParams &gp, int b, int v)
{
    return (long long)b * gp.s.H * gp.Gq + (long long)(v / gp.NG) * gp.Gq + (long long)(v % gp.NG) * gp.G;
}
// Workspace slot of piece i of (b, virtual head) bhv of slice `slice`: the
// piece_slot of the K/V head's decomposition (ranges), mapped to the CTA
// of that range and slice.
__device__ __forceinline__ long long vh_slot(const GqaParams &gp, const Ctx &ctx, long long bhv, unsigned i,
                                             int gf, long long off, int slice)
{
    const SplitParams &p = gp.s;
    if (p.decomp == DECOMP_SPLITS)
        return bhv * p.P + i;
    const long long sr = piece_slot(p, ctx, 0, i, gf, off);
    return ((sr >> 1) * gp.NG + slice) * 2 + (sr & 1);
}

// The chunk walk of the split kernel's producer over the CTA's chunks c =
// first, first + stride, ..., each chunk fetched as one K box and one V box
// (d/64 planes each) through the tensor maps.
//
// Paged K/V ([num_pages, Hkv, page_size, d]):
//  - page_size a multiple of CT: a chunk's tokens lie in one aligned
//    CT-token block of the sequence, hence in one page, so its rows are
//    consecutive rows of that page's (page, head) block; the box's rows past
//    them belong to something else and are masked like the rows past a
//    sequence's end.
//  - 16-token pages (P16): the chunk's aligned CT-token block spans two
//    pages.  Each page that holds some of the chunk's tokens is fetched as
//    one box [64, 16, d/64] into its half of the stage (stage_row), so stage
//    row r is token (t & ~(CT-1)) + r; the rows before the chunk's first
//    token are masked too.
template <typename C, bool P16> struct TmaProducer {
    Seg s;
    long long base;
    long long c;
    int stride;
    bool have;
    int t, ntok;
    int pg, pg2;      // paged: table entries of chunk c, loaded a chunk ahead
                      // (16-token pages: of the block's first and second page)

    __device__ __forceinline__ void locate(const GqaParams &gp, const Ctx &ctx)
    {
        const SplitParams &p = gp.s;
        while (s.valid && c >= base + seg_chunks<C::CT>(s)) {
            base += seg_chunks<C::CT>(s);
            seg_next(p, ctx, s);
        }
        have = s.valid;
        if (have) {
            chunk_coords<C::CT>(s, c - base, t, ntok);
            if (p.paged) {
                const int32_t *row = p.block_table + (long long)s.b * p.max_pages;
                if constexpr (P16) {
                    const int a = t & ~(C::CT - 1);   // the aligned block
                    pg = t < a + 16 ? __ldg(row + a / 16) : 0;
                    pg2 = t + ntok > a + 16 ? __ldg(row + a / 16 + 1) : 0;
                } else {
                    pg = __ldg(row + t / p.page_size);
                }
            }
        }
    }

    __device__ __forceinline__ void start(const GqaParams &gp, const Ctx &ctx, int first, int step)
    {
        seg_first(gp.s, ctx, s);
        base = 0;
        c = first;
        stride = step;
        locate(gp, ctx);
    }

    // A table entry checked before use: outside [0, num_pages) it is
    // recorded and replaced by page 0, so no row outside the pages is read.
    __device__ __forceinline__ static long long checked_page(const SplitParams &p, int entry)
    {
        long long page = entry;
        if (page < 0 || page >= p.num_pages) {
            atomicOr(p.status, STATUS_BAD_PAGE);
            page = 0;
        }
        return page;
    }

    // Copies the full CT-row boxes (rows past the tensor end read as zeros).
    __device__ __forceinline__ bool issue(const GqaParams &gp, const Ctx &ctx, uint32_t kdst,
                                          uint32_t bar, int lane)
    {
        if (!have)
            return false;
        if (lane == 0) {
            const SplitParams &p = gp.s;
            if constexpr (C::F8REG && P16) {
                // 16-token pages: a box of 16 E4M3 rows per page that holds
                // some of the chunk's tokens, into its half of the stage
                const int a = t & ~(C::CT - 1);
                const bool first = t < a + 16, second = t + ntok > a + 16;
                constexpr uint32_t HALF = 16 * 128;
                mbar_arrive_expect_tx(bar, 2 * HALF * ((first ? 1u : 0u) + (second ? 1u : 0u)));
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (half == 0 ? !first : !second)
                        continue;
                    const int blk = (int)(checked_page(p, half == 0 ? pg : pg2) * p.H + s.h);
                    tma_load_3d(kdst + half * HALF, &gp.tmk, 0, 0, blk, bar);
                    tma_load_3d(kdst + C::CHUNK_BYTES + half * HALF, &gp.tmv, 0, 0, blk, bar);
                }
            } else if constexpr (C::F8REG) {
                // a box of CT E4M3 rows (128 bytes each, 128-byte swizzle) per
                // operand; rows past the block's end read as zeros
                int y, blk;
                if (p.paged) {
                    y = t % p.page_size;
                    blk = (int)(checked_page(p, pg) * p.H + s.h);
                } else {
                    y = t;
                    blk = s.b * p.H + s.h;
                }
                mbar_arrive_expect_tx(bar, 2 * C::CHUNK_BYTES);
                tma_load_3d(kdst, &gp.tmk, 0, y, blk, bar);
                tma_load_3d(kdst + C::CHUNK_BYTES, &gp.tmv, 0, y, blk, bar);
            } else if constexpr (C::F8K && P16) {
                // 16-token pages: the chunk's rows in each of its (at most
                // two) pages, to the stage rows of their place in the
                // aligned block
                const int a = t & ~(C::CT - 1);
                const int t1 = t + ntok, mid = a + 16;
                const int n0 = t < mid ? min(t1, mid) - t : 0;   // tokens in the first page
                const int n1 = t1 > mid ? t1 - max(t, mid) : 0;  // and in the second
                mbar_arrive_expect_tx(bar, 2 * (uint32_t)(n0 + n1) * C::ROW);
                if (n0 > 0) {
                    const long long row = (checked_page(p, pg) * p.H + s.h) * 16 + (t - a);
                    const uint32_t dst = (uint32_t)(t - a) * C::ROW, bytes = (uint32_t)n0 * C::ROW;
                    bulk_g2s(kdst + dst, static_cast<const char *>(p.k) + row * C::ROW, bytes, bar);
                    bulk_g2s(kdst + C::CHUNK_BYTES + dst, static_cast<const char *>(p.v) + row * C::ROW, bytes, bar);
                }
                if (n1 > 0) {
                    const int r1 = max(t, mid) - mid;            // first row in the second page
                    const long long row = (checked_page(p, pg2) * p.H + s.h) * 16 + r1;
                    const uint32_t dst = (uint32_t)(16 + r1) * C::ROW, bytes = (uint32_t)n1 * C::ROW;
                    bulk_g2s(kdst + dst, static_cast<const char *>(p.k) + row * C::ROW, bytes, bar);
                    bulk_g2s(kdst + C::CHUNK_BYTES + dst, static_cast<const char *>(p.v) + row * C::ROW, bytes, bar);
                }
            } else if constexpr (C::F8K) {
                // the chunk's E4M3 rows as they are in memory: of the
                // sequence's (b, K/V head) block, or of the one page that
                // holds them (pages of a multiple of CT tokens)
                const long long row = p.paged ? (checked_page(p, pg) * p.H + s.h) * p.page_size + t % p.page_size
                                              : ((long long)s.b * p.H + s.h) * p.N + t;
                const uint32_t bytes = (uint32_t)ntok * C::ROW;
                mbar_arrive_expect_tx(bar, 2 * bytes);
                bulk_g2s(kdst, static_cast<const char *>(p.k) + row * C::ROW, bytes, bar);
                bulk_g2s(kdst + C::CHUNK_BYTES, static_cast<const char *>(p.v) + row * C::ROW, bytes, bar);
            } else if constexpr (P16) {
                const int a = t & ~(C::CT - 1);
                const bool first = t < a + 16, second = t + ntok > a + 16;
                constexpr uint32_t HALF = C::LINES * 16 * 128;   // one page: 16 rows, every plane
                mbar_arrive_expect_tx(bar, 2 * HALF * ((first ? 1u : 0u) + (second ? 1u : 0u)));
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (half == 0 ? !first : !second)
                        continue;
                    const int blk = (int)(checked_page(p, half == 0 ? pg : pg2) * p.H + s.h);
                    tma_load_4d(kdst + half * HALF, &gp.tmk, 0, 0, blk, 0, bar);
                    tma_load_4d(kdst + C::CHUNK_BYTES + half * HALF, &gp.tmv, 0, 0, blk, 0, bar);
                }
            } else {
                int y, blk;
                if (p.paged) {
                    y = t % p.page_size;
                    blk = (int)(checked_page(p, pg) * p.H + s.h);
                } else {
                    y = t;
                    blk = s.b * p.H + s.h;
                }
                mbar_arrive_expect_tx(bar, 2 * C::CHUNK_BYTES);
                tma_load_4d(kdst, &gp.tmk, 0, y, blk, 0, bar);
                tma_load_4d(kdst + C::CHUNK_BYTES, &gp.tmv, 0, y, blk, 0, bar);
            }
        }
        c += stride;
        locate(gp, ctx);
        return true;
    }
};

// Elements e and e + 1 of q (float32, float16 or bfloat16 by q_dtype; e
// even) as floats.
__device__ __forceinline__ float2 q_pair_f32(const void *q, int q_dtype, long long e)
{
    if (q_dtype == 0)
        return __ldg(reinterpret_cast<const float2 *>(static_cast<const float *>(q) + e));
    const uint32_t w = __ldg(reinterpret_cast<const unsigned int *>(static_cast<const uint16_t *>(q) + e));
    if (q_dtype == 1) {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    }
    __nv_bfloat162 h;
    memcpy(&h, &w, 4);
    return __bfloat1622float2(h);
}

// Two floats as an f16 pair (round to nearest even), the B-operand word of
// the f16 products.
__device__ __forceinline__ uint32_t f16_pair(float a, float b)
{
    const __half2 r = __floats2half2_rn(a, b);
    uint32_t u;
    memcpy(&u, &r, 4);
    return u;
}

// 2^e as a float for 0 <= e <= 127, built from its IEEE-754 bits (exact).
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }

// The power of two that brings a head's largest |q| (amax) below 2^14, as
// its exponent e >= 0: q is rounded to f16 for the E4M3 products, whose
// largest finite value is 65504, so a head with amax >= 2^14 is multiplied
// by 2^-e first (exact) and its scores by 2^e after.  0 for amax < 2^14,
// infinite or NaN.
__device__ __forceinline__ int q_range_exp(float amax)
{
    if (!(amax >= 16384.f) || !(amax <= 3.4028235e38f))
        return 0;
    return (int)((__float_as_uint(amax) >> 23) & 0xff) - 127 - 13;
}

// Score scale of one head column of S^T: one value for every head, or one
// per head column (E4M3 paths, whose heads may carry their own power of two).
struct UniformScale {
    float s;
    __device__ __forceinline__ float operator()(int, int) const { return s; }
};
template <int NQ> struct HeadScale {
    float s[NQ][2];   // [column tile][head 2(lane%4) + e]
    __device__ __forceinline__ float operator()(int j, int e) const { return s[j][e]; }
};

// 16 E4M3 bytes (elements 0..15) as 16 f16 values, exactly: elements 0..7
// in lo, 8..15 in hi (cvt.rn.f16x2.e4m3x2 takes a byte pair, the lower byte
// to the lower half).
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 &u, uint4 &lo, uint4 &hi)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("{\n\t.reg .b16 a, b;\n\t"
            "mov.b32 {a, b}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
            "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
            : "=r"(h[2 * i]), "=r"(h[2 * i + 1])
            : "r"(w[i]));
    lo = make_uint4(h[0], h[1], h[2], h[3]);
    hi = make_uint4(h[4], h[5], h[6], h[7]);
}

// A warp's 16 E4M3 rows (stage rows row0 .. row0+15, d bytes each) of K or
// V into its f16 area (stage_row<C, true> layout, rows 0..15); rows outside
// [vlo, vhi) become zeros.
template <typename C>
__device__ __forceinline__ void f8_rows_to_area(uint32_t stage, int row0, uint32_t area, int vlo, int vhi,
                                                int lane)
{
    constexpr int CPR = C::ROW / 16;               // 16-byte pieces per E4M3 row
    static_assert(CPR == 4 || CPR == 8 || CPR == 16, "d = 64, 128 or 256");
#pragma unroll
    for (int i = 0; i < 16 * CPR / 32; ++i) {
        // Each 8-lane phase of the 16-byte accesses takes two consecutive
        // rows, four pieces (64 bytes) of each: at d = 128 half a row's
        // pieces from the first and the other half from the second, at
        // d = 256 quarters of opposite parity.  Its loads then fall on all
        // 32 banks, and its stores on the two swizzle phases of adjacent
        // rows: no bank conflicts either way.
        int r, c16;
        if constexpr (CPR >= 8) {
            const int q = lane >> 2, hb = q & 1;
            r = 2 * (q >> 1) + hb + 8 * (i & 1);
            c16 = (lane & 3) + 4 * (hb ^ (i >> 1));
        } else {
            r = (lane >> 2) + 8 * i;
            c16 = lane & 3;
        }
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        if (r >= vlo && r < vhi) {
            const int sr = row0 + r;   // stage row
            // at d = 128 the rows were staged with the 128-byte swizzle
            const uint32_t src = C::F8REG ? stage + (uint32_t)(sr * 128 + ((c16 ^ (sr & 7)) << 4))
                                          : stage + (uint32_t)(sr * C::ROW + c16 * 16);
            uint4 u;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                         : "r"(src));
            e4m3x16_to_f16(u, lo, hi);
        }
        // elements 16 c16 .. 16 c16 + 15 are 16-byte columns 2 c16 and 2 c16 + 1
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(area + stage_off<C, true>(r, 2 * c16)),
                     "r"(lo.x), "r"(lo.y), "r"(lo.z), "r"(lo.w)
                     : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(area + stage_off<C, true>(r, 2 * c16 + 1)),
                     "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
                     : "memory");
    }
}

// Per-warp softmax state.  Query heads are the columns of S^T and O^T: in
// column tile j this thread has heads 8j + 2(lane%4) + {0, 1}, and of O^T
// the head dimensions 16i + lane/4 (+ 8) of every 16-row tile i (the mma
// accumulator layout).  m and l are per head; l is this thread's share.
template <typename C, int NQ> struct GqaState {
    float o[C::MT][NQ][4];
    float m[NQ][2];   // running max (base 2)
    float l[NQ][2];   // this thread's share of the running sums
};

// One warp's WT = 16 rows of a chunk (rows row0 .. row0+15 of the stage,
// rows vlo .. vhi-1 of them real tokens, vlo < vhi; V's other rows already
// zeroed): S^T = K Q^T on the tensor cores, the block-wise online-softmax
// update in fp32, then O^T += V^T (P_hi + P_lo)^T.  qb holds Q^T as B
// fragments: qb[j][s] = heads of column tile j, k-step s.
// kfrag(s, a) gives K's A fragments of k-step s (the default reads the
// stage with ldmatrix; E4M3 K converts them from registers).  scale(j, e)
// is the base-2 score scale of this thread's head column e of tile j.
template <typename T, typename C, int NQ, bool P16, typename KF, typename SC>
__device__ __forceinline__ void gqa_chunk_kf(KF kfrag, uint32_t vstage, int row0, int vlo, int vhi,
                                             const uint32_t (*qb)[C::KSTEPS][2], const SC &scale, int lane,
                                             GqaState<C, NQ> &st)
{
    // S^T for the warp's 16 tokens; even and odd k-steps accumulate
    // separately so the dependent MMA chains are half as long
    float sc[NQ][4], sx[NQ][4];
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
        sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
        sx[j][0] = sx[j][1] = sx[j][2] = sx[j][3] = 0.f;
    }
#pragma unroll
    for (int s = 0; s < C::KSTEPS; ++s) {
        uint32_t a[4];
        kfrag(s, a);
#pragma unroll
        for (int j = 0; j < NQ; ++j)
            Mma<T>::run((s & 1) ? sx[j] : sc[j], a, qb[j][s][0], qb[j][s][1]);
    }
    // base-2 scale; tokens lane/4 and lane/4 + 8 outside the valid rows are masked
    const int r = lane >> 2;
    const bool v0 = r >= vlo && r < vhi, v1 = r + 8 >= vlo && r + 8 < vhi;
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
        sc[j][0] = v0 ? (sc[j][0] + sx[j][0]) * scale(j, 0) : -INFINITY;
        sc[j][1] = v0 ? (sc[j][1] + sx[j][1]) * scale(j, 1) : -INFINITY;
        sc[j][2] = v1 ? (sc[j][2] + sx[j][2]) * scale(j, 0) : -INFINITY;
        sc[j][3] = v1 ? (sc[j][3] + sx[j][3]) * scale(j, 1) : -INFINITY;
    }
    // per head: the max over the chunk's 16 tokens (a head's tokens live in
    // the 8 lanes with the same lane % 4), the rescale, and P
    uint32_t ph[NQ][2], pl[NQ][2];
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
        float x0 = fmaxf(sc[j][0], sc[j][2]), x1 = fmaxf(sc[j][1], sc[j][3]);
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
            x0 = fmaxf(x0, __shfl_xor_sync(FULL_MASK, x0, o));
            x1 = fmaxf(x1, __shfl_xor_sync(FULL_MASK, x1, o));
        }
        const float mn0 = fmaxf(st.m[j][0], x0), mn1 = fmaxf(st.m[j][1], x1);  // finite: vhi > vlo
        const float a0 = ex2(st.m[j][0] - mn0), a1 = ex2(st.m[j][1] - mn1);
        st.m[j][0] = mn0;
        st.m[j][1] = mn1;
        const float p0 = ex2(sc[j][0] - mn0), p1 = ex2(sc[j][1] - mn1);
        const float p2 = ex2(sc[j][2] - mn0), p3 = ex2(sc[j][3] - mn1);
        st.l[j][0] = st.l[j][0] * a0 + (p0 + p2);
        st.l[j][1] = st.l[j][1] * a1 + (p1 + p3);
#pragma unroll
        for (int i = 0; i < C::MT; ++i) {
            st.o[i][j][0] *= a0;
            st.o[i][j][1] *= a1;
            st.o[i][j][2] *= a0;
            st.o[i][j][3] *= a1;
        }
        // P^T blocks (tokens 0-7 | 8-15) x (8 heads) as 16-bit pairs, high
        // part and the low part of its residual, turned into B fragments
        const uint32_t h0 = Mma<T>::pack(p0, p1), h1 = Mma<T>::pack(p2, p3);
        const float2 u0 = Mma<T>::unpack(h0), u1 = Mma<T>::unpack(h1);
        const uint32_t l0 = Mma<T>::pack(p0 - u0.x, p1 - u0.y), l1 = Mma<T>::pack(p2 - u1.x, p3 - u1.y);
        ph[j][0] = movmatrix_t(h0);
        ph[j][1] = movmatrix_t(h1);
        pl[j][0] = movmatrix_t(l0);
        pl[j][1] = movmatrix_t(l1);
    }
    // O^T += V^T P^T: V^T tiles (16 dims x 16 tokens) through ldmatrix.trans
    const int vtok = row0 + (lane & 7) + 8 * (lane >> 4);
#pragma unroll
    for (int i = 0; i < C::MT; ++i) {
        uint32_t a[4];
        ldsm_x4_t(vstage + stage_off<C, P16>(vtok, 2 * i + ((lane >> 3) & 1)), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            Mma<T>::run(st.o[i][j], a, ph[j][0], ph[j][1]);
            Mma<T>::run(st.o[i][j], a, pl[j][0], pl[j][1]);
        }
    }
}

// The chunk with K's fragments read from the stage.
template <typename T, typename C, int NQ, bool P16, typename SC>
__device__ __forceinline__ void gqa_chunk(uint32_t kstage, uint32_t vstage, int row0, int vlo, int vhi,
                                          const uint32_t (*qb)[C::KSTEPS][2], const SC &scale, int lane,
                                          GqaState<C, NQ> &st)
{
    const int ktok = row0 + (lane & 15);
    gqa_chunk_kf<T, C, NQ, P16>(
        [&](int s, uint32_t (&a)[4]) {
            ldsm_x4(kstage + stage_off<C, P16>(ktok, 2 * s + (lane >> 4)), a[0], a[1], a[2], a[3]);
        },
        vstage, row0, vlo, vhi, qb, scale, lane, st);
}

// E4M3 K at d = 128: the warp's 16 staged rows (128-byte swizzle) as raw
// ldmatrix fragments, two k-steps (two 16-byte columns) per x4 load; the
// stage can be freed once they and V's conversion are done.
template <typename C>
__device__ __forceinline__ void f8_k_raw(uint32_t stage, int row0, int lane, uint32_t (&kraw)[C::KSTEPS / 2][4])
{
    const int row = row0 + (lane & 15);
#pragma unroll
    for (int i = 0; i < C::KSTEPS / 2; ++i) {
        const int c = 2 * i + (lane >> 4);
        ldsm_x4(stage + (uint32_t)(row * 128 + ((c ^ (row & 7)) << 4)), kraw[i][0], kraw[i][1], kraw[i][2],
                kraw[i][3]);
    }
}

// A fragments of k-step s from the raw E4M3 K: thread (g, t) holds d values
// 16s + 4t .. 16s + 4t + 3 of rows g and g + 8; converted, they fill the
// fragment's k slots 2t, 2t+1 (a0, a1) and 2t+8, 2t+9 (a2, a3), so q's
// fragments take d = 16s + 4t (+1) and 16s + 4t + 2 (+3) in those slots.
__device__ __forceinline__ void f8_k_frag(const uint32_t *kr, uint32_t (&a)[4])
{
    asm("{\n\t.reg .b16 x, y;\n\t"
        "mov.b32 {x, y}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, x;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, y;\n\t}"
        : "=r"(a[0]), "=r"(a[2])
        : "r"(kr[0]));
    asm("{\n\t.reg .b16 x, y;\n\t"
        "mov.b32 {x, y}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, x;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, y;\n\t}"
        : "=r"(a[1]), "=r"(a[3])
        : "r"(kr[1]));
}

}  // namespace fd
