// fd_split.cuh -- the split-KV decode kernel (stage 1 of FlashDecoding, with
// an optional fused stage 2).
//
// What it computes: for each piece ("segment") [t0, t1) of a (b, h) sequence
// assigned to a CTA, the tile statistics of "FlashDecoding 数学推导" §2.4.1
// (m = max score, l = sum exp(s - m), o = sum exp(s - m) V / l), and either
// stores them (two-call path) or merges them with the other pieces of the
// same (b, h) using §2.4.2 (fused path).
//
// How (GB300): the path is bound by HBM bandwidth (every K/V byte is read
// once; ~1 flop per byte), so there are no tensor cores.  Each CTA is
// persistent (one per SM) and walks a contiguous list of segments.  Inside a
// CTA the warps form groups of GW; each group owns a ring of STAGES
// shared-memory stages.  A stage holds one chunk of CT tokens of K and the
// same tokens of V, filled by two 1-D bulk copies (cp.async.bulk, completion
// on a "full" mbarrier) issued by the group's first warp; each warp of the
// group takes its own WT rows of the chunk and signals an "empty" mbarrier
// when done, after which the stage is refilled.  Grouping keeps every copy
// large (GW * 4 KB) and the number of copies in flight per SM moderate,
// which the HBM/TMA path needs to stream near its peak.  Chunks of the CTA's
// token sequence go round-robin to the groups, so the CTA streams contiguous
// memory while groups never wait on each other inside a segment.
// Within a warp, LPT lanes cover one token row with 16-byte loads and the
// q.k partial sums are reduced with xor-shuffles.  The softmax state is
// updated once per chunk in the block form of the online-softmax update
// (running max, rescale by exp(m_old - m_new), unnormalised accumulator),
// with scores in base 2 (q pre-multiplied by scale*log2(e)) so that the
// exponentials are single ex2 instructions.  At a segment end each
// streaming warp hands its state to the CTA's merge warp through one of
// NBUF shared-memory buffers and goes on with the next segment; the merge
// warp merges the warps' states (the m/l/o merge), writes the result and,
// for a (b, h) split across CTAs, runs the last arriver's merge of the
// pieces.  No streaming warp waits for a merge, and after the set-up there
// is no block-wide barrier.
#pragma once

#include "fd_device.cuh"
#include "fd_internal.h"

namespace fd {

constexpr float LN2_F = 0.693147180559945309f;

#ifndef FD_WARPS
#define FD_WARPS 8
#endif
#ifndef FD_GROUP_WARPS
#define FD_GROUP_WARPS 2
#endif
#ifndef FD_STAGES
#define FD_STAGES 2
#endif
#ifndef FD_WARP_BYTES
#define FD_WARP_BYTES 4096
#endif
// packed two-lane fp32 FMAs (same operations, half the instructions)
#ifndef FD_NO_FMA2
#define FD_FMA2 1
#endif

// Ring shape per element type.  The FP8 cache carries twice the tokens per
// byte, so per byte it needs twice the arithmetic: it runs 15 streaming
// warps (more latency hiding) in groups of 5 with 3 KB per warp and stage,
// and 2 segment buffers to stay within shared memory (measured on GB300:
// 7.02 TB/s, as with 12 warps of 4 KB, which spill registers; 6.55 TB/s with
// 12 warps of 3 KB; 6.12 TB/s with the 16-bit shape).
#ifndef FD_FP8_WARPS
#define FD_FP8_WARPS 15
#endif
#ifndef FD_FP8_GROUP_WARPS
#define FD_FP8_GROUP_WARPS 5
#endif
#ifndef FD_FP8_STAGES
#define FD_FP8_STAGES FD_STAGES
#endif
#ifndef FD_FP8_WARP_BYTES
#define FD_FP8_WARP_BYTES 3072
#endif
// segment states in flight from the streaming warps to the merge warp
#ifndef FD_NBUF
#define FD_NBUF 4
#endif
#ifndef FD_FP8_NBUF
#define FD_FP8_NBUF 2
#endif
template <typename T> struct RingShape {
    static constexpr int WARPS = FD_WARPS, GW = FD_GROUP_WARPS, STAGES = FD_STAGES,
                         WARP_BYTES = FD_WARP_BYTES, NBUF = FD_NBUF;
};
template <> struct RingShape<__nv_fp8_e4m3> {
    static constexpr int WARPS = FD_FP8_WARPS, GW = FD_FP8_GROUP_WARPS, STAGES = FD_FP8_STAGES,
                         WARP_BYTES = FD_FP8_WARP_BYTES, NBUF = FD_FP8_NBUF;
};

template <typename T, int D> struct SplitCfg {
    using Elt = T;
    // only the FP8 cache takes q (and K/V scales) of another type
    static constexpr bool FP8 = std::is_same<T, __nv_fp8_e4m3>::value;
    static constexpr int ESZ = sizeof(T);
    static constexpr int VEC = Elem<T>::VEC;       // elements per lane vector (16 bytes)
    static constexpr int LPT = D / VEC;            // lanes per token row
    static constexpr int TPW = 32 / LPT;           // token rows per warp-wide load
    static constexpr int ROW = D * ESZ;            // bytes per token row
    static constexpr int WARPS = RingShape<T>::WARPS;   // streaming warps
    static constexpr int MW = WARPS;               // index of the merge warp
    static constexpr int THREADS = (WARPS + 1) * 32;
    static constexpr int GW = RingShape<T>::GW;    // warps sharing one ring
    static constexpr int GROUPS = WARPS / GW;
    static constexpr int STAGES = RingShape<T>::STAGES;
    static constexpr int WT = RingShape<T>::WARP_BYTES / ROW; // tokens per warp per chunk
    static constexpr int CT = GW * WT;             // tokens per chunk (per group)
    static constexpr int TOK = WT / TPW;           // tokens per lane group per chunk
    static constexpr int CHUNK_BYTES = CT * ROW;   // one of K or V
    static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;
    static constexpr int RING_BYTES = GROUPS * STAGES * STAGE_BYTES;
    static constexpr int NBUF = RingShape<T>::NBUF;   // segment states in flight to the merge warp
    static constexpr int SEG_FLOATS = 2 * WARPS + WARPS * D;   // per warp: m, l, then acc rows
    // ring full + empty, then segment full + free
    static constexpr int BAR_BYTES = GROUPS * STAGES * 2 * 8 + NBUF * 2 * 8;
    static constexpr int RED_BYTES = NBUF * SEG_FLOATS * 4;
    static_assert(LPT >= 1 && LPT <= 32 && 32 % LPT == 0, "row must map onto whole lanes");
    static_assert(WT % TPW == 0 && TOK >= 1, "chunk must cover whole warp steps");
    static_assert(WARPS % GW == 0, "warps must form whole groups");
    static_assert(D % 32 == 0, "the merge warp holds D / 32 output elements per lane");
    static_assert(RING_BYTES + BAR_BYTES + RED_BYTES + (BALANCED_MAX_B + 1) * 8 + BALANCED_MAX_B * 4 + 1024 <=
                      227 * 1024,
                  "ring, barriers, segment buffers, the balanced prefix sums and the static shared "
                  "memory fit in one CTA's 227 KB");

    static size_t smem_bytes(int decomp, int B)
    {
        size_t s = RING_BYTES + BAR_BYTES + RED_BYTES;
        if (decomp == DECOMP_BALANCED)
            s += (size_t)(B + 1) * 8 + (size_t)B * 4;
        return s;
    }
};

// A contiguous piece of one (b, h) sequence assigned to a CTA.
struct Seg {
    int b, h;
    int t0, t1;       // token range within the sequence
    int k;            // ordinal of the segment within the CTA's list
    int p;            // split index (DECOMP_SPLITS)
    long long pos;    // start in the concatenated token space (DECOMP_BALANCED)
    int span;         // its extent there (DECOMP_BALANCED)
    bool valid;
};

// Per-CTA view of the decomposition.
struct Ctx {
    int g;            // this CTA
    int G;            // CTAs launched
    int Geff;         // CTAs with work (balanced: min(G, T))
    long long T;      // total tokens over all (b, h) (balanced)
    long long beg, end;  // this CTA's range in the concatenated space
    const long long *cumH;  // [B+1] H * prefix sum of spans (balanced)
    const int *lenS;        // [B] clamped lengths (balanced)
};

// Extent of a (b, h) sequence of n tokens in the balanced decomposition's
// concatenated space: its tokens after a charge of seg_cost for starting it
// (the segment end before it, the query reload, the pipeline's refill), so
// that a CTA that switches sequences is given fewer tokens.  A segment
// covering [v0, v1) of that extent holds tokens [v0 - c, v1 - c) clamped at
// 0; one that falls inside the charge holds none and still counts as a
// piece.
__device__ __forceinline__ int bal_span(const SplitParams &p, int n)
{
    return n > 0 ? n + p.seg_cost : 0;
}

__device__ __forceinline__ void bal_tokens(const SplitParams &p, Seg &s, int v0, int v1)
{
    s.t0 = v0 > p.seg_cost ? v0 - p.seg_cost : 0;
    s.t1 = v1 > p.seg_cost ? v1 - p.seg_cost : 0;
    s.span = v1 - v0;
}

// Whether segment s is its whole (b, h) sequence of `len` tokens (its
// result then goes straight to the output).
__device__ __forceinline__ bool seg_whole(const SplitParams &p, const Seg &s, int len)
{
    if (p.decomp == DECOMP_SPLITS)
        return p.P == 1;
    return s.span == bal_span(p, len);
}

// Offset of (b, h) in the concatenated space.
__device__ __forceinline__ long long bal_offset(const SplitParams &p, const Ctx &c, int b, int h, int len)
{
    return c.cumH[b] + (long long)h * bal_span(p, len);
}

__device__ __forceinline__ int clamp_len(const SplitParams &p, int b)
{
    if (!p.lens)
        return p.N;
    int n = __ldg(p.lens + b);
    return n < 0 ? 0 : (n > p.N ? p.N : n);
}

__device__ __forceinline__ long long bal_bound(long long g, long long T, int Geff)
{
    return (g * T) / Geff;
}

// CTA owning token x of the concatenated space (balanced decomposition).
__device__ __forceinline__ int bal_owner(long long x, long long T, int Geff)
{
    return (int)(((x + 1) * (long long)Geff - 1) / T);
}

__device__ __forceinline__ int find_batch(const long long *cumH, int B, long long pos)
{
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (cumH[mid] <= pos)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void split_item(const SplitParams &p, long long item, Seg &s)
{
    const int bh = (int)(item / p.P);
    s.p = (int)(item % p.P);
    s.b = bh / p.H;
    s.h = bh % p.H;
    const int n = clamp_len(p, s.b);
    const long long chunk = ((long long)n + p.P - 1) / p.P;  // ceil(len / P)
    long long lo = (long long)s.p * chunk;
    if (lo > n)
        lo = n;
    long long hi = lo + chunk;
    if (hi > n)
        hi = n;
    s.t0 = (int)lo;
    s.t1 = (int)hi;
}

__device__ __forceinline__ void seg_first(const SplitParams &p, const Ctx &c, Seg &s)
{
    s.k = 0;
    if (p.decomp == DECOMP_SPLITS) {
        const long long items = (long long)p.B * p.H * p.P;
        s.valid = c.g < items;
        if (s.valid)
            split_item(p, c.g, s);
        return;
    }
    s.valid = c.g < c.Geff;
    if (!s.valid)
        return;
    s.pos = c.beg;
    s.b = find_batch(c.cumH, p.B, s.pos);
    const int span = bal_span(p, c.lenS[s.b]);
    const long long rel = s.pos - c.cumH[s.b];
    s.h = (int)(rel / span);
    const int v0 = (int)(rel % span);
    const long long room = c.end - s.pos;
    bal_tokens(p, s, v0, (long long)(span - v0) < room ? span : (int)(v0 + room));
}

__device__ __forceinline__ void seg_next(const SplitParams &p, const Ctx &c, Seg &s)
{
    s.k += 1;
    if (p.decomp == DECOMP_SPLITS) {
        const long long item = (long long)c.g + (long long)s.k * c.G;
        s.valid = item < (long long)p.B * p.H * p.P;
        if (s.valid)
            split_item(p, item, s);
        return;
    }
    s.pos += s.span;
    if (s.pos >= c.end) {
        s.valid = false;
        return;
    }
    // the previous segment ended at the end of its sequence
    s.h += 1;
    if (s.h == p.H) {
        s.h = 0;
        do {
            s.b += 1;
        } while (c.lenS[s.b] == 0);
    }
    const int span = bal_span(p, c.lenS[s.b]);
    const long long room = c.end - s.pos;
    bal_tokens(p, s, 0, (long long)span < room ? span : (int)room);
}

// Balanced decomposition set-up, run by every thread of the CTA: clamped
// lengths into lenS, H * exclusive prefix sums into cumH[0..B], and this
// CTA's range of the concatenated token space in ctx.  Contains barriers.
template <int THREADS, int WARPS>
__device__ __forceinline__ void balanced_setup(const SplitParams &p, Ctx &ctx, long long *cumH,
                                               int *lenS)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    constexpr int PER = (BALANCED_MAX_B + THREADS - 1) / THREADS;
    long long v[PER];
    long long run = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int b = tid * PER + i;
        long long x = 0;
        if (b < p.B) {
            const int n = clamp_len(p, b);
            lenS[b] = n;
            x = (long long)bal_span(p, n) * p.H;
        }
        v[i] = run;
        run += x;
    }
    // inclusive scan of per-thread totals across the block
    long long incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o)
            incl += y;
    }
    __shared__ long long warp_tot[WARPS];
    if (lane == 31)
        warp_tot[w] = incl;
    __syncthreads();
    long long wbase = 0;
    for (int i = 0; i < w; ++i)
        wbase += warp_tot[i];
    const long long excl = wbase + incl - run;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int b = tid * PER + i;
        if (b < p.B)
            cumH[b] = excl + v[i];
    }
    if (tid == THREADS - 1)
        cumH[p.B] = excl + run;
    __syncthreads();
    ctx.T = cumH[p.B];
    // at least BALANCED_MIN_TOKENS tokens per CTA: a small problem uses
    // fewer, fuller CTAs (fewer pieces to merge)
    const long long want = (ctx.T + BALANCED_MIN_TOKENS - 1) / BALANCED_MIN_TOKENS;
    ctx.Geff = (int)(want < (long long)ctx.G ? want : (long long)ctx.G);
    if (ctx.g < ctx.Geff) {
        ctx.beg = bal_bound(ctx.g, ctx.T, ctx.Geff);
        ctx.end = bal_bound(ctx.g + 1, ctx.T, ctx.Geff);
    }
}

// Chunks lie on a fixed grid of the sequence's token index (multiples of CT),
// so a chunk never straddles more pages than it must; a segment's first and
// last chunks may be partial.
template <int CT> __device__ __forceinline__ long long seg_chunks(const Seg &s)
{
    if (s.t1 <= s.t0)
        return 0;
    return (long long)((s.t1 + CT - 1) / CT - s.t0 / CT);
}

// First token and token count of chunk i of segment s.
template <int CT>
__device__ __forceinline__ void chunk_coords(const Seg &s, long long i, int &t, int &ntok)
{
    const long long blk = s.t0 / CT + i;
    const long long lo = blk * CT;
    t = (int)(lo > s.t0 ? lo : s.t0);
    const long long hi = lo + CT < s.t1 ? lo + CT : s.t1;
    ntok = (int)(hi - t);
}

// Producer side of a group's ring: walks the group's chunks (c = g, g+G,
// ...) of the CTA's chunk sequence and issues the bulk copies for the next.
// It always knows the coordinates of the chunk it will issue next and, for a
// paged cache, has that chunk's block-table entries already loading into
// registers (lane j holds pieces j and j+32), so a refill never waits on a
// table lookup.
template <typename C> struct Producer {
    Seg s;
    long long base;   // chunk index of s's first chunk
    long long c;      // next chunk to issue
    bool have;        // chunk c exists
    int t, ntok;      // its first token and token count
    int pg0, pg1;     // prefetched page entries of its pieces lane, lane + 32

    __device__ __forceinline__ void locate(const SplitParams &p, const Ctx &ctx, int lane)
    {
        while (s.valid && c >= base + seg_chunks<C::CT>(s)) {
            base += seg_chunks<C::CT>(s);
            seg_next(p, ctx, s);
        }
        have = s.valid;
        if (!have)
            return;
        chunk_coords<C::CT>(s, c - base, t, ntok);
        if (p.paged) {
            const int ps = p.page_size;
            const int first = t / ps;
            const int npieces = (t + ntok - 1) / ps - first + 1;
            const int32_t *row = p.block_table + (long long)s.b * p.max_pages + first;
            pg0 = lane < npieces ? __ldg(row + lane) : 0;
            pg1 = lane + 32 < npieces ? __ldg(row + lane + 32) : 0;
        }
    }

    __device__ __forceinline__ void start(const SplitParams &p, const Ctx &ctx, int first_chunk,
                                          int lane)
    {
        seg_first(p, ctx, s);
        base = 0;
        c = first_chunk;
        locate(p, ctx, lane);
    }

    __device__ __forceinline__ bool issue(const SplitParams &p, const Ctx &ctx, uint32_t kdst,
                                          uint32_t bar, int lane)
    {
        if (!have)
            return false;
        const uint32_t bytes = (uint32_t)ntok * C::ROW;
        if (lane == 0)
            mbar_arrive_expect_tx(bar, 2 * bytes);
        if (!p.paged) {
            if (lane == 0) {
                const long long row = ((long long)s.b * p.H + s.h) * p.N + t;
                const char *ksrc = static_cast<const char *>(p.k) + row * C::ROW;
                const char *vsrc = static_cast<const char *>(p.v) + row * C::ROW;
#ifdef FD_L2_EVICT_FIRST
                const uint64_t pol = policy_evict_first();
                bulk_g2s_hint(kdst, ksrc, bytes, bar, pol);
                bulk_g2s_hint(kdst + C::CHUNK_BYTES, vsrc, bytes, bar, pol);
#else
                bulk_g2s(kdst, ksrc, bytes, bar);
                bulk_g2s(kdst + C::CHUNK_BYTES, vsrc, bytes, bar);
#endif
            }
        } else {
            // the chunk's rows split at page boundaries: lane j copies pieces
            // j, j+32, ... (page entries prefetched by locate())
            __syncwarp();
            const int ps = p.page_size;
            const int first = t / ps;
            const int npieces = (t + ntok - 1) / ps - first + 1;
            for (int j = lane; j < npieces; j += 32) {
                const int lp = first + j;
                const int r0 = max(t, lp * ps);
                const int r1 = min(t + ntok, (lp + 1) * ps);
                long long pg = j < 32 ? pg0
                             : j < 64 ? pg1
                                      : __ldg(p.block_table + (long long)s.b * p.max_pages + lp);
                if (pg < 0 || pg >= p.num_pages) {
                    // never read outside the pages: record it, read page 0
                    atomicOr(p.status, STATUS_BAD_PAGE);
                    pg = 0;
                }
                const long long row = (pg * p.H + s.h) * ps + (r0 - lp * ps);
                const uint32_t nb = (uint32_t)(r1 - r0) * C::ROW;
                const uint32_t off = (uint32_t)(r0 - t) * C::ROW;
                bulk_g2s(kdst + off, static_cast<const char *>(p.k) + row * C::ROW, nb, bar);
                bulk_g2s(kdst + C::CHUNK_BYTES + off, static_cast<const char *>(p.v) + row * C::ROW, nb,
                         bar);
            }
        }
        c += C::GROUPS;
        locate(p, ctx, lane);
        return true;
    }
};

// Merge online-softmax state (m2, l2, a2) into (m, l, a); scores in base 2.
template <int VEC>
__device__ __forceinline__ void merge_state(float &m, float &l, float *a, float m2, float l2,
                                            const float *a2)
{
    const float M = fmaxf(m, m2);
    if (M == -INFINITY)
        return;  // both empty
    const float e1 = ex2(m - M), e2 = ex2(m2 - M);
    l = l * e1 + l2 * e2;
#pragma unroll
    for (int i = 0; i < VEC; ++i)
        a[i] = a[i] * e1 + a2[i] * e2;
    m = M;
}

// The warp's WT rows of one chunk: block-wise online-softmax update of the
// lane group's state with its TOK token rows (ntok valid rows from kbase /
// vbase).
template <typename T, int D, bool FULL>
__device__ __forceinline__ void process_chunk(uint32_t kbase, uint32_t vbase, int ntok, int grp,
                                              int col, const float *qf, float &m, float &l,
                                              float *acc)
{
    using C = SplitCfg<T, D>;
    float s[C::TOK];
#pragma unroll
    for (int t = 0; t < C::TOK; ++t) {
        const int row = t * C::TPW + grp;
        if (FULL || row < ntok) {
            const uint4 u = lds128(kbase + row * C::ROW + col * 16);
            float kf[C::VEC];
            Elem<T>::widen(u, kf);
#ifdef FD_FMA2
            uint64_t d2 = pack2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < C::VEC; i += 2)
                d2 = fma2(pack2(qf[i], qf[i + 1]), pack2(kf[i], kf[i + 1]), d2);
            float d0, d1;
            unpack2(d2, d0, d1);
#else
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int i = 0; i < C::VEC; i += 2) {
                d0 = fmaf(qf[i], kf[i], d0);
                d1 = fmaf(qf[i + 1], kf[i + 1], d1);
            }
#endif
            s[t] = d0 + d1;
        } else {
            s[t] = -INFINITY;
        }
    }
#pragma unroll
    for (int o = C::LPT / 2; o >= 1; o >>= 1) {
#pragma unroll
        for (int t = 0; t < C::TOK; ++t)
            s[t] += __shfl_xor_sync(FULL_MASK, s[t], o);
    }
    float cmax = s[0];
#pragma unroll
    for (int t = 1; t < C::TOK; ++t)
        cmax = fmaxf(cmax, s[t]);
    const float mnew = fmaxf(m, cmax);
    if (mnew == -INFINITY)
        return;  // this lane group has no valid row yet
    const float alpha = ex2(m - mnew);
    l *= alpha;
#pragma unroll
    for (int i = 0; i < C::VEC; ++i)
        acc[i] *= alpha;
#pragma unroll
    for (int t = 0; t < C::TOK; ++t) {
        const int row = t * C::TPW + grp;
        if (FULL || row < ntok) {
            const float pj = ex2(s[t] - mnew);
            l += pj;
            const uint4 u = lds128(vbase + row * C::ROW + col * 16);
            float vf[C::VEC];
            Elem<T>::widen(u, vf);
#ifdef FD_FMA2
            const uint64_t pp = pack2(pj, pj);
#pragma unroll
            for (int i = 0; i < C::VEC; i += 2) {
                const uint64_t a2 = fma2(pp, pack2(vf[i], vf[i + 1]), pack2(acc[i], acc[i + 1]));
                unpack2(a2, acc[i], acc[i + 1]);
            }
#else
#pragma unroll
            for (int i = 0; i < C::VEC; ++i)
                acc[i] = fmaf(pj, vf[i], acc[i]);
#endif
        }
    }
    m = mnew;
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        x = fmaxf(x, __shfl_xor_sync(FULL_MASK, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        x += __shfl_xor_sync(FULL_MASK, x, o);
    return x;
}

// An L2 load that a dry pass skips (its instruction still runs, predicated
// off, so the code is the same).
__device__ __forceinline__ float ldcg_if(bool live, const float *ptr)
{
    return live ? __ldcg(ptr) : 0.f;
}

// Workspace slot of the i-th piece of (b, h) (see the decompositions).
__device__ __forceinline__ long long piece_slot(const SplitParams &p, const Ctx &ctx, int bh,
                                                unsigned i, int gf, long long off)
{
    if (p.decomp == DECOMP_SPLITS)
        return (long long)bh * p.P + i;
    const long long g = gf + (long long)i;
    return (i == 0 && bal_bound(gf, ctx.T, ctx.Geff) != off) ? 2 * g + 1 : 2 * g;
}

// Stage 2, run by the merge warp of the last piece of (b, h) to arrive: the
// m/l/o merge of "FlashDecoding 数学推导" §2.4.2 over its `target` workspace
// partials (normalised o, m in base 2, l), read from L2.  Lane j owns output
// elements j, j + 32, ...; the pieces' weights are formed 32 at a time, one
// per lane, and broadcast by shuffles, so the merge needs no barrier.
template <int D>
__device__ __forceinline__ void merge_pieces(const SplitParams &p, const Ctx &ctx, int bh,
                                             unsigned target, int gf, long long off, int lane,
                                             bool live = true)
{
    constexpr int DPL = D / 32;
    // the first 32 pieces keep their slot and (m, l) in registers
    long long s0 = 0;
    float m0 = -INFINITY, l0 = 0.f;
    if ((unsigned)lane < target) {
        s0 = piece_slot(p, ctx, bh, (unsigned)lane, gf, off);
        m0 = ldcg_if(live, p.ws_ml + 2 * s0);
        l0 = ldcg_if(live, p.ws_ml + 2 * s0 + 1);
    }
    float mx = l0 > 0.f ? m0 : -INFINITY;
    for (unsigned i = lane + 32; i < target; i += 32) {
        const long long sl = piece_slot(p, ctx, bh, i, gf, off);
        if (ldcg_if(live, p.ws_ml + 2 * sl + 1) > 0.f)
            mx = fmaxf(mx, ldcg_if(live, p.ws_ml + 2 * sl));
    }
    const float M = warp_max(mx);
    float L = 0.f, O[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j)
        O[j] = 0.f;
    for (unsigned base = 0; base < target; base += 32) {
        long long sl = s0;
        float m = m0, l = l0;
        if (base > 0) {
            sl = 0;
            m = -INFINITY;
            l = 0.f;
            if (base + lane < target) {
                sl = piece_slot(p, ctx, bh, base + lane, gf, off);
                m = ldcg_if(live, p.ws_ml + 2 * sl);
                l = ldcg_if(live, p.ws_ml + 2 * sl + 1);
            }
        }
        const float e = l > 0.f ? ex2(m - M) * l : 0.f;
        L += e;
        const int n = (int)min(32u, target - base);
        // 4 pieces' rows in flight at a time (a larger batch only adds code,
        // fetched cold from memory when the merge runs once per sequence)
        for (int i0 = 0; i0 < n; i0 += 4) {
            float x[4][DPL], ei[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                ei[u] = __shfl_sync(FULL_MASK, e, i0 + u);
                const long long si = __shfl_sync(FULL_MASK, sl, i0 + u);
#pragma unroll
                for (int j = 0; j < DPL; ++j)
                    x[u][j] = (i0 + u < n) ? ldcg_if(live, p.ws_o + si * D + lane + 32 * j) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
#pragma unroll
                for (int j = 0; j < DPL; ++j)
                    O[j] = ei[u] > 0.f ? fmaf(ei[u], x[u][j], O[j]) : O[j];
            }
        }
    }
    L = warp_sum(L);
    const bool nonempty = L > 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j)
        if (live)
            store_out(p.out, (long long)bh * D + lane + 32 * j, p.out_dtype, nonempty ? O[j] / L : 0.f);
    if (live && lane == 0 && p.lse)
        p.lse[bh] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
}

// The merge warp.  It walks the CTA's segments in the streaming warps'
// order; for segment k it waits until every streaming warp has handed over
// its (m, l, acc) in buffer k % NBUF, merges them (the m/l/o merge of
// "FlashDecoding 数学推导" §2.4.2), frees the buffer, and writes the result:
// out and lse for a whole sequence, the two-call partial, or a workspace
// partial whose arrival it counts, merging all pieces of the (b, h) if it is
// the last to arrive.  The streaming warps never wait for any of this unless
// all NBUF buffers are taken.
template <typename C, int D>
__device__ __forceinline__ void merge_warp(const SplitParams &p, const Ctx &ctx, const float *red,
                                           uint32_t sfull, uint32_t sfree, int lane)
{
    constexpr int DPL = D / 32;
    Seg s;
    seg_first(p, ctx, s);
    int k = 0;
    // The first pass over the first segment runs this code with every store,
    // arrival and wait switched off: the merge warp is idle at the start, and
    // the pass brings the code into the instruction cache, where the real
    // merges find it (run once per segment, after an L2 flush or a long
    // stream it would otherwise be fetched from DRAM, line by line).
    bool live = false;
#pragma unroll 1
    while (s.valid) {
        // the segment's facts, worked out while its data streams
        const int bh = s.b * p.H + s.h;
        const int len = (p.decomp == DECOMP_BALANCED) ? ctx.lenS[s.b] : clamp_len(p, s.b);
        bool complete;
        long long slot;
        if (p.decomp == DECOMP_SPLITS) {
            complete = (p.P == 1);
            slot = (long long)bh * p.P + s.p;
        } else {
            complete = seg_whole(p, s, len);
            slot = 2LL * ctx.g + (s.k == 0 ? 0 : 1);
        }
        // V's dequantisation scale is common to every row of (b, h)
        const float vs = (C::FP8 && p.v_scale) ? __ldg(p.v_scale + bh) : 1.f;

        const int buf = k % C::NBUF;
        if (live && !mbar_wait_bounded_sleep(sfull + buf * 8, (uint32_t)(k / C::NBUF) & 1, 1000000)) {
            if (lane == 0)
                atomicOr(p.status, STATUS_TIMEOUT);
            return;
        }
        const float *rm = red + buf * C::SEG_FLOATS;
        const float *rl = rm + C::WARPS;
        const float *ra = rl + C::WARPS;
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < C::WARPS; ++i)
            if (rl[i] > 0.f)
                M = fmaxf(M, rm[i]);
        float L = 0.f, O[DPL];
#pragma unroll
        for (int j = 0; j < DPL; ++j)
            O[j] = 0.f;
#pragma unroll
        for (int i = 0; i < C::WARPS; ++i) {
            if (rl[i] > 0.f) {
                const float e = ex2(rm[i] - M);
                L = fmaf(e, rl[i], L);
#pragma unroll
                for (int j = 0; j < DPL; ++j)
                    O[j] = fmaf(e, ra[i * D + lane + 32 * j], O[j]);
            }
        }
        if (live)
            mbar_arrive(sfree + buf * 8);  // the streaming warps may refill the buffer
        const bool nonempty = L > 0.f;
        float o[DPL];
#pragma unroll
        for (int j = 0; j < DPL; ++j)
            o[j] = nonempty ? O[j] / L * vs : 0.f;

        if (p.out_kind == OUT_PARTIALS) {
#pragma unroll
            for (int j = 0; j < DPL; ++j)
                if (live)
                    p.o_part[slot * D + lane + 32 * j] = o[j];
            if (live && lane == 0) {
                p.m_part[slot] = nonempty ? M * LN2_F : -INFINITY;
                p.l_part[slot] = L;
                if (p.lse_part)
                    p.lse_part[slot] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
            }
        } else if (complete && live) {
#pragma unroll
            for (int j = 0; j < DPL; ++j)
                store_out(p.out, (long long)bh * D + lane + 32 * j, p.out_dtype, o[j]);
            if (lane == 0 && p.lse)
                p.lse[bh] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
        } else {
            // workspace partial: normalised o, m in base 2, l
#pragma unroll
            for (int j = 0; j < DPL; ++j)
                if (live)
                    p.ws_o[slot * D + lane + 32 * j] = o[j];
            if (live && lane == 0) {
                p.ws_ml[2 * slot] = nonempty ? M : -INFINITY;
                p.ws_ml[2 * slot + 1] = L;
            }
            // count the arrival; the last piece of this (b, h) merges all of them
            unsigned target;
            int gf = 0;
            long long off = 0;
            if (p.decomp == DECOMP_SPLITS) {
                target = (unsigned)p.P;
            } else {
                off = bal_offset(p, ctx, s.b, s.h, len);
                gf = bal_owner(off, ctx.T, ctx.Geff);
                const int gl = bal_owner(off + bal_span(p, len) - 1, ctx.T, ctx.Geff);
                target = (unsigned)(gl - gf + 1);
            }
            __threadfence();
            __syncwarp();
            unsigned old = target - 1;  // the dry pass runs the merge, to no effect
            if (live && lane == 0)
                old = atomicInc(p.ws_cnt + bh, target - 1);
            old = __shfl_sync(FULL_MASK, old, 0);
            if (old == target - 1) {
                __threadfence();
                merge_pieces<D>(p, ctx, bh, target, gf, off, lane, live);
            }
        }
        if (!live) {
            live = true;  // now the same segment for real
            continue;
        }
        ++k;
        seg_next(p, ctx, s);
    }
}

// This lane's slice of the query row of (b, h) = bh, pre-multiplied by the
// score scale in base 2 and, for the FP8 cache, by K's dequantisation scale.
// Only the FP8 kernel reads q of a run-time type: in the others q has the
// kernel's element type, one 16-byte load (a run-time type switch there
// slowed the 16-token paged cache by 11% on GB300).
template <typename C, int D>
__device__ __forceinline__ void load_q_scaled(const SplitParams &p, int bh, int col, float *qf)
{
    float qs = p.scale_log2;
    if constexpr (C::FP8) {
        load_q<C::VEC>(p.q, p.q_dtype, (long long)bh * D + col * C::VEC, qf);
        if (p.k_scale)
            qs *= __ldg(p.k_scale + bh);
    } else {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const char *>(p.q) +
                                                              ((long long)bh * D + col * C::VEC) * C::ESZ));
        Elem<typename C::Elt>::widen(u, qf);
    }
#pragma unroll
    for (int i = 0; i < C::VEC; ++i)
        qf[i] *= qs;
}

template <typename T, int D>
__global__ void __launch_bounds__(SplitCfg<T, D>::THREADS, FD_CTAS_PER_SM) split_kernel(const SplitParams p)
{
    using C = SplitCfg<T, D>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int w = tid >> 5;
    const int grp = lane / C::LPT;
    const int col = lane % C::LPT;

    unsigned char *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::RING_BYTES);
    float *red = reinterpret_cast<float *>(smem + C::RING_BYTES + C::BAR_BYTES);
    long long *cumH = reinterpret_cast<long long *>(smem + C::RING_BYTES + C::BAR_BYTES + C::RED_BYTES);
    int *lenS = reinterpret_cast<int *>(cumH + p.B + 1);

    // bars: ring full [GROUPS][STAGES], ring empty [GROUPS][STAGES], then
    // segment full [NBUF] (every streaming lane arrives) and segment free
    // [NBUF] (the merge warp's lanes arrive)
    const uint32_t sfull = smem_addr(&bars[2 * C::GROUPS * C::STAGES]);
    const uint32_t sfree = sfull + C::NBUF * 8;
    if (tid == 0) {
        for (int i = 0; i < C::GROUPS * C::STAGES; ++i) {
            mbar_init(smem_addr(&bars[i]), 1);
            mbar_init(smem_addr(&bars[C::GROUPS * C::STAGES + i]), C::GW);
        }
        for (int i = 0; i < C::NBUF; ++i) {
            mbar_init(sfull + i * 8, C::WARPS * 32);
            mbar_init(sfree + i * 8, 32);
        }
    }

    Ctx ctx;
    ctx.g = blockIdx.x;
    ctx.G = p.grid;
    ctx.cumH = cumH;
    ctx.lenS = lenS;
    ctx.T = 0;
    ctx.Geff = 0;
    ctx.beg = ctx.end = 0;
    if (p.decomp == DECOMP_BALANCED) {
        balanced_setup<C::THREADS, C::WARPS + 1>(p, ctx, cumH, lenS);
        // sequences of length 0 are touched by no CTA: write their result here
        for (long long bh = (long long)ctx.g * C::THREADS + tid; bh < (long long)p.B * p.H;
             bh += (long long)ctx.G * C::THREADS) {
            if (lenS[bh / p.H] == 0) {
                for (int i = 0; i < D; ++i)
                    store_out(p.out, bh * D + i, p.out_dtype, 0.f);
                if (p.lse)
                    p.lse[bh] = -INFINITY;
            }
        }
    }
    fence_mbar_init();
    __syncthreads();  // the last block-wide barrier: the roles part here

    // (the streaming warps' code comes first: it is what runs at start-up)
    if (w < C::MW) {
        const int grp_id = w / C::GW;     // this warp's group
        const int gw = w % C::GW;         // its index inside the group
        const bool issuer = (gw == 0);
        const uint32_t ring_base = smem_addr(ring) + (uint32_t)(grp_id * C::STAGES * C::STAGE_BYTES);
        const uint32_t bar_base = smem_addr(&bars[grp_id * C::STAGES]);                 // full
        const uint32_t ebar_base = smem_addr(&bars[(C::GROUPS + grp_id) * C::STAGES]);  // empty
        const uint32_t my_rows = (uint32_t)(gw * C::WT * C::ROW);  // this warp's rows in a stage

        // The first segment's query row is requested before any K/V copy: behind
        // the CTAs' first burst of copies its load would wait microseconds.
        const int qsize = C::FP8 ? (p.q_dtype == 0 ? 4 : 2) : C::ESZ;
        Seg cs;
        seg_first(p, ctx, cs);
        if (cs.valid) {
            const int bh0 = cs.b * p.H + cs.h;
            prefetch_l1(static_cast<const char *>(p.q) + ((long long)bh0 * D + col * C::VEC) * qsize);
            if (C::FP8 && p.k_scale && lane == 0)
                prefetch_l1(p.k_scale + bh0);
        }

        Producer<C> prod;
        if (issuer)
            prod.start(p, ctx, grp_id, lane);
        int issued = 0;   // chunks issued by this warp (issuers only)
        int landed = 0;   // chunks whose copies this warp has seen complete
        bool dead = false;
        if (issuer) {
#pragma unroll 1
            for (int s = 0; s < C::STAGES; ++s) {
                if (!prod.issue(p, ctx, ring_base + s * C::STAGE_BYTES, bar_base + s * 8, lane))
                    break;
                ++issued;
            }
        }

        float qf[C::VEC];
        if (cs.valid)
            load_q_scaled<C, D>(p, cs.b * p.H + cs.h, col, qf);
        long long cbase = 0;
        int consumed = 0;
        int k = 0;        // segment ordinal
#pragma unroll 1
        while (cs.valid) {
            const long long nc = seg_chunks<C::CT>(cs);
            Seg nx = cs;
            seg_next(p, ctx, nx);
            if (nx.valid) {
                // the next segment's query row (and K scale) start loading now
                const int nbh = nx.b * p.H + nx.h;
                prefetch_l1(static_cast<const char *>(p.q) + ((long long)nbh * D + col * C::VEC) * qsize);
                if (C::FP8 && p.k_scale && lane == 0)
                    prefetch_l1(p.k_scale + nbh);
            }
            float m = -INFINITY, l = 0.f, acc[C::VEC];
#pragma unroll
            for (int i = 0; i < C::VEC; ++i)
                acc[i] = 0.f;

            long long c = cbase + ((grp_id - cbase % C::GROUPS) % C::GROUPS + C::GROUPS) % C::GROUPS;
#pragma unroll 1
            for (; c < cbase + nc; c += C::GROUPS) {
                const int stage = consumed % C::STAGES;
                const uint32_t parity = (consumed / C::STAGES) & 1;
                ++consumed;
                if (!dead) {
                    if (mbar_wait_bounded(bar_base + stage * 8, parity))
                        ++landed;
                    else
                        dead = true;
                }
                int t, ntok_chunk;
                chunk_coords<C::CT>(cs, c - cbase, t, ntok_chunk);
                const int ntok = ntok_chunk - gw * C::WT;  // this warp's valid rows
                const uint32_t kb = ring_base + stage * C::STAGE_BYTES;
                if (!dead && ntok > 0) {
                    if (ntok >= C::WT)
                        process_chunk<T, D, true>(kb + my_rows, kb + C::CHUNK_BYTES + my_rows, C::WT,
                                                  grp, col, qf, m, l, acc);
                    else
                        process_chunk<T, D, false>(kb + my_rows, kb + C::CHUNK_BYTES + my_rows, ntok,
                                                   grp, col, qf, m, l, acc);
                }
                __syncwarp();
                if (C::GW > 1) {
                    // release the stage; the issuer refills it once every warp of
                    // the group has released it
                    if (!dead && lane == 0)
                        mbar_arrive(ebar_base + stage * 8);
                    if (issuer && !dead && !mbar_wait_bounded(ebar_base + stage * 8, parity))
                        dead = true;
                }
                if (issuer && !dead && prod.issue(p, ctx, kb, bar_base + stage * 8, lane))
                    ++issued;
            }

            // ---- segment end: merge the lane groups, hand the state over ----
#pragma unroll
            for (int o = C::LPT; o < 32; o <<= 1) {
                float a2[C::VEC];
                const float m2 = __shfl_xor_sync(FULL_MASK, m, o);
                const float l2 = __shfl_xor_sync(FULL_MASK, l, o);
#pragma unroll
                for (int i = 0; i < C::VEC; ++i)
                    a2[i] = __shfl_xor_sync(FULL_MASK, acc[i], o);
                merge_state<C::VEC>(m, l, acc, m2, l2, a2);
            }
            const int buf = k % C::NBUF;
            if (!dead && !mbar_wait_bounded(sfree + buf * 8, ((uint32_t)(k / C::NBUF) & 1) ^ 1))
                dead = true;
            if (!dead) {
                float *rm = red + buf * C::SEG_FLOATS;
                if (grp == 0) {
#pragma unroll
                    for (int i = 0; i < C::VEC; ++i)
                        rm[2 * C::WARPS + w * D + col * C::VEC + i] = acc[i];
                    if (col == 0) {
                        rm[w] = m;
                        rm[C::WARPS + w] = l;
                    }
                }
                mbar_arrive(sfull + buf * 8);  // every lane: releases its own writes
            }
            ++k;
            cbase += nc;
            cs = nx;
            if (cs.valid)
                load_q_scaled<C, D>(p, cs.b * p.H + cs.h, col, qf);
        }

        if (dead) {
            if (lane == 0)
                atomicOr(p.status, STATUS_TIMEOUT);
            // wait (bounded) for this warp's copies still in flight
            for (int i = landed; i < issued; ++i)
                mbar_wait_bounded(bar_base + (i % C::STAGES) * 8, (i / C::STAGES) & 1);
        }
    } else {
        merge_warp<C, D>(p, ctx, red, sfull, sfree, lane);
    }
}

template <typename T, int D>
cudaError_t launch_split_t(const SplitParams &p, size_t smem, cudaStream_t s)
{
    auto kern = split_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kern<<<p.grid, SplitCfg<T, D>::THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace fd
