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
// CTA every warp owns a private ring of STAGES shared-memory stages; a stage
// holds one chunk of CT tokens of K and the same tokens of V, filled by two
// 1-D bulk copies (cp.async.bulk, completion on an mbarrier).  Chunks of the
// CTA's token sequence go round-robin to the warps, so the CTA streams
// contiguous memory while warps never wait on each other inside a segment.
// Within a warp, LPT lanes cover one token row with 16-byte loads and the
// q.k partial sums are reduced with xor-shuffles.  The softmax state is
// updated once per chunk in the block form of the online-softmax update
// (running max, rescale by exp(m_old - m_new), unnormalised accumulator),
// with scores in base 2 (q pre-multiplied by scale*log2(e)) so that the
// exponentials are single ex2 instructions.  At a segment end the warps'
// states are merged through shared memory (the m/l/o merge).
#pragma once

#include "fd_device.cuh"
#include "fd_internal.h"

namespace fd {

constexpr float LN2_F = 0.693147180559945309f;

template <typename T, int D> struct SplitCfg {
    static constexpr int ESZ = sizeof(T);
    static constexpr int VEC = Elem<T>::VEC;       // elements per lane vector (16 bytes)
    static constexpr int LPT = D / VEC;            // lanes per token row
    static constexpr int TPW = 32 / LPT;           // token rows per warp-wide load
    static constexpr int ROW = D * ESZ;            // bytes per token row
    static constexpr int WARPS = 8;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int STAGES = 3;
    static constexpr int CT = 4096 / ROW;          // tokens per chunk
    static constexpr int TOK = CT / TPW;           // tokens per lane group per chunk
    static constexpr int CHUNK_BYTES = CT * ROW;   // one of K or V
    static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;
    static constexpr int RING_BYTES = WARPS * STAGES * STAGE_BYTES;
    static constexpr int BAR_BYTES = WARPS * STAGES * 8;
    static constexpr int RED_BYTES = (2 * WARPS + WARPS * D) * 4 + 16;
    static_assert(LPT >= 1 && LPT <= 32 && 32 % LPT == 0, "row must map onto whole lanes");
    static_assert(CT % TPW == 0 && TOK >= 1, "chunk must cover whole warp steps");
    static_assert(D <= THREADS, "one thread per output element in the merge");

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
    bool valid;
};

// Per-CTA view of the decomposition.
struct Ctx {
    int g;            // this CTA
    int G;            // CTAs launched
    int Geff;         // CTAs with work (balanced: min(G, T))
    long long T;      // total tokens over all (b, h) (balanced)
    long long beg, end;  // this CTA's range in the concatenated space
    const long long *cumH;  // [B+1] H * prefix sum of lengths (balanced)
    const int *lenS;        // [B] clamped lengths (balanced)
};

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
    const int len = c.lenS[s.b];
    const long long rel = s.pos - c.cumH[s.b];
    s.h = (int)(rel / len);
    s.t0 = (int)(rel % len);
    const long long room = c.end - s.pos;
    s.t1 = (long long)(len - s.t0) < room ? len : (int)(s.t0 + room);
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
    s.pos += s.t1 - s.t0;
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
    const int len = c.lenS[s.b];
    s.t0 = 0;
    const long long room = c.end - s.pos;
    s.t1 = (long long)len < room ? len : (int)room;
}

template <int CT> __device__ __forceinline__ long long seg_chunks(const Seg &s)
{
    return ((long long)(s.t1 - s.t0) + CT - 1) / CT;
}

// Producer side of a warp's ring: walks the warp's chunks (c = w, w+W, ...)
// of the CTA's chunk sequence and issues the bulk copies for the next one.
template <typename C> struct Producer {
    Seg s;
    long long base;   // chunk index of s's first chunk
    long long c;      // next chunk to issue

    __device__ __forceinline__ bool issue(const SplitParams &p, const Ctx &ctx, uint32_t kdst,
                                          uint32_t bar, int lane)
    {
        while (s.valid && c >= base + seg_chunks<C::CT>(s)) {
            base += seg_chunks<C::CT>(s);
            seg_next(p, ctx, s);
        }
        if (!s.valid)
            return false;
        const int t = s.t0 + (int)((c - base) * C::CT);
        const int ntok = min(C::CT, s.t1 - t);
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)ntok * C::ROW;
            const long long row = ((long long)s.b * p.H + s.h) * p.N + t;
            const char *ksrc = static_cast<const char *>(p.k) + row * C::ROW;
            const char *vsrc = static_cast<const char *>(p.v) + row * C::ROW;
            mbar_arrive_expect_tx(bar, 2 * bytes);
            bulk_g2s(kdst, ksrc, bytes, bar);
            bulk_g2s(kdst + C::CHUNK_BYTES, vsrc, bytes, bar);
        }
        c += C::WARPS;
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

// One chunk of the warp's ring: block-wise online-softmax update of the lane
// group's state with its TOK token rows.
template <typename T, int D, bool FULL>
__device__ __forceinline__ void process_chunk(uint32_t kbase, int ntok, int grp, int col,
                                              const float *qf, float &m, float &l, float *acc)
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
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int i = 0; i < C::VEC; i += 2) {
                d0 = fmaf(qf[i], kf[i], d0);
                d1 = fmaf(qf[i + 1], kf[i + 1], d1);
            }
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
    const uint32_t vbase = kbase + C::CHUNK_BYTES;
#pragma unroll
    for (int t = 0; t < C::TOK; ++t) {
        const int row = t * C::TPW + grp;
        if (FULL || row < ntok) {
            const float pj = ex2(s[t] - mnew);
            l += pj;
            const uint4 u = lds128(vbase + row * C::ROW + col * 16);
            float vf[C::VEC];
            Elem<T>::widen(u, vf);
#pragma unroll
            for (int i = 0; i < C::VEC; ++i)
                acc[i] = fmaf(pj, vf[i], acc[i]);
        }
    }
    m = mnew;
}

template <typename T, int D>
__global__ void __launch_bounds__(SplitCfg<T, D>::THREADS, 1) split_kernel(const SplitParams p)
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
    float *red_m = reinterpret_cast<float *>(smem + C::RING_BYTES + C::BAR_BYTES);
    float *red_l = red_m + C::WARPS;
    float *red_acc = red_l + C::WARPS;
    int *flag = reinterpret_cast<int *>(red_acc + C::WARPS * D);
    long long *cumH = reinterpret_cast<long long *>(smem + C::RING_BYTES + C::BAR_BYTES + C::RED_BYTES);
    int *lenS = reinterpret_cast<int *>(cumH + p.B + 1);

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < C::STAGES; ++s)
            mbar_init(smem_addr(&bars[w * C::STAGES + s]), 1);
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
        // clamped lengths and H * exclusive prefix sums, by a block scan
        constexpr int PER = (BALANCED_MAX_B + C::THREADS - 1) / C::THREADS;
        long long v[PER];
        long long run = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int b = tid * PER + i;
            long long x = 0;
            if (b < p.B) {
                const int n = clamp_len(p, b);
                lenS[b] = n;
                x = (long long)n * p.H;
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
        __shared__ long long warp_tot[C::WARPS];
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
        if (tid == C::THREADS - 1)
            cumH[p.B] = excl + run;
        __syncthreads();
        ctx.T = cumH[p.B];
        ctx.Geff = (int)(ctx.T < (long long)ctx.G ? ctx.T : (long long)ctx.G);
        if (ctx.g < ctx.Geff) {
            ctx.beg = bal_bound(ctx.g, ctx.T, ctx.Geff);
            ctx.end = bal_bound(ctx.g + 1, ctx.T, ctx.Geff);
        }
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
    __syncthreads();

    const uint32_t ring_base = smem_addr(ring) + (uint32_t)(w * C::STAGES * C::STAGE_BYTES);
    const uint32_t bar_base = smem_addr(&bars[w * C::STAGES]);

    Producer<C> prod;
    seg_first(p, ctx, prod.s);
    prod.base = 0;
    prod.c = w;
    int issued = 0;   // chunks issued by this warp
    int landed = 0;   // chunks whose copies this warp has seen complete
    bool dead = false;
#pragma unroll 1
    for (int s = 0; s < C::STAGES; ++s) {
        if (!prod.issue(p, ctx, ring_base + s * C::STAGE_BYTES, bar_base + s * 8, lane))
            break;
        ++issued;
    }

    Seg cs;
    seg_first(p, ctx, cs);
    long long cbase = 0;
    int consumed = 0;
#pragma unroll 1
    while (cs.valid) {
        const long long nc = seg_chunks<C::CT>(cs);
        const int bh = cs.b * p.H + cs.h;
        float qf[C::VEC];
        {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(
                static_cast<const char *>(p.q) + ((long long)bh * D) * C::ESZ + col * 16));
            Elem<T>::widen(u, qf);
#pragma unroll
            for (int i = 0; i < C::VEC; ++i)
                qf[i] *= p.scale_log2;
        }
        float m = -INFINITY, l = 0.f, acc[C::VEC];
#pragma unroll
        for (int i = 0; i < C::VEC; ++i)
            acc[i] = 0.f;

        long long c = cbase + ((w - cbase % C::WARPS) % C::WARPS + C::WARPS) % C::WARPS;
#pragma unroll 1
        for (; c < cbase + nc; c += C::WARPS) {
            const int stage = consumed % C::STAGES;
            const uint32_t parity = (consumed / C::STAGES) & 1;
            ++consumed;
            if (!dead) {
                if (mbar_wait_bounded(bar_base + stage * 8, parity))
                    ++landed;
                else
                    dead = true;
            }
            const int t = cs.t0 + (int)((c - cbase) * C::CT);
            const int ntok = min(C::CT, cs.t1 - t);
            const uint32_t kb = ring_base + stage * C::STAGE_BYTES;
            if (!dead) {
                if (ntok == C::CT)
                    process_chunk<T, D, true>(kb, ntok, grp, col, qf, m, l, acc);
                else
                    process_chunk<T, D, false>(kb, ntok, grp, col, qf, m, l, acc);
            }
            __syncwarp();
            if (!dead && prod.issue(p, ctx, kb, bar_base + stage * 8, lane))
                ++issued;
        }

        // ---- segment end: merge lane groups, then warps ----
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
        if (grp == 0) {
#pragma unroll
            for (int i = 0; i < C::VEC; ++i)
                red_acc[w * D + col * C::VEC + i] = acc[i];
            if (col == 0) {
                red_m[w] = m;
                red_l[w] = l;
            }
        }
        __syncthreads();

        const int len = (p.decomp == DECOMP_BALANCED) ? lenS[cs.b] : clamp_len(p, cs.b);
        bool complete;
        long long slot = 0;
        if (p.decomp == DECOMP_SPLITS) {
            complete = (p.P == 1);
            slot = (long long)bh * p.P + cs.p;
        } else {
            complete = (cs.t0 == 0 && cs.t1 == len);
            slot = 2LL * ctx.g + (cs.k == 0 ? 0 : 1);
        }

        if (tid < D) {
            float M = -INFINITY;
#pragma unroll
            for (int i = 0; i < C::WARPS; ++i)
                if (red_l[i] > 0.f)
                    M = fmaxf(M, red_m[i]);
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int i = 0; i < C::WARPS; ++i) {
                if (red_l[i] > 0.f) {
                    const float e = ex2(red_m[i] - M);
                    L = fmaf(e, red_l[i], L);
                    O = fmaf(e, red_acc[i * D + tid], O);
                }
            }
            const bool nonempty = L > 0.f;
            const float o = nonempty ? O / L : 0.f;
            if (p.out_kind == OUT_PARTIALS) {
                p.o_part[slot * D + tid] = o;
                if (tid == 0) {
                    p.m_part[slot] = nonempty ? M * LN2_F : -INFINITY;
                    p.l_part[slot] = L;
                    if (p.lse_part)
                        p.lse_part[slot] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
                }
            } else if (complete) {
                store_out(p.out, (long long)bh * D + tid, p.out_dtype, o);
                if (tid == 0 && p.lse)
                    p.lse[bh] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
            } else {
                // workspace partial: normalised o, m in base 2, l
                p.ws_o[slot * D + tid] = o;
                if (tid == 0) {
                    p.ws_ml[2 * slot] = nonempty ? M : -INFINITY;
                    p.ws_ml[2 * slot + 1] = L;
                }
            }
        }

        if (p.out_kind == OUT_FUSED && !complete) {
            // last piece of this (b, h) to arrive merges all of them
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
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                const unsigned old = atomicInc(p.ws_cnt + bh, target - 1);
                *flag = (old == target - 1);
            }
            __syncthreads();
            if (*flag) {
                __threadfence();
                if (tid < D) {
                    float M = -INFINITY;
                    for (unsigned i = 0; i < target; ++i) {
                        long long sl;
                        if (p.decomp == DECOMP_SPLITS) {
                            sl = (long long)bh * p.P + i;
                        } else {
                            const long long g = gf + (long long)i;
                            sl = (i == 0 && bal_bound(gf, ctx.T, ctx.Geff) != off) ? 2 * g + 1 : 2 * g;
                        }
                        const float ml = __ldcg(p.ws_ml + 2 * sl);
                        const float ll = __ldcg(p.ws_ml + 2 * sl + 1);
                        if (ll > 0.f)
                            M = fmaxf(M, ml);
                    }
                    float L = 0.f, O = 0.f;
                    for (unsigned i = 0; i < target; ++i) {
                        long long sl;
                        if (p.decomp == DECOMP_SPLITS) {
                            sl = (long long)bh * p.P + i;
                        } else {
                            const long long g = gf + (long long)i;
                            sl = (i == 0 && bal_bound(gf, ctx.T, ctx.Geff) != off) ? 2 * g + 1 : 2 * g;
                        }
                        const float ll = __ldcg(p.ws_ml + 2 * sl + 1);
                        if (ll > 0.f) {
                            const float e = ex2(__ldcg(p.ws_ml + 2 * sl) - M) * ll;
                            L += e;
                            O = fmaf(e, __ldcg(p.ws_o + sl * D + tid), O);
                        }
                    }
                    const bool nonempty = L > 0.f;
                    store_out(p.out, (long long)bh * D + tid, p.out_dtype, nonempty ? O / L : 0.f);
                    if (tid == 0 && p.lse)
                        p.lse[bh] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
                }
            }
        }
        __syncthreads();

        cbase += nc;
        seg_next(p, ctx, cs);
    }

    if (dead) {
        if (lane == 0)
            atomicOr(p.status, STATUS_TIMEOUT);
        // wait (bounded) for this warp's copies still in flight
        for (int i = landed; i < issued; ++i)
            mbar_wait_bounded(bar_base + (i % C::STAGES) * 8, (i / C::STAGES) & 1);
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
