// fd_gqa_kernel.cuh -- the grouped-query decode kernel (see fd_gqa.cuh) and
// its launch templates, instantiated per storage type by fd_gqa_bf16.cu and
// fd_gqa_f16.cu (two translation units that compile in parallel).
#pragma once
#include "fd_gqa.cuh"

namespace fd {

// Stage 2 of a (b, virtual head) for its Gv query rows (first row qrow0;
// workspace rows slot * G + g), by the last piece to arrive: the m/l/o merge
// ("FlashDecoding 数学推导" §2.4.2) of the `target` workspace partials of
// each row.  All threads: the pieces' slots and (m, l)
// are staged in shared memory (scr, at least 128 + 130 G floats), the
// weights exp(m_p - M) l_p formed once per (piece, row), then every output
// element sums its pieces with all its loads in flight.  Up to MERGE_PB
// pieces; more go through gqa_merge_pieces_long.
constexpr int MERGE_PB = 64;

template <typename C, int D>
__device__ __forceinline__ void gqa_merge_pieces(const GqaParams &gp, const Ctx &ctx, long long bhv, int slice,
                                                 int G, int Gv, long long qrow0, unsigned target, int gf,
                                                 long long off, int tid, float *scr)
{
    const SplitParams &p = gp.s;
    constexpr int EMAX = (C::MAXG * D + C::THREADS - 1) / C::THREADS;
    const int n = (int)target;
    long long *ss = reinterpret_cast<long long *>(scr);  // [n] workspace slots
    float *sm = scr + 2 * MERGE_PB;                       // [n][G] m, then the weights
    float *sw = sm + MERGE_PB * G;                        // [n][G] l
    float *sM = sw + MERGE_PB * G;                        // [G]
    float *sL = sM + G;                                   // [G]
    for (int i = tid; i < n; i += C::THREADS)
        ss[i] = vh_slot(gp, ctx, bhv, (unsigned)i, gf, off, slice);
    __syncthreads();
    for (int i = tid; i < n * G; i += C::THREADS) {
        if (i % G >= Gv)
            continue;   // rows past this virtual head's query heads were never written
        const long long r = ss[i / G] * G + i % G;
        const float l = __ldcg(p.ws_ml + 2 * r + 1);
        sm[i] = l > 0.f ? __ldcg(p.ws_ml + 2 * r) : -INFINITY;
        sw[i] = l;
    }
    __syncthreads();
    if (tid < Gv) {
        float M = -INFINITY;
        for (int i = 0; i < n; ++i)
            M = fmaxf(M, sm[i * G + tid]);
        float L = 0.f;
        for (int i = 0; i < n; ++i) {
            const float l = sw[i * G + tid];
            const float e = l > 0.f ? ex2(sm[i * G + tid] - M) * l : 0.f;
            sm[i * G + tid] = e;   // the weight replaces m
            L += e;
        }
        sM[tid] = M;
        sL[tid] = L;
    }
    __syncthreads();
    float O[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e)
        O[e] = 0.f;
#pragma unroll 2
    for (int i = 0; i < n; ++i) {
        const long long s0 = ss[i] * G;
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
            const int idx = tid + e * C::THREADS;
            if (idx < Gv * D) {
                const int g = idx / D, dim = idx % D;
                const float w = sm[i * G + g];
                if (w > 0.f)
                    O[e] = fmaf(w, __ldcg(p.ws_o + (s0 + g) * D + dim), O[e]);
            }
        }
    }
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int idx = tid + e * C::THREADS;
        if (idx < Gv * D) {
            const int g = idx / D, dim = idx % D;
            const float L = sL[g];
            const long long qrow = qrow0 + g;
            const bool nonempty = L > 0.f;
            store_out(p.out, qrow * D + dim, p.out_dtype, nonempty ? O[e] / L : 0.f);
            if (dim == 0 && p.lse)
                p.lse[qrow] = nonempty ? (sM[g] + log2f(L)) * LN2_F : -INFINITY;
        }
    }
}

// The same merge for more than MERGE_PB pieces: each thread walks the
// pieces for its output elements.
template <typename C, int D>
__device__ __forceinline__ void gqa_merge_pieces_long(const GqaParams &gp, const Ctx &ctx, long long bhv,
                                                      int slice, int G, int Gv, long long qrow0,
                                                      unsigned target, int gf, long long off, int tid)
{
    const SplitParams &p = gp.s;
    for (int idx = tid; idx < Gv * D; idx += C::THREADS) {
        const int g = idx / D, dim = idx % D;
        float M = -INFINITY;
        for (unsigned i = 0; i < target; ++i) {
            const long long r = vh_slot(gp, ctx, bhv, i, gf, off, slice) * G + g;
            if (__ldcg(p.ws_ml + 2 * r + 1) > 0.f)
                M = fmaxf(M, __ldcg(p.ws_ml + 2 * r));
        }
        float L = 0.f, O = 0.f;
        for (unsigned i = 0; i < target; ++i) {
            const long long r = vh_slot(gp, ctx, bhv, i, gf, off, slice) * G + g;
            const float ll = __ldcg(p.ws_ml + 2 * r + 1);
            if (ll > 0.f) {
                const float e = ex2(__ldcg(p.ws_ml + 2 * r) - M) * ll;
                L += e;
                O = fmaf(e, __ldcg(p.ws_o + r * D + dim), O);
            }
        }
        const long long qrow = qrow0 + g;
        const bool nonempty = L > 0.f;
        store_out(p.out, qrow * D + dim, p.out_dtype, nonempty ? O / L : 0.f);
        if (dim == 0 && p.lse)
            p.lse[qrow] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
    }
}

// NQ: column tiles of 8 query heads (G <= 8: 1; G <= 16: 2).  CTA i works
// on range i / NG of the K/V heads' decomposition for slice i % NG of their
// query heads (see vh_slot).
template <typename T, int D, int NQ, bool P16, bool F8>
__global__ void __launch_bounds__(GqaCfg<T, D, F8>::THREADS, 1) gqa_kernel(const __grid_constant__ GqaParams gp)
{
    using C = GqaCfg<T, D, F8>;
    const SplitParams &p = gp.s;
    const int G = gp.G;            // query heads per slice (row stride of red and the workspace)
    const int slice = (int)(blockIdx.x % gp.NG);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int w = tid >> 5;
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned ring
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::RING_BYTES + C::AREAS);
    float *red = reinterpret_cast<float *>(smem + C::RING_BYTES + C::AREAS + C::BAR_BYTES);  // [WARPS][G][D+2]
    int *flag = reinterpret_cast<int *>(red + C::WARPS * G * (D + 2));
    long long *cumH = reinterpret_cast<long long *>(flag + 4);
    int *lenS = reinterpret_cast<int *>(cumH + p.B + 1);

    // bars: full [GROUPS][STAGES] (the issuer's arrival plus the copies'
    // bytes), then empty [GROUPS][STAGES] (the group's GW warps)
    if (tid == 0) {
        for (int i = 0; i < C::GROUPS * C::STAGES; ++i) {
            mbar_init(smem_addr(&bars[i]), 1);
            mbar_init(smem_addr(&bars[C::GROUPS * C::STAGES + i]), C::GW);
        }
        if constexpr (!C::F8K || C::F8REG) {   // E4M3 at d = 64 comes by 1-D bulk copies, without maps
            prefetch_tmap(&gp.tmk);
            prefetch_tmap(&gp.tmv);
        }
    }

    Ctx ctx;
    ctx.g = (int)(blockIdx.x / gp.NG);   // range
    ctx.G = p.grid / gp.NG;              // ranges
    ctx.cumH = cumH;
    ctx.lenS = lenS;
    ctx.T = 0;
    ctx.Geff = 0;
    ctx.beg = ctx.end = 0;
    if (p.decomp == DECOMP_BALANCED) {
        balanced_setup<C::THREADS, C::WARPS>(p, ctx, cumH, lenS);
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
    __syncthreads();

    {
        const int grp_id = w / C::GW;
        const int gw = w % C::GW;
        const bool issuer = (gw == 0);   // the group's first warp also issues its copies
        const uint32_t ring_base = smem_addr(smem) + (uint32_t)(grp_id * C::STAGES * C::STAGE_BYTES);
        const uint32_t bar_base = smem_addr(&bars[grp_id * C::STAGES]);
        const uint32_t ebar_base = smem_addr(&bars[(C::GROUPS + grp_id) * C::STAGES]);
        const int row0 = gw * C::WT;  // this warp's first row in a stage
        // F8: this warp's f16 area (K rows, then V rows)
        const uint32_t area = smem_addr(smem) + (uint32_t)(C::RING_BYTES + w * C::AREA_BYTES);

        TmaProducer<C, P16> prod;
        int issued = 0, landed = 0;
        bool dead = false;
        if (issuer) {
            prod.start(gp, ctx, grp_id, C::GROUPS);
#pragma unroll 1
            for (int s = 0; s < C::STAGES; ++s) {
                if (!prod.issue(gp, ctx, ring_base + s * C::STAGE_BYTES, bar_base + s * 8, lane))
                    break;
                ++issued;
            }
        }

        const int qn = lane >> 2;          // B fragments: head 8j + lane/4, dims 2(lane%4) (+1, +8, +9)
        const int qk = 2 * (lane & 3);
        Seg cs;
        seg_first(p, ctx, cs);
        long long cbase = 0;
        int consumed = 0;
#pragma unroll 1
        while (cs.valid) {
            const long long nc = seg_chunks<C::CT>(cs);
            const int vh = cs.h * gp.NG + slice;            // virtual head
            const long long bhv = (long long)cs.b * p.H * gp.NG + vh;   // its counter
            const int gv = vh_count(gp, vh);                 // its query heads
            const long long qrow0 = vh_qrow0(gp, cs.b, vh);
            // score scale of the segment (E4M3 K: times its dequantisation
            // scale) and V's scale, applied to the output at the segment end
            float seg_scale = p.scale_log2;
            float vsc = 1.f;
            if constexpr (C::F8K) {
                seg_scale *= __ldg(gp.k_scale + cs.b * p.H + cs.h);
                vsc = __ldg(gp.v_scale + cs.b * p.H + cs.h);
            }
            // Q^T of the head group as mma B fragments (heads >= gv are zero)
            uint32_t qb[NQ][C::KSTEPS][2];
            // E4M3: each head's base-2 score scale, with the power of two that
            // brought its q into the f16 range (q_range_exp)
            HeadScale<NQ> hsc;
            {
                const uint32_t *q32 = static_cast<const uint32_t *>(p.q);
                const long long qbase = qrow0 * D;  // elements
#pragma unroll
                for (int j = 0; j < NQ; ++j) {
                    const int n = 8 * j + qn;
                    if constexpr (C::F8K) {   // q of any dtype, as f16 pairs
                        float2 qf[C::KSTEPS][2];
                        float amax = 0.f;
#pragma unroll
                        for (int s = 0; s < C::KSTEPS; ++s) {
                            // F8REG: d permuted as K's fragments (f8_k_frag)
                            const long long e0 = qbase + (long long)n * D + 16 * s + (C::F8REG ? 4 * (lane & 3) : qk);
                            const long long e1 = e0 + (C::F8REG ? 2 : 8);
                            qf[s][0] = n < gv ? q_pair_f32(p.q, p.q_dtype, e0) : make_float2(0.f, 0.f);
                            qf[s][1] = n < gv ? q_pair_f32(p.q, p.q_dtype, e1) : make_float2(0.f, 0.f);
                            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(qf[s][0].x), fabsf(qf[s][0].y)),
                                                     fmaxf(fabsf(qf[s][1].x), fabsf(qf[s][1].y))));
                        }
                        // the head's 4 lanes (same lane / 4) hold all its d values
                        amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, 1));
                        amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, 2));
                        const int ex = q_range_exp(amax);
                        const float down = 1.f / pow2i(ex);   // exact: a power of two
#pragma unroll
                        for (int s = 0; s < C::KSTEPS; ++s) {
                            qb[j][s][0] = f16_pair(qf[s][0].x * down, qf[s][0].y * down);
                            qb[j][s][1] = f16_pair(qf[s][1].x * down, qf[s][1].y * down);
                        }
                        // the accumulator's head columns 2(lane%4) + e of this
                        // tile belong to lanes 4 (2(lane%4) + e)
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            hsc.s[j][e] = seg_scale * pow2i(__shfl_sync(FULL_MASK, ex, 4 * (2 * (lane & 3) + e)));
                    } else {
#pragma unroll
                        for (int s = 0; s < C::KSTEPS; ++s) {
                            const long long e = qbase + (long long)n * D + 16 * s + qk;
                            qb[j][s][0] = n < gv ? __ldg(q32 + e / 2) : 0u;
                            qb[j][s][1] = n < gv ? __ldg(q32 + (e + 8) / 2) : 0u;
                        }
                    }
                }
            }
            GqaState<C, NQ> st;
#pragma unroll
            for (int i = 0; i < C::MT; ++i)
#pragma unroll
                for (int j = 0; j < NQ; ++j)
                    st.o[i][j][0] = st.o[i][j][1] = st.o[i][j][2] = st.o[i][j][3] = 0.f;
#pragma unroll
            for (int j = 0; j < NQ; ++j) {
                st.m[j][0] = st.m[j][1] = -INFINITY;
                st.l[j][0] = st.l[j][1] = 0.f;
            }

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
                // stage row of the chunk's first token: 0, or with 16-token
                // pages its place in the aligned block
                const int lead = P16 ? (t & (C::CT - 1)) : 0;
                const int vlo = max(lead - row0, 0);                   // this warp's valid
                const int vhi = min(lead + ntok_chunk - row0, C::WT);  // rows [vlo, vhi)
                const uint32_t kb = ring_base + stage * C::STAGE_BYTES;
                if constexpr (C::F8REG) {
                    // V's rows into the area, K's as raw fragments; free the
                    // stage (the issuer refills it), then compute
                    const bool work = !dead && vhi > vlo;
                    uint32_t kraw[C::KSTEPS / 2][4];
                    if (work) {
                        f8_rows_to_area<C>(kb + C::CHUNK_BYTES, row0, area, vlo, vhi, lane);
                        f8_k_raw<C>(kb, row0, lane, kraw);
                    }
                    __syncwarp();
                    if (!dead && lane == 0)
                        mbar_arrive(ebar_base + stage * 8);
                    if (issuer && !dead && !mbar_wait_bounded(ebar_base + stage * 8, parity))
                        dead = true;
                    if (issuer && !dead && prod.issue(gp, ctx, kb, bar_base + stage * 8, lane))
                        ++issued;
                    if (work)
                        gqa_chunk_kf<T, C, NQ, true>(
                            [&](int s, uint32_t (&a)[4]) { f8_k_frag(&kraw[s >> 1][2 * (s & 1)], a); }, area, 0,
                            vlo, vhi, qb, hsc, lane, st);
                    __syncwarp();   // the area is rewritten by the next chunk
                    continue;
                } else if constexpr (C::F8K) {
                    // convert the warp's rows into its area, free the stage
                    // (the issuer refills it), then compute from the area
                    const bool work = !dead && vhi > vlo;
                    if (work) {
                        f8_rows_to_area<C>(kb, row0, area, vlo, vhi, lane);
                        f8_rows_to_area<C>(kb + C::CHUNK_BYTES, row0, area + C::AREA_BYTES / 2, vlo, vhi, lane);
                    }
                    __syncwarp();
                    if (!dead && lane == 0)
                        mbar_arrive(ebar_base + stage * 8);
                    if (issuer && !dead && !mbar_wait_bounded(ebar_base + stage * 8, parity))
                        dead = true;
                    if (issuer && !dead && prod.issue(gp, ctx, kb, bar_base + stage * 8, lane))
                        ++issued;
                    if (work)
                        gqa_chunk<T, C, NQ, true>(area, area + C::AREA_BYTES / 2, 0, vlo, vhi, qb, hsc, lane,
                                                  st);
                    __syncwarp();   // the area is rewritten by the next chunk
                    continue;
                }
                if (!dead && vhi > vlo) {
                    if (vlo > 0 || vhi < C::WT) {
                        // rows outside the chunk's tokens may hold padding or other
                        // rows: zero them in every plane of V (a row is 128
                        // contiguous bytes of a plane)
#pragma unroll
                        for (int j = 0; j < C::LINES; ++j) {
                            const uint32_t z0 = kb + C::CHUNK_BYTES + stage_row<C, P16>(row0, j);
#pragma unroll
                            for (int off = lane * 16; off < C::WT * 128; off += 32 * 16) {
                                const int rr = off >> 7;
                                if (rr < vlo || rr >= vhi)
                                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(z0 + off),
                                                 "r"(0u)
                                                 : "memory");
                            }
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                    }
                    gqa_chunk<T, C, NQ, P16>(kb, kb + C::CHUNK_BYTES, row0, vlo, vhi, qb, UniformScale{seg_scale},
                                             lane, st);
                }
                __syncwarp();
                // release the stage; the issuer refills it once both warps have
                if (!dead && lane == 0)
                    mbar_arrive(ebar_base + stage * 8);
                if (issuer && !dead && !mbar_wait_bounded(ebar_base + stage * 8, parity))
                    dead = true;
                if (issuer && !dead && prod.issue(gp, ctx, kb, bar_base + stage * 8, lane))
                    ++issued;
            }

            // ---- segment end: full sums per head, then merge the warps per head ----
            {
                float *rw = red + w * G * (D + 2);
#pragma unroll
                for (int j = 0; j < NQ; ++j) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float l = st.l[j][e];
                        l += __shfl_xor_sync(FULL_MASK, l, 4);
                        l += __shfl_xor_sync(FULL_MASK, l, 8);
                        l += __shfl_xor_sync(FULL_MASK, l, 16);
                        const int g = 8 * j + qk + e;   // this thread's head
                        if (g < gv) {
                            float *rg = rw + g * (D + 2);
#pragma unroll
                            for (int i = 0; i < C::MT; ++i) {
                                rg[16 * i + qn] = st.o[i][j][e] * vsc;
                                rg[16 * i + qn + 8] = st.o[i][j][e + 2] * vsc;
                            }
                            if (qn == 0) {
                                rg[D] = st.m[j][e];
                                rg[D + 1] = l;
                            }
                        }
                    }
                }
            }
            __syncthreads();

            const int len = (p.decomp == DECOMP_BALANCED) ? lenS[cs.b] : clamp_len(p, cs.b);
            bool complete;
            long long slot;
            if (p.decomp == DECOMP_SPLITS) {
                complete = (p.P == 1);
                slot = bhv * p.P + cs.p;
            } else {
                complete = seg_whole(p, cs, len);
                slot = 2LL * blockIdx.x + (cs.k == 0 ? 0 : 1);
            }
            // warp w merges heads w, w + WARPS, ...: the head's max, weights and
            // sum once per lane, then its dims lane, lane + 32, ...
            for (int g = w; g < gv; g += C::WARPS) {
                float M = -INFINITY;
#pragma unroll
                for (int i = 0; i < C::WARPS; ++i) {
                    const float *ri = red + (i * G + g) * (D + 2);
                    if (ri[D + 1] > 0.f)
                        M = fmaxf(M, ri[D]);
                }
                float L = 0.f, e[C::WARPS];
#pragma unroll
                for (int i = 0; i < C::WARPS; ++i) {
                    const float *ri = red + (i * G + g) * (D + 2);
                    e[i] = ri[D + 1] > 0.f ? ex2(ri[D] - M) : 0.f;
                    L = fmaf(e[i], ri[D + 1], L);
                }
                const bool nonempty = L > 0.f;
                const long long qrow = qrow0 + g;
                const long long r = slot * G + g;
#pragma unroll
                for (int dd = 0; dd < D / 32; ++dd) {
                    const int dim = lane + 32 * dd;
                    float O = 0.f;
#pragma unroll
                    for (int i = 0; i < C::WARPS; ++i)
                        O = fmaf(e[i], red[(i * G + g) * (D + 2) + dim], O);
                    const float o = nonempty ? O / L : 0.f;
                    if (complete)
                        store_out(p.out, qrow * D + dim, p.out_dtype, o);
                    else
                        p.ws_o[r * D + dim] = o;
                }
                if (lane == 0) {
                    if (complete) {
                        if (p.lse)
                            p.lse[qrow] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
                    } else {
                        p.ws_ml[2 * r] = nonempty ? M : -INFINITY;
                        p.ws_ml[2 * r + 1] = L;
                    }
                }
            }

            if (!complete) {
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
                // the barrier orders every thread's partial before thread 0's
                // fence and arrival
                __syncthreads();
                if (tid == 0) {
                    __threadfence();
                    const unsigned old = atomicInc(p.ws_cnt + bhv, target - 1);
                    *flag = (old == target - 1);
                }
                __syncthreads();
                if (*flag) {
                    __threadfence();
                    // red is free again: every thread has passed its reads
                    if (target <= (unsigned)MERGE_PB)
                        gqa_merge_pieces<C, D>(gp, ctx, bhv, slice, G, gv, qrow0, target, gf, off, tid, red);
                    else
                        gqa_merge_pieces_long<C, D>(gp, ctx, bhv, slice, G, gv, qrow0, target, gf, off, tid);
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
}

template <typename T, int D, int NQ, bool P16, bool F8 = false>
static cudaError_t launch_gqa_p(const GqaParams &gp, cudaStream_t s)
{
    using C = GqaCfg<T, D, F8>;
    const size_t smem = C::smem_bytes(gp.s.decomp, gp.s.B, gp.G);
    auto kern = gqa_kernel<T, D, NQ, P16, F8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kern<<<gp.s.grid, C::THREADS, smem, s>>>(gp);
    return cudaGetLastError();
}

template <typename T, int D, int NQ>
static cudaError_t launch_gqa_t(const GqaParams &gp, cudaStream_t s)
{
    return gp.pages16 ? launch_gqa_p<T, D, NQ, true>(gp, s) : launch_gqa_p<T, D, NQ, false>(gp, s);
}

template <typename T, int D>
static cudaError_t launch_gqa_d(const GqaParams &gp, cudaStream_t s)
{
    if constexpr (D == 256)
        return launch_gqa_t<T, D, 1>(gp, s);   // G <= 8
    else
        return gp.G <= 8 ? launch_gqa_t<T, D, 1>(gp, s) : launch_gqa_t<T, D, 2>(gp, s);
}

template <typename T> static cudaError_t launch_gqa_dt(int d, const GqaParams &gp, cudaStream_t s)
{
    if (d == 64)
        return launch_gqa_d<T, 64>(gp, s);
    if (d == 128)
        return launch_gqa_d<T, 128>(gp, s);
    return launch_gqa_d<T, 256>(gp, s);
}

}  // namespace fd
