// fd_gqa.cu -- the grouped-query decode kernel (see fd_gqa.cuh) and its
// launcher.
#include "fd_gqa.cuh"

namespace fd {

// Stage 2 of a (b, kv head) for its G query rows, by the last piece to
// arrive: the m/l/o merge ("FlashDecoding 数学推导" §2.4.2) of the `target`
// workspace partials of each row.
template <typename C, int D>
__device__ __forceinline__ void gqa_merge_pieces(const SplitParams &p, const Ctx &ctx, int bh, int G,
                                                 unsigned target, int gf, long long off, int tid)
{
    const int Hq = p.H * G;
    const int b = bh / p.H, hk = bh % p.H;
    for (int idx = tid; idx < G * D; idx += C::THREADS) {
        const int g = idx / D, dim = idx % D;
        float M = -INFINITY;
        for (unsigned i = 0; i < target; ++i) {
            const long long r = piece_slot(p, ctx, bh, i, gf, off) * G + g;
            if (__ldcg(p.ws_ml + 2 * r + 1) > 0.f)
                M = fmaxf(M, __ldcg(p.ws_ml + 2 * r));
        }
        float L = 0.f, O = 0.f;
        for (unsigned i = 0; i < target; ++i) {
            const long long r = piece_slot(p, ctx, bh, i, gf, off) * G + g;
            const float ll = __ldcg(p.ws_ml + 2 * r + 1);
            if (ll > 0.f) {
                const float e = ex2(__ldcg(p.ws_ml + 2 * r) - M) * ll;
                L += e;
                O = fmaf(e, __ldcg(p.ws_o + r * D + dim), O);
            }
        }
        const long long qrow = (long long)b * Hq + (long long)hk * G + g;
        const bool nonempty = L > 0.f;
        store_out(p.out, qrow * D + dim, p.out_dtype, nonempty ? O / L : 0.f);
        if (dim == 0 && p.lse)
            p.lse[qrow] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(GqaCfg<T, D>::THREADS, 1) gqa_kernel(const __grid_constant__ GqaParams gp)
{
    using C = GqaCfg<T, D>;
    const SplitParams &p = gp.s;
    const int G = gp.G;
    const int Hq = p.H * G;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int w = tid >> 5;
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned ring
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::RING_BYTES);
    float *red = reinterpret_cast<float *>(smem + C::RING_BYTES + C::BAR_BYTES);  // [WARPS][G][D+2]
    int *flag = reinterpret_cast<int *>(red + C::WARPS * G * (D + 2));
    long long *cumH = reinterpret_cast<long long *>(flag + 4);
    int *lenS = reinterpret_cast<int *>(cumH + p.B + 1);

    const int grp_id = w / C::GW;
    const int gw = w % C::GW;
    const bool issuer = (gw == 0);
    if (issuer && lane == 0) {
#pragma unroll
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_addr(&bars[grp_id * C::STAGES + s]), 1);
            mbar_init(smem_addr(&bars[(C::GROUPS + grp_id) * C::STAGES + s]), C::GW);
        }
    }
    if (tid == 0) {
        prefetch_tmap(&gp.tmk);
        prefetch_tmap(&gp.tmv);
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
        balanced_setup<C::THREADS, C::WARPS>(p, ctx, cumH, lenS);
        // (b, kv head) of length 0 are touched by no CTA: write their G rows here
        for (long long bh = (long long)ctx.g * C::THREADS + tid; bh < (long long)p.B * p.H;
             bh += (long long)ctx.G * C::THREADS) {
            if (lenS[bh / p.H] == 0) {
                const long long q0 = (bh / p.H) * Hq + (bh % p.H) * G;
                for (int g = 0; g < G; ++g) {
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

    const uint32_t ring_base = smem_addr(smem) + (uint32_t)(grp_id * C::STAGES * C::STAGE_BYTES);
    const uint32_t bar_base = smem_addr(&bars[grp_id * C::STAGES]);
    const uint32_t ebar_base = smem_addr(&bars[(C::GROUPS + grp_id) * C::STAGES]);
    const int row0 = gw * C::WT;  // this warp's first row in a stage

    TmaProducer<C> prod;
    int issued = 0, landed = 0;
    bool dead = false;
    if (issuer) {
        prod.start(p, ctx, grp_id);
#pragma unroll 1
        for (int s = 0; s < C::STAGES; ++s) {
            if (!prod.issue(gp, ctx, ring_base + s * C::STAGE_BYTES, bar_base + s * 8, lane))
                break;
            ++issued;
        }
    }

    const int r0 = lane >> 2;         // this thread's rows r0, r0 + 8
    const int cb = 2 * (lane & 3);    // and columns cb, cb + 1 of each tile
    Seg cs;
    seg_first(p, ctx, cs);
    long long cbase = 0;
    int consumed = 0;
#pragma unroll 1
    while (cs.valid) {
        const long long nc = seg_chunks<C::CT>(cs);
        const int bh = cs.b * p.H + cs.h;
        // Q of the head group as mma A fragments (rows >= G are zero)
        uint32_t qa[C::KSTEPS][4];
        {
            const uint32_t *q32 = static_cast<const uint32_t *>(p.q);
            const long long qbase = ((long long)cs.b * Hq + (long long)cs.h * G) * D;  // elements
#pragma unroll
            for (int s = 0; s < C::KSTEPS; ++s) {
                const int col = 16 * s + cb;
                qa[s][0] = r0 < G ? __ldg(q32 + (qbase + r0 * D + col) / 2) : 0u;
                qa[s][1] = r0 + 8 < G ? __ldg(q32 + (qbase + (r0 + 8) * D + col) / 2) : 0u;
                qa[s][2] = r0 < G ? __ldg(q32 + (qbase + r0 * D + col + 8) / 2) : 0u;
                qa[s][3] = r0 + 8 < G ? __ldg(q32 + (qbase + (r0 + 8) * D + col + 8) / 2) : 0u;
            }
        }
        GqaState<C> st;
#pragma unroll
        for (int n = 0; n < C::NT; ++n)
            st.o[n][0] = st.o[n][1] = st.o[n][2] = st.o[n][3] = 0.f;
        st.m0 = st.m1 = -INFINITY;
        st.l0 = st.l1 = 0.f;

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
            const int nv = ntok_chunk - row0;  // this warp's valid rows
            const uint32_t kb = ring_base + stage * C::STAGE_BYTES;
            if (!dead && nv > 0) {
                if (nv < C::WT) {
                    // rows past the last token may hold padding: zero them in V
                    const uint32_t z0 = kb + C::CHUNK_BYTES + (uint32_t)(row0 + nv) * C::ROW;
                    const int nbytes = (C::WT - nv) * C::ROW;
                    for (int off = lane * 16; off < nbytes; off += 32 * 16)
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(z0 + off), "r"(0u)
                                     : "memory");
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                }
                gqa_chunk<T, C>(kb, kb + C::CHUNK_BYTES, row0, nv, qa, p.scale_log2, lane, st);
            }
            __syncwarp();
            if (!dead && lane == 0)
                mbar_arrive(ebar_base + stage * 8);
            if (issuer && !dead && !mbar_wait_bounded(ebar_base + stage * 8, parity))
                dead = true;
            if (issuer && !dead && prod.issue(gp, ctx, kb, bar_base + stage * 8, lane))
                ++issued;
        }

        // ---- segment end: full row sums, then merge the warps per row ----
        st.l0 += __shfl_xor_sync(FULL_MASK, st.l0, 1);
        st.l0 += __shfl_xor_sync(FULL_MASK, st.l0, 2);
        st.l1 += __shfl_xor_sync(FULL_MASK, st.l1, 1);
        st.l1 += __shfl_xor_sync(FULL_MASK, st.l1, 2);
        {
            float *rw = red + w * G * (D + 2);
            if (r0 < G) {
#pragma unroll
                for (int n = 0; n < C::NT; ++n) {
                    rw[r0 * (D + 2) + 8 * n + cb] = st.o[n][0];
                    rw[r0 * (D + 2) + 8 * n + cb + 1] = st.o[n][1];
                }
                if ((lane & 3) == 0) {
                    rw[r0 * (D + 2) + D] = st.m0;
                    rw[r0 * (D + 2) + D + 1] = st.l0;
                }
            }
            if (r0 + 8 < G) {
#pragma unroll
                for (int n = 0; n < C::NT; ++n) {
                    rw[(r0 + 8) * (D + 2) + 8 * n + cb] = st.o[n][2];
                    rw[(r0 + 8) * (D + 2) + 8 * n + cb + 1] = st.o[n][3];
                }
                if ((lane & 3) == 0) {
                    rw[(r0 + 8) * (D + 2) + D] = st.m1;
                    rw[(r0 + 8) * (D + 2) + D + 1] = st.l1;
                }
            }
        }
        __syncthreads();

        const int len = (p.decomp == DECOMP_BALANCED) ? lenS[cs.b] : clamp_len(p, cs.b);
        bool complete;
        long long slot;
        if (p.decomp == DECOMP_SPLITS) {
            complete = (p.P == 1);
            slot = (long long)bh * p.P + cs.p;
        } else {
            complete = (cs.t0 == 0 && cs.t1 == len);
            slot = 2LL * ctx.g + (cs.k == 0 ? 0 : 1);
        }
        for (int idx = tid; idx < G * D; idx += C::THREADS) {
            const int g = idx / D, dim = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int i = 0; i < C::WARPS; ++i) {
                const float *ri = red + (i * G + g) * (D + 2);
                if (ri[D + 1] > 0.f)
                    M = fmaxf(M, ri[D]);
            }
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int i = 0; i < C::WARPS; ++i) {
                const float *ri = red + (i * G + g) * (D + 2);
                if (ri[D + 1] > 0.f) {
                    const float e = ex2(ri[D] - M);
                    L = fmaf(e, ri[D + 1], L);
                    O = fmaf(e, ri[dim], O);
                }
            }
            const bool nonempty = L > 0.f;
            const float o = nonempty ? O / L : 0.f;
            const long long qrow = (long long)cs.b * Hq + (long long)cs.h * G + g;
            if (complete) {
                store_out(p.out, qrow * D + dim, p.out_dtype, o);
                if (dim == 0 && p.lse)
                    p.lse[qrow] = nonempty ? (M + log2f(L)) * LN2_F : -INFINITY;
            } else {
                const long long r = slot * G + g;
                p.ws_o[r * D + dim] = o;
                if (dim == 0) {
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
                gqa_merge_pieces<C, D>(p, ctx, bh, G, target, gf, off, tid);
            }
        }
        __syncthreads();

        cbase += nc;
        seg_next(p, ctx, cs);
    }

    if (dead) {
        if (lane == 0)
            atomicOr(p.status, STATUS_TIMEOUT);
        for (int i = landed; i < issued; ++i)
            mbar_wait_bounded(bar_base + (i % C::STAGES) * 8, (i / C::STAGES) & 1);
    }
}

template <typename T, int D>
static cudaError_t launch_gqa_t(const GqaParams &gp, cudaStream_t s)
{
    using C = GqaCfg<T, D>;
    const size_t smem = C::smem_bytes(gp.s.decomp, gp.s.B, gp.G);
    auto kern = gqa_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kern<<<gp.s.grid, C::THREADS, smem, s>>>(gp);
    return cudaGetLastError();
}

cudaError_t launch_gqa(int dtype, int d, const GqaParams &gp, cudaStream_t s)
{
    if (dtype == 2)
        return d == 64 ? launch_gqa_t<__nv_bfloat16, 64>(gp, s) : launch_gqa_t<__nv_bfloat16, 128>(gp, s);
    return d == 64 ? launch_gqa_t<__half, 64>(gp, s) : launch_gqa_t<__half, 128>(gp, s);
}

}  // namespace fd
