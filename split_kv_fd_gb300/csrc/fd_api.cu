// fd_api.cu -- host side of the C ABI declared in include/fd.h: argument
// checks, the choice of decomposition and grid, workspace carving, and the
// launches.  Nothing here computes attention; every step runs in the kernels.
#include "fd.h"
#include "fd_gqa.cuh"
#include "fd_gqa_tc8.cuh"
#include "fd_internal.h"
#include "fd_split.cuh"

#include <algorithm>
#include <atomic>
#include <cuda.h>

#include <cuda_runtime.h>
#include <stdint.h>

namespace fd {

// Device status word (per device): set by a kernel that gave up waiting on
// its own copies.
__device__ unsigned g_status_word;

namespace {

constexpr int MAX_DEVICES = 64;
// Cached device address of g_status_word, per device.  Host threads whose
// first calls on a device coincide may each look it up; they store the same
// value, and the atomic makes that well defined.
std::atomic<unsigned *> g_status_ptr[MAX_DEVICES];

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return -1;
    return dev;
}

int sm_count()
{
    const int dev = current_device();
    if (dev < 0)
        return -1;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    return n;
}

unsigned *status_ptr()
{
    const int dev = current_device();
    if (dev < 0)
        return nullptr;
    if (dev < MAX_DEVICES) {
        unsigned *cached = g_status_ptr[dev].load(std::memory_order_acquire);
        if (cached)
            return cached;
    }
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess)
        return nullptr;
    if (dev < MAX_DEVICES)
        g_status_ptr[dev].store(static_cast<unsigned *>(ptr), std::memory_order_release);
    return static_cast<unsigned *>(ptr);
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool valid_dtype(int t) { return t == FD_F32 || t == FD_F16 || t == FD_BF16; }

// The plan of one fd_decode call.
struct Plan {
    int decomp;
    int P;        // splits (DECOMP_SPLITS)
    int grid;
    long long slots;
};

Plan make_plan(int B, int H, int N, int d, int num_splits, int sms, int dtype = FD_BF16)
{
    Plan pl;
    const int ctas = sms * FD_CTAS_PER_SM;  // persistent grid
    if (num_splits == 0 && B <= BALANCED_MAX_B) {
        pl.decomp = DECOMP_BALANCED;
        pl.P = 0;
        pl.grid = ctas;
        pl.slots = 2LL * ctas;
    } else {
        pl.decomp = DECOMP_SPLITS;
        pl.P = num_splits > 0 ? num_splits : fd_auto_num_splits(B, H, N, d, (fd_dtype)dtype, sms);
        const long long items = (long long)B * H * pl.P;
        pl.grid = (int)(items < ctas ? items : ctas);
        pl.slots = (long long)B * H * pl.P;
    }
    return pl;
}

struct WsLayout {
    size_t o_off, ml_off, cnt_off, total;
};

WsLayout ws_layout(long long slots, int d, long long rows)
{
    WsLayout w;
    w.o_off = 0;
    w.ml_off = round_up((size_t)slots * d * sizeof(float), 256);
    w.cnt_off = w.ml_off + round_up((size_t)slots * 2 * sizeof(float), 256);
    w.total = w.cnt_off + round_up((size_t)rows * sizeof(unsigned), 256);
    return w;
}

bool sizes_ok(int B, int H, int N, int d)
{
    return B >= 0 && H >= 0 && N >= 0 && d > 0 && (long long)B * H <= (1LL << 31) - 1;
}

// Head dims of the split kernel: 64 and 128 for every storage type, 256 for
// 16-bit and E4M3 storage (a float32 row of 256 would span 64 lanes).
bool split_dim_ok(int dtype, int d)
{
    return d == 64 || d == 128 || (d == 256 && dtype != FD_F32);
}

// Head dims of the grouped-query kernel.
bool gqa_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }

// The G query heads of a K/V head as NG virtual heads of at most Gs each:
// the kernel holds at most MAXG heads per warp (16 at d = 64 and 128, 8 at
// 256), so larger groups (MQA with many heads) are sliced evenly.
void gqa_slices(int d, int G, int &NG, int &Gs, bool f8 = false)
{
    const int maxg = f8 ? GqaCfg<__half, 128, true>::MAXG
                        : (d == 256 ? GqaCfg<__half, 256>::MAXG : GqaCfg<__half, 128>::MAXG);
    NG = (G + maxg - 1) / maxg;
    Gs = (G + NG - 1) / NG;
}

// Whether a grouped-query call runs the tcgen05 kernel (fd_gqa_tc.cuh): 16-bit
// K/V in a contiguous cache, head dim 64 or 128, and groups large enough
// that staging each chunk once per 16 heads (the mma.sync kernel) would
// bound it.
bool gqa_use_tc(int in_dtype, int d, int G, bool paged)
{
    return !paged && (in_dtype == FD_F16 || in_dtype == FD_BF16) && (d == 64 || d == 128) &&
           G >= FD_GQA_TC_MIN_G;
}

// What the balanced decomposition charges the tcgen05 kernel for each (b, K/V
// head) sequence a CTA starts, in tokens: measured at full load, a CTA's
// switch of sequences (the segment end with its partial's stores and
// arrival, the query reload, the pipeline's refill) takes about as long as
// streaming FD_TC_SEG_COST_KB of K and V.
#ifndef FD_TC_SEG_COST_KB
#define FD_TC_SEG_COST_KB 768
#endif
// The same for the FP8 tcgen05 kernel (fd_gqa_tc8.cuh).
#ifndef FD_TC8_SEG_COST_KB
#define FD_TC8_SEG_COST_KB 256
#endif
// In tokens of K and V rows of d elements of `es` bytes.
int seg_cost_tokens(long long kb, int d, int es)
{
    return (int)(kb * 1024LL / (2LL * es * d));
}

// The block-table view of a paged K/V cache.
struct PagedKV {
    const int32_t *table;
    int page_size, max_pages;
    long long num_pages;
};

// Whether an E4M3 grouped-query call runs the FP8 tcgen05 kernel
// (fd_gqa_tc8.cuh): head dim 128, a contiguous cache or pages of a multiple
// of its 128-token chunk, two or more query heads per K/V head.
bool gqa_use_tc8(int in_dtype, int d, int G, const PagedKV *paged)
{
    return in_dtype == FD_E4M3 && d == 128 && G >= 2 &&
           (!paged || paged->page_size % Tc8Cfg<128>::CT == 0);
}

// The tcgen05 kernel's slices: up to 128 query heads (its MMA rows) each.
void gqa_tc_slices(int G, int &NG, int &Gs)
{
    constexpr int maxg = TcCfg<__half, 128>::MAXG;
    NG = (G + maxg - 1) / maxg;
    Gs = (G + NG - 1) / NG;
}

// The grouped-query plan: the decomposition of the K/V heads' token space
// over grid / NG ranges, each run by NG adjacent CTAs (one per slice of the
// query heads); slots and arrival counters per (b, virtual head).
Plan gqa_plan(int B, int Hkv, int N, int d, int num_splits, int sms, int NG)
{
    Plan pl = make_plan(B, Hkv, N, d, num_splits, sms);
    const int ranges = std::max(1, sms * FD_CTAS_PER_SM / NG);
    if (pl.decomp == DECOMP_BALANCED) {
        pl.grid = ranges * NG;
        pl.slots = 2LL * pl.grid;
    } else {
        const long long items = (long long)B * Hkv * pl.P;
        pl.grid = (int)std::min<long long>(items, ranges) * NG;
        pl.slots = (long long)B * Hkv * NG * pl.P;
    }
    return pl;
}

template <typename T> size_t split_smem_t(int d, int decomp, int B)
{
    return d == 64    ? SplitCfg<T, 64>::smem_bytes(decomp, B)
           : d == 128 ? SplitCfg<T, 128>::smem_bytes(decomp, B)
                      : SplitCfg<T, 256>::smem_bytes(decomp, B);
}

size_t split_smem(int dtype, int d, int decomp, int B)
{
    if (dtype == FD_E4M3)
        return split_smem_t<__nv_fp8_e4m3>(d, decomp, B);
    if (dtype == FD_F32)
        return d == 64 ? SplitCfg<float, 64>::smem_bytes(decomp, B) : SplitCfg<float, 128>::smem_bytes(decomp, B);
    if (dtype == FD_F16)
        return split_smem_t<__half>(d, decomp, B);
    return split_smem_t<__nv_bfloat16>(d, decomp, B);
}

fd_status launch(int dtype, int d, const SplitParams &p, int decomp, cudaStream_t s)
{
    const size_t smem = split_smem(dtype, d, decomp, p.B);
    cudaError_t e;
    if (dtype == FD_F32)
        e = launch_split_f32(d, p, smem, s);
    else if (dtype == FD_E4M3)
        e = launch_split_fp8(d, p, smem, s);
    else if (dtype == FD_F16)
        e = launch_split_f16(d, p, smem, s);
    else
        e = launch_split_bf16(d, p, smem, s);
    return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

// cuTensorMapEncodeTiled, fetched from the driver through the runtime (no
// link-time dependency on the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled()
{
    // looked up once; concurrent first calls store the same pointer
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (f)
        return f;
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    f = reinterpret_cast<EncodeTiledFn>(ptr);
    fn.store(f, std::memory_order_release);
    return f;
}

// K or V as `blocks` blocks of n rows of d 16-bit elements (a (b, K/V head)
// of a contiguous cache, or a (page, K/V head) of a paged one), viewed as
// the 4-D map [64 elements, n, blocks, d/64 planes] (strides d*2, n*d*2 and
// 128 bytes) with boxes [64, box_rows, 1, box_planes] and the 128-byte
// swizzle: a box lands in shared memory plane by plane.  A row is addressed
// by (row in block, block), two coordinates below 2^31, so the cache may
// hold any number of rows in all.
bool make_kv_map(CUtensorMap *m, const void *base, int dtype, int d, long long n, long long blocks,
                 int box_rows, int box_planes)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn)
        return false;
    const cuuint64_t dims[4] = {64, (cuuint64_t)n, (cuuint64_t)blocks, (cuuint64_t)(d / 64)};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)n * d * 2, 128};
    const cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, (cuuint32_t)box_planes};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, dtype == FD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
              const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 K or V as `blocks` blocks of n rows of 128 bytes: the 3-D map [128,
// n, blocks] of bytes (strides 128 and n*128) with boxes [128, box_rows, 1]
// and the 128-byte swizzle.
bool make_f8_map(CUtensorMap *m, const void *base, long long n, long long blocks, int box_rows)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)n, (cuuint64_t)blocks};
    const cuuint64_t strides[2] = {128, (cuuint64_t)n * 128};
    const cuuint32_t box[3] = {128, (cuuint32_t)box_rows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// What every fused entry point sets alike: the score scale in base 2, the
// plan, the outputs, the workspace carve-up and the status word.
void set_fused(SplitParams &p, const Plan &pl, const WsLayout &wl, void *workspace, float scale,
               void *out, int out_dtype, float *lse, unsigned *status)
{
    p.scale_log2 = scale * 1.4426950408889634f;
    p.decomp = pl.decomp;
    p.P = pl.P;
    p.grid = pl.grid;
    p.out_kind = OUT_FUSED;
    p.out = out;
    p.out_dtype = out_dtype;
    p.lse = lse;
    char *ws = static_cast<char *>(workspace);
    p.ws_o = reinterpret_cast<float *>(ws + wl.o_off);
    p.ws_ml = reinterpret_cast<float *>(ws + wl.ml_off);
    p.ws_cnt = reinterpret_cast<unsigned *>(ws + wl.cnt_off);
    p.status = status;
}

// The arrival counters of `rows` sequences start at zero on every call: a
// reused workspace may hold anything at these bytes.  One split per
// sequence (nothing to merge) uses none.
bool clear_counters(const SplitParams &p, long long rows, cudaStream_t s)
{
    if (p.decomp == DECOMP_SPLITS && p.P == 1)
        return true;
    return cudaMemsetAsync(p.ws_cnt, 0, (size_t)rows * sizeof(unsigned), s) == cudaSuccess;
}

// The grouped-query launch once an entry point has checked its arguments:
// plan, workspace, the K and V tensor maps over `kv_blocks` blocks of
// `kv_n` rows of d elements (none when kv_blocks is 0), and the kernel's
// parameters.  `paged` is null for contiguous K/V [B, Hkv, N, d].
fd_status gqa_common(const void *q, const void *k, const void *v, const int32_t *seqlens, int B, int Hq,
                     int Hkv, int N, int d, int in_dtype, int num_splits, float scale, void *out,
                     int out_dtype, float *lse, void *workspace, size_t workspace_bytes, void *stream,
                     long long kv_n, long long kv_blocks, const PagedKV *paged, const float *k_scale = nullptr,
                     const float *v_scale = nullptr, int q_dtype = -1)
{
    const bool f8 = in_dtype == FD_E4M3;   // then q_dtype is q's own and no tensor maps are made
    const int G = Hq / Hkv;
    const bool tc = gqa_use_tc(in_dtype, d, G, paged != nullptr);
    const bool tc8 = gqa_use_tc8(in_dtype, d, G, paged);
    int NG, Gs;
    if (tc)
        gqa_tc_slices(G, NG, Gs);
    else
        gqa_slices(d, G, NG, Gs, f8);   // the FP8 tcgen05 kernel's slices are the E4M3 kernel's
    const long long Hv = (long long)Hkv * NG;   // virtual heads
    const int sms = sm_count();
    unsigned *st = status_ptr();
    if (sms <= 0 || !st)
        return FD_ERR_CUDA;
    const Plan pl = gqa_plan(B, Hkv, N, d, num_splits, sms, NG);
    const WsLayout wl = ws_layout(pl.slots * Gs, d, (long long)B * Hv);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 256))
        return FD_ERR_WORKSPACE;

    GqaParams gp;
    memset(&gp, 0, sizeof gp);
    // boxes of one chunk (CT rows, every plane), or with 16-token pages of one
    // page (16 rows, every plane)
    gp.pages16 = (paged && paged->page_size == 16) ? 1 : 0;
    const int box_rows = tc ? TcCfg<__half, 128>::CT
                         : tc8        ? Tc8Cfg<128>::CT
                         : gp.pages16 ? 16
                                      : GqaCfg<__half, 128>::CT;
    const int box_planes = d / 64;
    const bool maps = kv_n > 0 && kv_blocks > 0;
    if (maps && !f8) {
        if (!make_kv_map(&gp.tmk, k, in_dtype, d, kv_n, kv_blocks, box_rows, box_planes) ||
            !make_kv_map(&gp.tmv, v, in_dtype, d, kv_n, kv_blocks, box_rows, box_planes))
            return FD_ERR_CUDA;
    } else if (maps && d == 128) {   // E4M3 at d = 128: swizzled byte boxes
        if (!make_f8_map(&gp.tmk, k, kv_n, kv_blocks, box_rows) ||
            !make_f8_map(&gp.tmv, v, kv_n, kv_blocks, box_rows))
            return FD_ERR_CUDA;
    }
    gp.G = Gs;
    gp.NG = NG;
    gp.Gq = G;
    SplitParams &p = gp.s;
    p.q = q;
    p.k = k;
    p.v = v;
    p.lens = seqlens;
    p.B = B;
    p.H = Hkv;
    p.N = N;
    if (paged) {
        p.paged = 1;
        p.block_table = paged->table;
        p.page_size = paged->page_size;
        p.max_pages = paged->max_pages;
        p.num_pages = paged->num_pages;
    }
    p.q_dtype = f8 ? q_dtype : in_dtype;
    gp.k_scale = k_scale;
    gp.v_scale = v_scale;
    set_fused(p, pl, wl, workspace, scale, out, out_dtype, lse, st);
    if (pl.decomp == DECOMP_BALANCED && (tc || tc8))
        p.seg_cost = tc ? seg_cost_tokens(FD_TC_SEG_COST_KB, d, 2) : seg_cost_tokens(FD_TC8_SEG_COST_KB, d, 1);
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (!clear_counters(p, (long long)B * Hv, cs))
        return FD_ERR_CUDA;
    const cudaError_t e = tc    ? launch_gqa_tc(in_dtype, d, gp, cs)
                          : tc8 ? launch_gqa_tc8(d, gp, cs)
                          : f8  ? launch_gqa_f8(d, gp, cs)
                                : launch_gqa(in_dtype, d, gp, cs);
    return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

}  // namespace
}  // namespace fd

namespace fd {
// the bounded-wait self-test kernel (fd_combine.cu)
cudaError_t launch_wait_selftest(unsigned *status, cudaStream_t s);
}  // namespace fd

using namespace fd;

extern "C" {

const char *fd_status_str(fd_status status)
{
    switch ((int)status) {
    case FD_OK: return "FD_OK";
    case FD_ERR_INVALID_ARG: return "FD_ERR_INVALID_ARG: null or misaligned pointer, or bad size";
    case FD_ERR_UNSUPPORTED: return "FD_ERR_UNSUPPORTED: head dim or dtype not supported";
    case FD_ERR_WORKSPACE: return "FD_ERR_WORKSPACE: workspace missing or too small";
    case FD_ERR_CUDA: return "FD_ERR_CUDA: a CUDA runtime call or launch failed";
    case FD_ERR_DEVICE_TIMEOUT: return "FD_ERR_DEVICE_TIMEOUT: a kernel gave up waiting on its copies";
    case FD_ERR_BAD_PAGE:
        return "FD_ERR_BAD_PAGE: a block-table entry named no page (its rows were read from page 0)";
    case FD_ERR_SCRATCH_TOO_SMALL:
        return "FD_ERR_SCRATCH_TOO_SMALL: the problem needs more scratch than fd_decode_noalloc's "
               "static buffer (FD_NOALLOC_SCRATCH_BYTES) holds; use fd_decode with a workspace";
    default: return "FD_UNKNOWN_STATUS";
    }
}

int fd_version(void) { return 100; }

int fd_num_sms(void) { return sm_count(); }

int fd_auto_num_splits(int B, int H, int N, int d, fd_dtype dtype, int sms)
{
    if (!sizes_ok(B, H, N, d) || sms <= 0 || !(valid_dtype(dtype) || dtype == FD_E4M3))
        return -1;
    const long long bh = (long long)B * H;
    if (bh == 0)
        return 1;
    // several work items per CTA so the persistent grid balances, but never
    // splits shorter than 256 tokens
    const long long want = (4LL * sms + bh - 1) / bh;
    long long cap = N / 256;
    if (cap < 1)
        cap = 1;
    long long lo = want < cap ? want : cap;
    if (lo < 1)
        lo = 1;
    if (lo > FD_MAX_COMBINE_SPLITS)
        lo = FD_MAX_COMBINE_SPLITS;
    // the items go round-robin to the CTAs: from lo up to 4 lo (within the
    // cap), take the split count whose items fill the last round best; a
    // larger count only if it fills more than 1% better
    long long hi = 4 * lo < cap ? 4 * lo : cap;
    if (hi > FD_MAX_COMBINE_SPLITS)
        hi = FD_MAX_COMBINE_SPLITS;
    const long long G = (long long)sms * FD_CTAS_PER_SM;
    long long best = lo;
    double best_fill = -1.0;
    for (long long P = lo; P <= hi; ++P) {
        const long long items = bh * P;
        const double fill = (double)items / (double)(G * ((items + G - 1) / G));
        if (fill > best_fill + 0.01) {
            best_fill = fill;
            best = P;
        }
    }
    return (int)best;
}

size_t fd_workspace_size(int B, int H, int N, int d, int num_splits)
{
    if (!sizes_ok(B, H, N, d) || num_splits < 0)
        return 0;
    const int sms = sm_count();
    if (sms <= 0)
        return 0;
    const Plan pl = make_plan(B, H, N, d, num_splits, sms);
    return ws_layout(pl.slots, d, (long long)B * H).total;
}

fd_status fd_decode(const void *q, const void *k, const void *v, const int32_t *seqlens, int B, int H,
                    int N, int d, fd_dtype in_dtype, int num_splits, float scale, void *out,
                    fd_dtype out_dtype, float *lse, void *workspace, size_t workspace_bytes,
                    void *stream)
{
    if (!sizes_ok(B, H, N, d) || num_splits < 0 || num_splits > 65535)
        return FD_ERR_INVALID_ARG;
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype) || !split_dim_ok(in_dtype, d))
        return FD_ERR_UNSUPPORTED;
    if ((long long)B * H == 0)
        return FD_OK;
    // K and V are never read when N == 0
    if (!q || (N > 0 && (!k || !v)) || !out || !aligned(q, 16) || !aligned(k, 16) ||
        !aligned(v, 16) || !aligned(out, 16) || (seqlens && !aligned(seqlens, 4)) ||
        (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    const int sms = sm_count();
    unsigned *st = status_ptr();
    if (sms <= 0 || !st)
        return FD_ERR_CUDA;
    const Plan pl = make_plan(B, H, N, d, num_splits, sms, in_dtype);
    const WsLayout wl = ws_layout(pl.slots, d, (long long)B * H);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 256))
        return FD_ERR_WORKSPACE;

    SplitParams p = {};
    p.q = q;
    p.k = k;
    p.v = v;
    p.lens = seqlens;
    p.B = B;
    p.H = H;
    p.N = N;
    p.q_dtype = in_dtype;
    set_fused(p, pl, wl, workspace, scale, out, out_dtype, lse, st);
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (!clear_counters(p, (long long)B * H, cs))
        return FD_ERR_CUDA;
    return launch(in_dtype, d, p, pl.decomp, cs);
}

fd_status fd_decode_split(const void *q, const void *k, const void *v, const int32_t *seqlens, int B,
                          int H, int N, int d, fd_dtype in_dtype, int num_splits, float scale,
                          float *o_part, float *m_part, float *l_part, float *lse_part, void *stream)
{
    if (!sizes_ok(B, H, N, d) || num_splits < 1 || num_splits > FD_MAX_COMBINE_SPLITS)
        return FD_ERR_INVALID_ARG;
    if (!valid_dtype(in_dtype) || !split_dim_ok(in_dtype, d))
        return FD_ERR_UNSUPPORTED;
    if ((long long)B * H == 0)
        return FD_OK;
    if (!q || (N > 0 && (!k || !v)) || !o_part || !m_part || !l_part || !aligned(q, 16) || !aligned(k, 16) ||
        !aligned(v, 16) || !aligned(o_part, 16) || !aligned(m_part, 4) || !aligned(l_part, 4) ||
        (lse_part && !aligned(lse_part, 4)) || (seqlens && !aligned(seqlens, 4)))
        return FD_ERR_INVALID_ARG;
    const int sms = sm_count();
    unsigned *st = status_ptr();
    if (sms <= 0 || !st)
        return FD_ERR_CUDA;
    const long long items = (long long)B * H * num_splits;
    const int ctas = sms * FD_CTAS_PER_SM;

    SplitParams p = {};
    p.q = q;
    p.k = k;
    p.v = v;
    p.lens = seqlens;
    p.B = B;
    p.H = H;
    p.N = N;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.q_dtype = in_dtype;
    p.decomp = DECOMP_SPLITS;
    p.P = num_splits;
    p.grid = (int)(items < ctas ? items : ctas);
    p.out_kind = OUT_PARTIALS;
    p.o_part = o_part;
    p.m_part = m_part;
    p.l_part = l_part;
    p.lse_part = lse_part;
    p.status = st;
    return launch(in_dtype, d, p, DECOMP_SPLITS, static_cast<cudaStream_t>(stream));
}

static fd_status combine_common(const float *o_part, const float *a, const float *b, bool lse_form,
                                int B, int H, int P, int d, void *out, fd_dtype out_dtype, float *lse,
                                void *stream)
{
    if (B < 0 || H < 0 || P < 1 || P > FD_MAX_COMBINE_SPLITS || d <= 0 || (long long)B * H > (1LL << 31) - 1)
        return FD_ERR_INVALID_ARG;
    if (!valid_dtype(out_dtype) || (d != 64 && d != 128 && d != 256))
        return FD_ERR_UNSUPPORTED;
    if ((long long)B * H == 0)
        return FD_OK;
    if (!o_part || !a || (!lse_form && !b) || !out || !aligned(o_part, 16) || !aligned(a, 4) ||
        (b && !aligned(b, 4)) || !aligned(out, 16) || (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    CombineParams p = {};
    p.o_part = o_part;
    if (lse_form) {
        p.lse_part = a;
    } else {
        p.m_part = a;
        p.l_part = b;
    }
    p.rows = B * H;
    p.P = P;
    p.d = d;
    p.out = out;
    p.out_dtype = out_dtype;
    p.lse = lse;
    cudaError_t e = lse_form ? launch_combine_lse(p, static_cast<cudaStream_t>(stream))
                             : launch_combine_mlo(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

fd_status fd_combine_mlo(const float *o_part, const float *m_part, const float *l_part, int B, int H,
                         int P, int d, void *out, fd_dtype out_dtype, float *lse, void *stream)
{
    return combine_common(o_part, m_part, l_part, false, B, H, P, d, out, out_dtype, lse, stream);
}

fd_status fd_combine_lse(const float *o_part, const float *lse_part, int B, int H, int P, int d,
                         void *out, fd_dtype out_dtype, float *lse, void *stream)
{
    return combine_common(o_part, lse_part, nullptr, true, B, H, P, d, out, out_dtype, lse, stream);
}

fd_status fd_merge_lse(const float *o_a, const float *lse_a, const float *o_b, const float *lse_b,
                       int rows, int d, float *o_out, float *lse_out, void *stream)
{
    if (rows < 0 || d <= 0 || d % 4 != 0)
        return FD_ERR_INVALID_ARG;
    if (rows == 0)
        return FD_OK;
    if (!o_a || !lse_a || !o_b || !lse_b || !o_out || !lse_out || !aligned(o_a, 16) ||
        !aligned(o_b, 16) || !aligned(o_out, 16) || !aligned(lse_a, 4) || !aligned(lse_b, 4) ||
        !aligned(lse_out, 4))
        return FD_ERR_INVALID_ARG;
    return launch_merge_lse(o_a, lse_a, o_b, lse_b, rows, d, o_out, lse_out,
                            static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? FD_OK
               : FD_ERR_CUDA;
}

fd_status fd_selftest_wait_timeout(void *stream)
{
    unsigned *st = status_ptr();
    if (!st)
        return FD_ERR_CUDA;
    return launch_wait_selftest(st, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FD_OK
                                                                                       : FD_ERR_CUDA;
}

fd_status fd_device_status(int reset)
{
    if (cudaDeviceSynchronize() != cudaSuccess)
        return FD_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof v) != cudaSuccess)
        return FD_ERR_CUDA;
    if (reset) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess)
            return FD_ERR_CUDA;
    }
    if (v & STATUS_TIMEOUT)
        return FD_ERR_DEVICE_TIMEOUT;
    return (v & STATUS_BAD_PAGE) ? FD_ERR_BAD_PAGE : FD_OK;
}

size_t fd_workspace_size_gqa(int B, int Hq, int Hkv, int N, int d, int num_splits)
{
    if (Hkv <= 0 || Hq < 0 || Hq % Hkv != 0)
        return 0;
    if (Hq == Hkv)
        return fd_workspace_size(B, Hq, N, d, num_splits);
    if (!sizes_ok(B, Hq, N, d) || num_splits < 0 || !gqa_dim_ok(d))
        return 0;
    const int sms = sm_count();
    if (sms <= 0)
        return 0;
    // the largest of the grouped-query kernels' layouts (their slices differ):
    // mma.sync 16-bit, mma.sync E4M3 and tcgen05
    size_t total = 0;
    for (int kind = 0; kind < 3; ++kind) {
        if (kind == 2 && d > 128)
            continue;
        if (kind == 2 && !gqa_use_tc(FD_BF16, d, Hq / Hkv, false))
            continue;
        int NG, Gs;
        if (kind == 2)
            gqa_tc_slices(Hq / Hkv, NG, Gs);
        else
            gqa_slices(d, Hq / Hkv, NG, Gs, kind == 1);
        const Plan pl = gqa_plan(B, Hkv, N, d, num_splits, sms, NG);
        total = std::max(total, ws_layout(pl.slots * Gs, d, (long long)B * Hkv * NG).total);
    }
    return total;
}

fd_status fd_decode_gqa(const void *q, const void *k, const void *v, const int32_t *seqlens, int B,
                        int Hq, int Hkv, int N, int d, fd_dtype in_dtype, int num_splits, float scale,
                        void *out, fd_dtype out_dtype, float *lse, void *workspace,
                        size_t workspace_bytes, void *stream)
{
    if (Hkv <= 0 || Hq < 0 || Hq % Hkv != 0)
        return FD_ERR_INVALID_ARG;
    if (Hq == Hkv)
        return fd_decode(q, k, v, seqlens, B, Hq, N, d, in_dtype, num_splits, scale, out, out_dtype,
                         lse, workspace, workspace_bytes, stream);
    if (!sizes_ok(B, Hq, N, d) || num_splits < 0 || num_splits > 65535)
        return FD_ERR_INVALID_ARG;
    if (!valid_dtype(out_dtype) || !gqa_dim_ok(d) ||
        (in_dtype != FD_F16 && in_dtype != FD_BF16))
        return FD_ERR_UNSUPPORTED;
    if ((long long)B * Hq == 0)
        return FD_OK;
    if (!q || (N > 0 && (!k || !v)) || !out || !aligned(q, 16) || !aligned(k, 16) ||
        !aligned(v, 16) || !aligned(out, 16) || (seqlens && !aligned(seqlens, 4)) ||
        (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    return gqa_common(q, k, v, seqlens, B, Hq, Hkv, N, d, in_dtype, num_splits, scale, out, out_dtype,
                      lse, workspace, workspace_bytes, stream, N, (long long)B * Hkv, nullptr);
}

fd_status fd_decode_gqa_paged(const void *q, const void *k_pages, const void *v_pages,
                              const int32_t *block_table, const int32_t *seqlens, int B, int Hq, int Hkv,
                              int d, int page_size, int max_pages, long long num_pages, fd_dtype in_dtype,
                              int num_splits, float scale, void *out, fd_dtype out_dtype, float *lse,
                              void *workspace, size_t workspace_bytes, void *stream)
{
    if (Hkv <= 0 || Hq < 0 || Hq % Hkv != 0)
        return FD_ERR_INVALID_ARG;
    if (page_size < 1 || max_pages < 0 || num_pages < 0 ||
        (long long)page_size * max_pages > 0x7fffffffLL)
        return FD_ERR_INVALID_ARG;
    if (Hq == Hkv)
        return fd_decode_paged(q, k_pages, v_pages, block_table, seqlens, B, Hq, d, page_size, max_pages,
                               num_pages, in_dtype, num_splits, scale, out, out_dtype, lse, workspace,
                               workspace_bytes, stream);
    const int N = page_size * max_pages;
    if (!sizes_ok(B, Hq, N, d) || num_splits < 0 || num_splits > 65535)
        return FD_ERR_INVALID_ARG;
    if (!valid_dtype(out_dtype) || !gqa_dim_ok(d) ||
        (in_dtype != FD_F16 && in_dtype != FD_BF16))
        return FD_ERR_UNSUPPORTED;
    // a chunk of CT tokens lies in one page, or 16-token pages are fetched a
    // page at a time; a (page, K/V head) block is a 32-bit tensor-map
    // coordinate
    if ((page_size % GqaCfg<__half, 128>::CT != 0 && page_size != 16) || num_pages * Hkv >= (1LL << 31))
        return FD_ERR_UNSUPPORTED;
    if ((long long)B * Hq == 0)
        return FD_OK;
    const bool pages = N > 0;
    if (!q || !seqlens || !out || (pages && (!k_pages || !v_pages || !block_table || num_pages < 1)) ||
        !aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(seqlens, 4) || !aligned(block_table, 4) || (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    const PagedKV pk = {block_table, page_size, max_pages, num_pages};
    return gqa_common(q, k_pages, v_pages, seqlens, B, Hq, Hkv, N, d, in_dtype, num_splits, scale, out,
                      out_dtype, lse, workspace, workspace_bytes, stream, page_size, pages ? num_pages * Hkv : 0,
                      &pk);
}

fd_status fd_decode_gqa_fp8(const void *q, fd_dtype q_dtype, const void *k, const void *v,
                            const float *k_scale, const float *v_scale, const int32_t *seqlens, int B,
                            int Hq, int Hkv, int N, int d, int num_splits, float scale, void *out,
                            fd_dtype out_dtype, float *lse, void *workspace, size_t workspace_bytes,
                            void *stream)
{
    if (Hkv <= 0 || Hq < 0 || Hq % Hkv != 0)
        return FD_ERR_INVALID_ARG;
    if (Hq == Hkv)
        return fd_decode_fp8(q, q_dtype, k, v, k_scale, v_scale, seqlens, B, Hq, N, d, num_splits, scale, out,
                             out_dtype, lse, workspace, workspace_bytes, stream);
    if (!sizes_ok(B, Hq, N, d) || num_splits < 0 || num_splits > 65535)
        return FD_ERR_INVALID_ARG;
    if (!valid_dtype(q_dtype) || !valid_dtype(out_dtype) || !gqa_dim_ok(d))
        return FD_ERR_UNSUPPORTED;
    if ((long long)B * Hq == 0)
        return FD_OK;
    if (!q || (N > 0 && (!k || !v)) || !k_scale || !v_scale || !out || !aligned(q, 16) || !aligned(k, 16) ||
        !aligned(v, 16) || !aligned(out, 16) || !aligned(k_scale, 4) || !aligned(v_scale, 4) ||
        (seqlens && !aligned(seqlens, 4)) || (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    return gqa_common(q, k, v, seqlens, B, Hq, Hkv, N, d, FD_E4M3, num_splits, scale, out, out_dtype, lse,
                      workspace, workspace_bytes, stream, N, (long long)B * Hkv, nullptr, k_scale, v_scale,
                      q_dtype);
}

fd_status fd_decode_gqa_paged_fp8(const void *q, fd_dtype q_dtype, const void *k_pages, const void *v_pages,
                                  const float *k_scale, const float *v_scale, const int32_t *block_table,
                                  const int32_t *seqlens, int B, int Hq, int Hkv, int d, int page_size,
                                  int max_pages, long long num_pages, int num_splits, float scale, void *out,
                                  fd_dtype out_dtype, float *lse, void *workspace, size_t workspace_bytes,
                                  void *stream)
{
    if (Hkv <= 0 || Hq < 0 || Hq % Hkv != 0)
        return FD_ERR_INVALID_ARG;
    if (page_size < 1 || max_pages < 0 || num_pages < 0 ||
        (long long)page_size * max_pages > 0x7fffffffLL)
        return FD_ERR_INVALID_ARG;
    const int N = page_size * max_pages;
    if (!sizes_ok(B, Hq, N, d) || num_splits < 0 || num_splits > 65535)
        return FD_ERR_INVALID_ARG;
    // E4M3 pages: the grouped-query kernel at d = 64, 128 or 256, G >= 1
    // (one query per K/V head runs it too), pages of 16 or a multiple of 32
    // tokens
    if (!valid_dtype(q_dtype) || !valid_dtype(out_dtype) || !gqa_dim_ok(d))
        return FD_ERR_UNSUPPORTED;
    if ((page_size % GqaCfg<__half, 128>::CT != 0 && page_size != 16) || num_pages * Hkv >= (1LL << 31))
        return FD_ERR_UNSUPPORTED;
    if ((long long)B * Hq == 0)
        return FD_OK;
    const bool pages = N > 0;
    if (!q || !seqlens || !out || !k_scale || !v_scale ||
        (pages && (!k_pages || !v_pages || !block_table || num_pages < 1)) || !aligned(q, 16) ||
        !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) || !aligned(seqlens, 4) ||
        !aligned(block_table, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4) || (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    const PagedKV pk = {block_table, page_size, max_pages, num_pages};
    return gqa_common(q, k_pages, v_pages, seqlens, B, Hq, Hkv, N, d, FD_E4M3, num_splits, scale, out, out_dtype,
                      lse, workspace, workspace_bytes, stream, page_size, pages ? num_pages * Hkv : 0, &pk, k_scale,
                      v_scale, q_dtype);
}

fd_status fd_decode_fp8(const void *q, fd_dtype q_dtype, const void *k, const void *v,
                        const float *k_scale, const float *v_scale, const int32_t *seqlens, int B,
                        int H, int N, int d, int num_splits, float scale, void *out,
                        fd_dtype out_dtype, float *lse, void *workspace, size_t workspace_bytes,
                        void *stream)
{
    if (!sizes_ok(B, H, N, d) || num_splits < 0 || num_splits > 65535)
        return FD_ERR_INVALID_ARG;
    if (!valid_dtype(q_dtype) || !valid_dtype(out_dtype) || !split_dim_ok(FD_E4M3, d))
        return FD_ERR_UNSUPPORTED;
    if ((long long)B * H == 0)
        return FD_OK;
    if (!q || (N > 0 && (!k || !v)) || !k_scale || !v_scale || !out || !aligned(q, 16) ||
        !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(k_scale, 4) ||
        !aligned(v_scale, 4) || (seqlens && !aligned(seqlens, 4)) || (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    const int sms = sm_count();
    unsigned *st = status_ptr();
    if (sms <= 0 || !st)
        return FD_ERR_CUDA;
    const Plan pl = make_plan(B, H, N, d, num_splits, sms, FD_E4M3);
    const WsLayout wl = ws_layout(pl.slots, d, (long long)B * H);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 256))
        return FD_ERR_WORKSPACE;

    SplitParams p = {};
    p.q = q;
    p.k = k;
    p.v = v;
    p.lens = seqlens;
    p.B = B;
    p.H = H;
    p.N = N;
    p.q_dtype = q_dtype;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    set_fused(p, pl, wl, workspace, scale, out, out_dtype, lse, st);
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (!clear_counters(p, (long long)B * H, cs))
        return FD_ERR_CUDA;
    return launch(FD_E4M3, d, p, pl.decomp, cs);
}

fd_status fd_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                          const int32_t *block_table, const int32_t *seqlens, int B, int H, int d,
                          int page_size, int max_pages, long long num_pages, fd_dtype in_dtype,
                          int num_splits, float scale, void *out, fd_dtype out_dtype, float *lse,
                          void *workspace, size_t workspace_bytes, void *stream)
{
    if (page_size < 1 || max_pages < 0 || num_pages < 0 ||
        (long long)page_size * max_pages > 0x7fffffffLL)
        return FD_ERR_INVALID_ARG;
    const int N = page_size * max_pages;
    if (!sizes_ok(B, H, N, d) || num_splits < 0 || num_splits > 65535)
        return FD_ERR_INVALID_ARG;
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype) || !split_dim_ok(in_dtype, d))
        return FD_ERR_UNSUPPORTED;
    if ((long long)B * H == 0)
        return FD_OK;
    const bool pages = N > 0;
    if (!q || !seqlens || !out || (pages && (!k_pages || !v_pages || !block_table || num_pages < 1)) ||
        !aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(seqlens, 4) || !aligned(block_table, 4) || (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    const int sms = sm_count();
    unsigned *st = status_ptr();
    if (sms <= 0 || !st)
        return FD_ERR_CUDA;
    const Plan pl = make_plan(B, H, N, d, num_splits, sms, in_dtype);
    const WsLayout wl = ws_layout(pl.slots, d, (long long)B * H);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 256))
        return FD_ERR_WORKSPACE;

    SplitParams p = {};
    p.q = q;
    p.k = k_pages;
    p.v = v_pages;
    p.lens = seqlens;
    p.B = B;
    p.H = H;
    p.N = N;
    p.paged = 1;
    p.block_table = block_table;
    p.page_size = page_size;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.q_dtype = in_dtype;
    set_fused(p, pl, wl, workspace, scale, out, out_dtype, lse, st);
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (!clear_counters(p, (long long)B * H, cs))
        return FD_ERR_CUDA;
    return launch(in_dtype, d, p, pl.decomp, cs);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// fd_decode_noalloc: fd_decode whose scratch is a static device array.
//
// Some callers cannot allocate device memory when they decode: a serving
// engine that hands all GPU memory to its own pool at start-up and forbids
// allocation on the per-token path (cudaMalloc may synchronise the device
// and stall every stream), or a plugin slot of an inference runtime that is
// given only input/output pointers and a stream.  This entry point needs no
// workspace from them: the partials and arrival counters live in the array
// below, which every GPU that loads this library holds until the process
// exits.  All calls share it, so calls that overlap on the GPU (different
// streams, or different host threads) race and must be serialised by the
// caller.
// ---------------------------------------------------------------------------
namespace fd {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FD_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, looked up once per device.  In host
// code the array's name is only a host-side stand-in, never a device
// address, so kernels must be given this pointer instead.
// Host threads whose first calls on a device coincide may each look it up;
// they store the same value, and the atomic makes that well defined.
std::atomic<void *> g_noalloc_ptr[MAX_DEVICES];

void *noalloc_scratch()
{
    const int dev = current_device();
    if (dev < 0 || dev >= MAX_DEVICES)
        return nullptr;
    void *cached = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (cached)
        return cached;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess)
        return nullptr;
    g_noalloc_ptr[dev].store(ptr, std::memory_order_release);
    return ptr;
}

}  // namespace
}  // namespace fd

extern "C" fd_status fd_decode_noalloc(const void *q, const void *k, const void *v,
                                       const int32_t *seqlens, int B, int H, int N, int d,
                                       fd_dtype in_dtype, int num_splits, float scale, void *out,
                                       fd_dtype out_dtype, float *lse, void *stream)
{
    if (!sizes_ok(B, H, N, d) || num_splits < 0 || num_splits > 65535)
        return FD_ERR_INVALID_ARG;
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype) || !split_dim_ok(in_dtype, d))
        return FD_ERR_UNSUPPORTED;
    if ((long long)B * H == 0)
        return FD_OK;
    if (!q || (N > 0 && (!k || !v)) || !out || !aligned(q, 16) || !aligned(k, 16) ||
        !aligned(v, 16) || !aligned(out, 16) || (seqlens && !aligned(seqlens, 4)) ||
        (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    const int sms = sm_count();
    unsigned *st = status_ptr();
    if (sms <= 0 || !st)
        return FD_ERR_CUDA;
    const Plan pl = make_plan(B, H, N, d, num_splits, sms, in_dtype);
    const WsLayout wl = ws_layout(pl.slots, d, (long long)B * H);
    if (wl.total > (size_t)FD_NOALLOC_SCRATCH_BYTES)
        return FD_ERR_SCRATCH_TOO_SMALL;
    void *scratch = noalloc_scratch();  // first call on a device: symbol lookup
    if (!scratch)
        return FD_ERR_CUDA;

    SplitParams p = {};
    p.q = q;
    p.k = k;
    p.v = v;
    p.lens = seqlens;
    p.B = B;
    p.H = H;
    p.N = N;
    p.q_dtype = in_dtype;
    set_fused(p, pl, wl, scratch, scale, out, out_dtype, lse, st);
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (!clear_counters(p, (long long)B * H, cs))
        return FD_ERR_CUDA;
    return launch(in_dtype, d, p, pl.decomp, cs);
}
