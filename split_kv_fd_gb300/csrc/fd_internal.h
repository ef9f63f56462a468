// fd_internal.h -- parameter blocks and launcher declarations shared by the
// host API (fd_api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fd {

// How the (b, h, token) space is divided over CTAs.
enum Decomp : int {
    DECOMP_SPLITS = 0,    // each sequence in P pieces of ceil(len/P) tokens;
                          // CTA g takes items g, g+G, g+2G, ... (item = (b,h,p))
    DECOMP_BALANCED = 1,  // the concatenated token space of all (b, h) is cut
                          // into G equal contiguous ranges, one per CTA
};

// What a finished piece ("segment") of a (b, h) writes.
enum OutKind : int {
    OUT_PARTIALS = 0,  // user partial buffers [B, H, P] (the two-call path)
    OUT_FUSED = 1,     // final out/lse; split pieces go through the workspace
                       // and the last piece to arrive merges them
};

struct SplitParams {
    const void *q;
    const void *k;
    const void *v;
    const int32_t *lens;  // device, may be null => all N
    int B, H, N;          // N: padded length (paged: max_pages * page_size)
    // paged KV cache: K/V are [num_pages, H, page_size, d]; logical token t
    // of sequence b is row t % page_size of page block_table[b*max_pages + t/page_size]
    int paged;
    const int32_t *block_table;
    int page_size, max_pages;
    long long num_pages;
    float scale_log2;     // scale * log2(e): scores are kept in base 2
    int q_dtype;          // 0 f32, 1 f16, 2 bf16 (K/V: the kernel's element type)
    const float *k_scale; // [B*H] K dequantisation scales, or null (1)
    const float *v_scale; // [B*H] V dequantisation scales, or null (1)
    int decomp;
    int seg_cost;         // DECOMP_BALANCED: tokens charged for starting each (b, h) sequence
    int P;                // splits per sequence for DECOMP_SPLITS
    int grid;             // number of CTAs launched (G)
    int out_kind;
    // OUT_PARTIALS
    float *o_part, *m_part, *l_part, *lse_part;
    // OUT_FUSED
    void *out;
    int out_dtype;
    float *lse;
    float *ws_o;          // [slots, d]   normalised partial o
    float *ws_ml;         // [slots, 2]   (m natural-log, l)
    unsigned *ws_cnt;     // [B*H]        arrival counters (zero between calls)
    unsigned *status;     // device status word
};

struct CombineParams {
    const float *o_part, *m_part, *l_part, *lse_part;
    int rows, P, d;
    void *out;
    int out_dtype;
    float *lse;
};

// Persistent CTAs launched per SM by the split kernel.
#ifndef FD_CTAS_PER_SM
#define FD_CTAS_PER_SM 1
#endif

// The balanced decomposition gives every CTA it uses at least this many
// tokens (a small problem runs on fewer CTAs rather than on slivers).
constexpr long long BALANCED_MIN_TOKENS = 128;

// Largest batch the balanced decomposition keeps its length prefix sums for
// in shared memory; larger batches use DECOMP_SPLITS.
constexpr int BALANCED_MAX_B = 1024;

// Per-(dtype, d) launchers; each returns the cudaError_t of the launch.
struct LaunchInfo {
    int threads;
    size_t smem_bytes;
};

LaunchInfo split_launch_info(int dtype, int d, int decomp, int B);
cudaError_t launch_split(int dtype, int d, const SplitParams &p, cudaStream_t s);
cudaError_t launch_split_f32(int d, const SplitParams &p, size_t smem, cudaStream_t s);
cudaError_t launch_split_f16(int d, const SplitParams &p, size_t smem, cudaStream_t s);
cudaError_t launch_split_bf16(int d, const SplitParams &p, size_t smem, cudaStream_t s);
cudaError_t launch_split_fp8(int d, const SplitParams &p, size_t smem, cudaStream_t s);

cudaError_t launch_combine_mlo(const CombineParams &p, cudaStream_t s);
cudaError_t launch_combine_lse(const CombineParams &p, cudaStream_t s);
cudaError_t launch_merge_lse(const float *oa, const float *sa, const float *ob, const float *sb,
                             int rows, int d, float *out, float *sout, cudaStream_t s);

}  // namespace fd
