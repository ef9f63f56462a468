/*
 * fd.h -- C ABI of the split-KV decode attention library (FlashDecoding) for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation: for every batch row b and head h, one query row attends
 * over the first len_b tokens of a KV cache,
 *     out[b,h,:] = softmax(scale * q[b,h,:] . K[b,h,j,:]) . V[b,h,j,:]
 *     lse[b,h]   = ln sum_j exp(scale * q[b,h,:] . K[b,h,j,:])
 * ("FlashDecoding 数学推导", §2.1.1; lse as in "FlashDecoding 数学推导：
 * 传统 m/l/o 方法与 LSE 方法", §2.3.2).  The KV cache is split along the
 * sequence axis into tiles processed in parallel; each tile yields a partial
 * (m, l, o) or (S, o), and an online-softmax merge combines them exactly
 * ("FlashDecoding 数学推导", §2.4-§2.6; "...LSE 方法", §2.3.4).
 *
 * Conventions for every call:
 *   - Every pointer argument is a DEVICE pointer owned by the caller; the
 *     library allocates no memory and keeps no reference after returning.
 *   - Layouts are contiguous row-major:
 *       q   [B, H, d]        K, V [B, H, N, d]      seqlens [B] int32
 *       out [B, H, d]        lse  [B, H] float32
 *       o_part [B, H, P, d] float32,  m_part / l_part / lse_part [B, H, P]
 *     Tokens at index >= seqlens[b] are never read.
 *   - q, K and V share one storage dtype, except for E4M3 K/V, whose q is
 *     f32, f16 or bf16; accumulation is always float32.
 *   - Supported head dims: 64 and 128; also 256 with f16, bf16 or E4M3 K/V
 *     (fd_decode, fd_decode_split, the combines, fd_decode_paged,
 *     fd_decode_fp8, fd_decode_noalloc, and grouped-query decode, paged
 *     or not, with f16, bf16 or E4M3 K/V).  q, K, V, out,
 *     o_part must be 16-byte aligned; seqlens, lse, m/l/lse partials 4-byte
 *     aligned.
 *   - All m and lse values are natural-log quantities of the *scaled* scores.
 *     An empty split is (o = 0, m = -inf, l = 0, lse = -inf); an empty
 *     sequence (len 0) gives out = 0, lse = -inf.
 *   - seqlens values are clamped to [0, N] on the device.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous and stream-ordered; nothing synchronises.
 *   - Errors that the host can detect (null or misaligned pointers, bad
 *     sizes, unsupported d or dtype, short workspace) are returned before
 *     anything is launched.  A failed launch returns FD_ERR_CUDA.  Faults
 *     during execution surface at the caller's next synchronisation.  A
 *     kernel that gives up waiting on its own memory copies (an internal
 *     bound, far above any real copy time) records it in a device status
 *     word read by fd_device_status().
 */
#ifndef FD_H
#define FD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* FD_E4M3 (OCP FP8 E4M3, one byte) is a KV-cache element type for
 * fd_decode_fp8, fd_decode_gqa_fp8 and fd_decode_gqa_paged_fp8 only. */
typedef enum { FD_F32 = 0, FD_F16 = 1, FD_BF16 = 2, FD_E4M3 = 3 } fd_dtype;

typedef enum {
    FD_OK = 0,
    FD_ERR_INVALID_ARG = 1,     /* null / misaligned pointer, negative size   */
    FD_ERR_UNSUPPORTED = 2,     /* head dim or dtype outside the support set  */
    FD_ERR_WORKSPACE = 3,       /* workspace missing or smaller than required */
    FD_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed       */
    FD_ERR_DEVICE_TIMEOUT = 5,  /* a kernel gave up waiting on its own copies */
    FD_ERR_SCRATCH_TOO_SMALL = 6, /* fd_decode_noalloc: problem exceeds its scratch */
    FD_ERR_BAD_PAGE = 7         /* a block-table entry named no page (see fd_decode_paged) */
} fd_status;

/* Human-readable name of a status code (static string, never NULL; an
 * unknown code gives "FD_UNKNOWN_STATUS"). */
const char *fd_status_str(fd_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int fd_version(void);

/* Number of SMs of the current device, or -1 on a CUDA error. */
int fd_num_sms(void);

/*
 * Split count the two-call path (fd_decode_split + fd_combine_*) would use
 * for this shape on a device with `sm_count` SMs, and that fd_decode uses
 * for num_splits == 0 when the batch is too large for its balanced
 * decomposition.  The split-count heuristic of "adv04: Flash-Decoding" (Q2:
 * about seq/1024, capped) is replaced by one that fills every SM: enough
 * (b, h, split) work items for several waves (at least 4 per SM), splits of
 * at least 256 tokens, and among counts from that minimum up to 4 times it,
 * the one whose items fill the last round-robin wave over the CTAs best;
 * never more than FD_MAX_COMBINE_SPLITS.
 *   dtype  the K/V storage type (FD_F32, FD_F16, FD_BF16 or FD_E4M3).  The
 *          rule is the same for every storage type (a split's fixed cost
 *          is per split, its streaming cost per token), so that
 *          fd_workspace_size, which takes no dtype, sizes every type's
 *          workspace; the argument is checked and reserved.
 * Returns >= 1, or -1 for invalid sizes or an unknown dtype.
 */
int fd_auto_num_splits(int B, int H, int N, int d, fd_dtype dtype, int sm_count);

/* The largest split count whose partials fd_combine_mlo / fd_combine_lse
 * merge (their per-split weights live in shared memory), and so the largest
 * num_splits fd_decode_split accepts.  fd_decode and its variants merge in
 * the kernel and accept up to 65535. */
#define FD_MAX_COMBINE_SPLITS 8192

/*
 * Bytes of device workspace fd_decode needs for this shape and num_splits
 * (0 = automatic) on the current device.  The workspace holds per-split
 * partials and one arrival counter per (b, h).  It needs no initialisation:
 * fd_decode clears the counters it uses, on its stream, before its kernel
 * runs.  Two calls that overlap on the GPU must not share one workspace.
 * Returns 0 for invalid sizes.
 */
size_t fd_workspace_size(int B, int H, int N, int d, int num_splits);

/*
 * Fused split-KV decode attention: split kernel plus an in-kernel merge by
 * the last tile of each (b, h) to finish ("FlashDecoding 数学推导", §2.5,
 * stage 1 and stage 2, in one launch).
 *   q, k, v      inputs in `in_dtype` (layouts above)
 *   seqlens      per-sequence lengths, or NULL for "all N"
 *   num_splits   0 = automatic: the (b, h, token) space is divided evenly
 *                over the SMs, so a (b, h) may be split at any token; > 0 =
 *                each sequence is split into num_splits pieces of
 *                ceil(len/num_splits) tokens ("adv04: Flash-Decoding" §4).
 *                The result does not depend on the split (up to rounding).
 *   scale        score scale (normally 1/sqrt(d))
 *   out          [B, H, d] in `out_dtype` (round-to-nearest-even)
 *   lse          [B, H] float32, or NULL
 *   workspace    device buffer of at least fd_workspace_size(...) bytes,
 *                256-byte aligned (see above)
 */
fd_status fd_decode(const void *q, const void *k, const void *v, const int32_t *seqlens,
                    int B, int H, int N, int d, fd_dtype in_dtype, int num_splits,
                    float scale, void *out, fd_dtype out_dtype, float *lse,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * fd_decode over a paged KV cache: the block-table indirection of "adv04:
 * Flash-Decoding" §5 (FlashInfer's 分页 KV Cache, block_table) and
 * "从第一性原理推导 Flash Attention" §7.1.  Same operation and results as
 * fd_decode on the gathered rows.
 *   k_pages, v_pages  [num_pages, H, page_size, d] in `in_dtype`: every
 *                     (page, head) holds page_size consecutive token rows
 *   block_table       [B, max_pages] int32: logical page j of sequence b is
 *                     physical page block_table[b*max_pages + j]
 *   seqlens           [B] int32, required; clamped to [0, max_pages*page_size];
 *                     only table entries of pages holding tokens < seqlens[b]
 *                     are read
 *   workspace         fd_workspace_size(B, H, max_pages*page_size, d, num_splits)
 * A table entry outside [0, num_pages) is never dereferenced: its rows are
 * read from page 0 instead and fd_device_status() reports FD_ERR_BAD_PAGE
 * (the results of that sequence are then meaningless).
 */
fd_status fd_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                          const int32_t *block_table, const int32_t *seqlens, int B, int H, int d,
                          int page_size, int max_pages, long long num_pages, fd_dtype in_dtype,
                          int num_splits, float scale, void *out, fd_dtype out_dtype, float *lse,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * Grouped-query decode (MQA / GQA, "从第一性原理推导 Flash Attention" §8):
 * Hq = G * Hkv query heads, query head h attending with K/V head h / G, so
 * every K/V byte serves G query rows.  Same results as fd_decode with each
 * K/V head repeated G times.
 *   q    [B, Hq, d]          k, v [B, Hkv, N, d]      out [B, Hq, d]
 *   lse  [B, Hq] float32 or NULL
 * G == 1 is fd_decode.  For G >= 2 the per-chunk contraction runs on the
 * tensor cores, which need 16-bit operands: in_dtype f16 or bf16.  The
 * cache may hold any number of rows in all (the copies address a row by its
 * place in its (b, K/V head) block and the block's index).  Up to 16
 * query heads per K/V head (and any group with d = 256 or a paged cache),
 * the products are mma.sync and a K/V head's query heads are processed in
 * even slices of at most 16 (8 at d = 256), each reading that K/V head's
 * rows, side by side so that the repeated reads are mostly served from L2.
 * From 17 query heads per K/V head (MQA included; contiguous cache, d = 64
 * or 128) they are tcgen05 products with accumulators in tensor memory, all
 * of a K/V head's query heads (slices of at most 128) served from one copy
 * of each K/V chunk.  With num_splits == 0 the tcgen05 kernels divide the
 * (b, K/V head, token) space after charging every (b, K/V head) a fixed
 * start cost (the segment end and the reload that switching sequences
 * takes), so a CTA that starts a sequence streams fewer tokens; the result
 * does not depend on the division (up to rounding).  The workspace size is
 * fd_workspace_size_gqa(...), one size for fd_decode_gqa,
 * fd_decode_gqa_paged and fd_decode_gqa_fp8.  Returns FD_ERR_UNSUPPORTED for
 * f32 with G > 1.
 */
size_t fd_workspace_size_gqa(int B, int Hq, int Hkv, int N, int d, int num_splits);

fd_status fd_decode_gqa(const void *q, const void *k, const void *v, const int32_t *seqlens,
                        int B, int Hq, int Hkv, int N, int d, fd_dtype in_dtype, int num_splits,
                        float scale, void *out, fd_dtype out_dtype, float *lse, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * Grouped-query decode over an E4M3 KV cache: fd_decode_gqa with the K/V
 * storage of fd_decode_fp8 (FP8 KV cache, "从第一性原理推导 Flash
 * Attention" §6.2 and §8).
 *   q         [B, Hq, d] in q_dtype (f32, f16 or bf16)
 *   k, v      [B, Hkv, N, d] OCP E4M3 bytes; K[b,h,t,i] = k_scale[b*Hkv+h] *
 *             e4m3(byte), likewise V
 *   k_scale, v_scale  [B*Hkv] float32, device
 *   workspace fd_workspace_size_gqa(B, Hq, Hkv, N, d, num_splits) bytes
 * d must be 64, 128 or 256.  At d = 128 (G >= 2) both products run in FP8
 * on the tcgen05 tensor cores straight from the cache bytes: q and P are
 * each split into three E4M3 parts of weights 1, 2^-4 and 2^-8 (about 12
 * significant bits), q brought to amax in [128, 256) per query head by a
 * power of two that the scores undo.  At d = 64 and 256 the E4M3 rows are
 * converted exactly to f16 in shared memory and the products run on the
 * tensor cores in f16 with fp32 accumulation, q brought into the f16 range
 * the same way.  Query heads in slices of at most 8.  G == 1 is
 * fd_decode_fp8.
 */
fd_status fd_decode_gqa_fp8(const void *q, fd_dtype q_dtype, const void *k, const void *v,
                            const float *k_scale, const float *v_scale, const int32_t *seqlens, int B,
                            int Hq, int Hkv, int N, int d, int num_splits, float scale, void *out,
                            fd_dtype out_dtype, float *lse, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * Grouped-query decode over a paged E4M3 KV cache: fd_decode_gqa_fp8 with
 * the block-table indirection of fd_decode_gqa_paged (the layouts, table
 * rules and bad-entry handling of fd_decode_paged; "从第一性原理推导 Flash
 * Attention" §6.2, §7.1, §8).
 *   k_pages, v_pages  [num_pages, Hkv, page_size, d] E4M3 bytes
 *   k_scale, v_scale  [B*Hkv] float32 (per sequence and K/V head)
 *   workspace         fd_workspace_size_gqa(B, Hq, Hkv, max_pages*page_size,
 *                     d, num_splits) bytes
 * d must be 64, 128 or 256, page_size 16 or a multiple of 32 and
 * num_pages*Hkv < 2^31; any G >= 1 (G = 1 runs the same kernel).  At
 * d = 128 with G >= 2 and pages of a multiple of 128 tokens the FP8
 * tcgen05 products of fd_decode_gqa_fp8 run, else the f16 conversion.
 * Other head dims or page sizes return FD_ERR_UNSUPPORTED.
 */
fd_status fd_decode_gqa_paged_fp8(const void *q, fd_dtype q_dtype, const void *k_pages, const void *v_pages,
                                  const float *k_scale, const float *v_scale, const int32_t *block_table,
                                  const int32_t *seqlens, int B, int Hq, int Hkv, int d, int page_size,
                                  int max_pages, long long num_pages, int num_splits, float scale, void *out,
                                  fd_dtype out_dtype, float *lse, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * Grouped-query decode over a paged KV cache: fd_decode_gqa with the
 * block-table indirection of fd_decode_paged ("从第一性原理推导 Flash
 * Attention" §7.1 and §8; "adv04: Flash-Decoding" §5).  Same results as
 * fd_decode_gqa on the gathered rows: bit for bit when page_size is a
 * multiple of 32 (the same chunks, the same arithmetic); with 16-token pages
 * a chunk is staged from its aligned 32-token block, so its tokens may be
 * shared between warps differently and the rounding may differ.
 *   q                 [B, Hq, d]; out [B, Hq, d]; lse [B, Hq] or NULL
 *   k_pages, v_pages  [num_pages, Hkv, page_size, d] in `in_dtype` (f16 or
 *                     bf16): every (page, K/V head) holds page_size
 *                     consecutive token rows
 *   block_table       [B, max_pages] int32, as in fd_decode_paged
 *   seqlens           [B] int32, required; clamped to [0, max_pages*page_size]
 *   workspace         fd_workspace_size_gqa(B, Hq, Hkv, max_pages*page_size,
 *                     d, num_splits) bytes, 256-byte aligned
 * page_size must be 16 or a multiple of 32 (a 32-token chunk then lies in
 * one page, or in two 16-token pages fetched one by one) and
 * num_pages*Hkv < 2^31 (a (page, K/V head) block is a 32-bit copy
 * coordinate; the pool's total row count is not limited); otherwise
 * FD_ERR_UNSUPPORTED.  Bad table entries are handled as in fd_decode_paged
 * (page 0 read instead, FD_ERR_BAD_PAGE reported).  G == 1 is
 * fd_decode_paged.
 */
fd_status fd_decode_gqa_paged(const void *q, const void *k_pages, const void *v_pages,
                              const int32_t *block_table, const int32_t *seqlens, int B, int Hq,
                              int Hkv, int d, int page_size, int max_pages, long long num_pages,
                              fd_dtype in_dtype, int num_splits, float scale, void *out,
                              fd_dtype out_dtype, float *lse, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * fd_decode over an FP8 KV cache: K and V hold OCP E4M3 bytes with one
 * float32 dequantisation scale per (b, h); the value of K[b,h,t,i] is
 * k_scale[b*H+h] * e4m3(k[b,h,t,i]), likewise V.  Storing the cache in FP8
 * is the "FP8 support" of "从第一性原理推导 Flash Attention" §6.2 applied to
 * the decode cache: half the bytes per token, so about twice the tokens per
 * second at the same HBM bandwidth.  The attention itself is fd_decode's,
 * in float32.
 *   q          [B, H, d] in q_dtype (f32, f16 or bf16)
 *   k, v       [B, H, N, d] E4M3 bytes (16-byte aligned)
 *   k_scale, v_scale  [B, H] float32
 * All other arguments as in fd_decode; the workspace size is
 * fd_workspace_size(B, H, N, d, num_splits).
 */
fd_status fd_decode_fp8(const void *q, fd_dtype q_dtype, const void *k, const void *v,
                        const float *k_scale, const float *v_scale, const int32_t *seqlens,
                        int B, int H, int N, int d, int num_splits, float scale, void *out,
                        fd_dtype out_dtype, float *lse, void *workspace, size_t workspace_bytes,
                        void *stream);

/*
 * Stage 1 alone: per-split partials for num_splits >= 1 splits of every
 * sequence, split p covering tokens [p*c, min((p+1)*c, len)), c =
 * ceil(len/num_splits) ("adv04: Flash-Decoding" §4).  For each split
 * ("FlashDecoding 数学推导", §2.4.1 direct form; "...LSE 方法", §2.3.3):
 *   m_part   = max_j s_j,   l_part = sum_j exp(s_j - m),
 *   o_part   = sum_j exp(s_j - m) V_j / l   (normalised, float32),
 *   lse_part = m + ln l   (may be NULL).
 * Empty splits get (0, -inf, 0, -inf).  1 <= num_splits <=
 * FD_MAX_COMBINE_SPLITS, so that the combines below can merge the result.
 */
fd_status fd_decode_split(const void *q, const void *k, const void *v, const int32_t *seqlens,
                          int B, int H, int N, int d, fd_dtype in_dtype, int num_splits,
                          float scale, float *o_part, float *m_part, float *l_part,
                          float *lse_part, void *stream);

/*
 * Stage 2, m/l/o form ("FlashDecoding 数学推导", §2.4.2 / §2.5 stage 2):
 *   m_g = max_p m_p,  l_g = sum_p exp(m_p - m_g) l_p,
 *   out = sum_p exp(m_p - m_g) l_p o_p / l_g,  lse = m_g + ln l_g.
 * Splits with l_p == 0 get weight 0.  1 <= P <= FD_MAX_COMBINE_SPLITS.
 * lse may be NULL.
 */
fd_status fd_combine_mlo(const float *o_part, const float *m_part, const float *l_part,
                         int B, int H, int P, int d, void *out, fd_dtype out_dtype,
                         float *lse, void *stream);

/*
 * Stage 2, LSE form ("FlashDecoding 数学推导：传统 m/l/o 方法与 LSE 方法",
 * §2.3.4): S_g = ln sum_p exp(S_p) (max-shifted), out = sum_p exp(S_p - S_g)
 * o_p, lse = S_g.  Splits with S_p == -inf get weight 0.
 * 1 <= P <= FD_MAX_COMBINE_SPLITS.  lse may be NULL.
 */
fd_status fd_combine_lse(const float *o_part, const float *lse_part,
                         int B, int H, int P, int d, void *out, fd_dtype out_dtype,
                         float *lse, void *stream);

/*
 * Merge two sets of normalised partial results, row by row, with the
 * operator (+) of "FlashDecoding 数学推导：传统 m/l/o 方法与 LSE 方法"
 * §2.3.5, in the safe two-term form of its §3.2.1 stage 2:
 *   S   = max(S_a, S_b) + log1p(exp(min - max)),
 *   out = o_a exp(S_a - S) + o_b exp(S_b - S),   lse_out = S.
 * (+) is associative, so the partials of a sequence split across several
 * calls, streams or devices (each one fd_decode over its range of tokens,
 * with float32 out and lse) fold to the unsplit result in any order or tree.
 * A row with S = -inf on one side takes the other side unchanged.
 *   o_a, o_b, o_out      [rows, d] float32, 16-byte aligned, d % 4 == 0
 *   lse_a, lse_b, lse_out [rows] float32 (natural log)
 * The outputs may alias either input.
 */
fd_status fd_merge_lse(const float *o_a, const float *lse_a, const float *o_b, const float *lse_b,
                       int rows, int d, float *o_out, float *lse_out, void *stream);

/*
 * Reads (and if `reset` is non-zero, clears) the current device's status
 * word, which a kernel sets when it gives up waiting on its own copies or
 * meets a block-table entry that names no page.  Synchronises the device.
 * Returns FD_OK, FD_ERR_DEVICE_TIMEOUT, FD_ERR_BAD_PAGE or FD_ERR_CUDA.
 */
fd_status fd_device_status(int reset);

/*
 * Test hook for the failure path (the pages have no counterpart: this checks
 * the library's own failure reporting).  Launches, on `stream`, a one-warp
 * kernel that waits, with the kernels' own bounded wait, on a barrier that
 * nothing completes.  After the wait's limit (1 s) it gives up and records
 * FD_ERR_DEVICE_TIMEOUT in the device status word, as a kernel whose copies
 * never landed would; the kernel then ends, and the context stays usable.
 * Read the result with fd_device_status().  Returns FD_OK when launched, else
 * FD_ERR_CUDA.
 */
fd_status fd_selftest_wait_timeout(void *stream);

/*
 * Size of the static device scratch that fd_decode_noalloc uses: 1 MiB.
 * Every GPU on which this library is loaded holds it until the process
 * exits.
 */
#define FD_NOALLOC_SCRATCH_BYTES (1u << 20)

/*
 * fd_decode_noalloc -- fd_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart to this call: it is an addition to
 * the library's interface, not a step of the method.
 *
 * Who needs it: code that may not allocate GPU memory while it decodes, for
 * example a serving engine that gives all device memory to its own pool at
 * start-up and forbids allocation on the per-token path (cudaMalloc can
 * synchronise the device and stall every stream), or a plugin slot of an
 * inference runtime that receives only input and output pointers and a
 * stream.  Such callers cannot provide fd_decode's workspace.
 *
 * What it does: exactly fd_decode (same arguments, same results, same
 * kernels) with the workspace replaced by a static device array of
 * FD_NOALLOC_SCRATCH_BYTES inside this library.  The caller still passes
 * q, K, V, seqlens, out and lse.  Nothing is allocated: no cudaMalloc,
 * cudaFree or allocating library routine is called.
 *
 * Limits and rules:
 *   - A problem whose partials and counters need more than
 *     FD_NOALLOC_SCRATCH_BYTES returns FD_ERR_SCRATCH_TOO_SMALL before
 *     anything is launched.  The need is (each term rounded up to 256
 *     bytes):
 *       num_splits == 0 and B <= 1024 (the balanced decomposition):
 *         2*SMs*(d+2)*4 + 4*B*H bytes, e.g. B*H up to ~220,000 for
 *         d = 128 on a 152-SM GPU;
 *       num_splits == 0 and B > 1024: the automatic split count P =
 *         fd_auto_num_splits(B, H, N, d, in_dtype, SMs) is used, and the
 *         need is B*H*P*(d+2)*4 + 4*B*H bytes (B = 2048, H = 1, d = 128
 *         already exceeds 1 MiB);
 *       num_splits = P > 0: B*H*P*(d+2)*4 + 4*B*H bytes.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The looked-up address is cached per
 *     device; host threads that make their first calls at once may each
 *     look it up, and store the same value (the cache is atomic).
 *   - Every call uses the same array and it keeps the previous call's
 *     contents; each call clears, on its stream, the counters it relies on.
 *     Calls that overlap on the GPU (other streams, other host threads) race
 *     on the array: the caller must serialise them.
 */
fd_status fd_decode_noalloc(const void *q, const void *k, const void *v, const int32_t *seqlens,
                            int B, int H, int N, int d, fd_dtype in_dtype, int num_splits,
                            float scale, void *out, fd_dtype out_dtype, float *lse, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FD_H */
