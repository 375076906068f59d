/*
 * gqa.h -- C interface of the B300 (sm_103a) grouped-query attention library.
 *
 * Grouped-query attention (GQA): h_q query heads share g key/value heads;
 * query head i reads K/V head i / (h_q / g) (integer division), and each
 * (batch, query head) computes softmax(Q K^T * scale) V. Sources: the
 * GroupedQueryAttention code and the attention formula in "Modern LLM
 * architecture (1): GQA and RMSNorm" (zeeklog.com), sections 2.1 and 2.3;
 * the index map kv_head_id = query_head_id // group_size in the "Qwen,
 * DeepSeek and LLaMA3 attention survey" (jsqmd.com), section 2.2; the KV
 * cache layout [batch, g, seq_len, d_head] and its growth by concatenation in
 * the "What is Grouped-Query Attention" explainer (ijyty.com), sections 2.2
 * and 3.2.
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller, dense and
 *    row-major in the layout stated, 16-byte aligned. The library never
 *    allocates, frees or synchronises; work is queued on `stream` (a
 *    cudaStream_t passed as void*, NULL = the legacy default stream).
 *  - bf16 means IEEE bfloat16 (the upper 16 bits of a binary32).
 *  - Arguments are checked on the host before anything is launched; a
 *    failed check returns its status and queues no work.
 *  - `status_dev` (optional, may be NULL) is a device int32 the kernels set
 *    to a nonzero gqa_status_t when they detect a problem at run time
 *    (a bounded wait that ran out, an append that did not fit). The first
 *    problem recorded wins; the caller clears it and reads it after the
 *    stream has been synchronised.
 *  - Supported shapes: d in {64, 128}; g >= 1 divides h_q; the group size
 *    G = h_q / g is a power of two no larger than 128; all sizes >= 1
 *    (prefill) and their products fit the index types (B*L*h_q*d < 2^31,
 *    B*g*S_max < 2^31).
 *  - Kernels are built for sm_103a only; another device yields GQA_ERR_CUDA.
 *
 * Where these declarations differ from the interface as first specified:
 * every entry point returns int (a gqa_status_t value) and gqa_status_string
 * takes int, so FFI callers see a fixed 32-bit type whatever width a C
 * compiler picks for the enum; the output arguments (o, o_dtype, lse) sit
 * together right after the inputs, before the sizes; and every launching
 * entry point takes the optional device status word status_dev, the only
 * channel through which a kernel can report a run-time problem.
 */
#ifndef GQA_B300_H
#define GQA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GQA_OK = 0,
  GQA_ERR_NULL = 1,        /* a required pointer is NULL                          */
  GQA_ERR_SHAPE = 2,       /* a size is out of range or inconsistent              */
  GQA_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned                    */
  GQA_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required          */
  GQA_ERR_CACHE_FULL = 5,  /* (device) appended rows did not fit; they were dropped */
  GQA_ERR_CUDA = 6,        /* a CUDA runtime call or a launch failed              */
  GQA_ERR_TIMEOUT = 7,     /* (device) a bounded wait inside a kernel ran out     */
  GQA_ERR_BAD_LENGTH = 8,  /* (device) a seq_lens entry was negative or > S_max   */
  GQA_ERR_SCRATCH_LIMIT = 9, /* the sizes need more scratch than the built-in array */
  GQA_ERR_BAD_PAGE = 10     /* (device) a block-table entry in use was outside the pool */
} gqa_status_t;

typedef enum {
  GQA_OUT_F32 = 0,   /* output written as fp32 */
  GQA_OUT_BF16 = 1   /* output written as bf16 (round to nearest even) */
} gqa_out_dtype_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* gqa_status_string(int status);

/* Library version, encoded as major*10000 + minor*100 + patch. */
int gqa_version(void);

/*
 * gqa_prefill_fwd -- attention over a whole sequence (prefill).
 *
 *   O[b,i,h,:] = sum_j softmax_j(scale * Q[b,i,h,:] . K[b,j,h/G,:]) V[b,j,h/G,:]
 *
 * with j over all L keys, or over j <= i when `causal` != 0 (query and key
 * positions coincide). The K/V head of query head h is h / G, G = h_q / g;
 * K and V are read in place, never duplicated per query head (the pages'
 * GroupedQueryAttention code, sections 2.1 and 2.3 of the zeeklog.com page).
 *
 *   q      [B, L, h_q, d] bf16   (projection-output layout)
 *   k, v   [B, L, g,   d] bf16
 *   o      [B, L, h_q, d] fp32 or bf16 per o_dtype (written, never read)
 *   lse    optional fp32 [B, h_q, L]: natural-log sum of exp(scale * q.k)
 *          over the visible keys of each row (written when non-NULL)
 *   scale  softmax scale, usually 1/sqrt(d); must be finite and > 0
 *
 * Returns GQA_OK once the work is queued, or an error with nothing queued.
 */
int gqa_prefill_fwd(const void* q, const void* k, const void* v, void* o,
                    int o_dtype, float* lse, int B, int L, int h_q, int g, int d,
                    float scale, int causal, int32_t* status_dev, void* stream);

/*
 * gqa_prefill_fwd_ex -- gqa_prefill_fwd with the score-bias variants the pages
 * name: Mistral's sliding-window attention (the model table of the zeeklog.com
 * page, section 2.4) and ALiBi's per-head distance penalty (the jsqmd.com
 * survey, section 3.2).
 *
 *   window        0, or W > 0 (requires causal != 0): row i also hides every
 *                 key j <= i - W, i.e. it sees the W keys i-W+1 .. i
 *   alibi_slopes  NULL, or device fp32 [h_q]: slope_h * |i - j| (natural
 *                 units) is subtracted from scale * q.k before the softmax
 *
 * Same layouts, ownership and errors as gqa_prefill_fwd; a window with
 * causal == 0 or a negative window is GQA_ERR_SHAPE.
 */
int gqa_prefill_fwd_ex(const void* q, const void* k, const void* v, void* o, int o_dtype,
                       float* lse, int B, int L, int h_q, int g, int d, float scale, int causal,
                       int window, const float* alibi_slopes, int32_t* status_dev,
                       void* stream);

/*
 * gqa_prefill_kvcache_fwd -- chunked prefill: T new tokens per sequence attend
 * to everything already in the KV cache and, causally, to each other (the
 * cache concatenation of the ijyty.com explainer, section 3.2, for more than
 * one new token; bottom-right causal alignment).
 *
 *   q          [B, T, h_q, d] bf16, the T newest tokens of every sequence
 *   k_cache,
 *   v_cache    [B, g, S_max, d] bf16 that already hold those tokens' K/V
 *              (kv_cache_append them first); rows at or past seq_lens[b]
 *              are never used (they may hold anything, NaN included)
 *   seq_lens   device int32 [B], rows per sequence, each in [T, S_max];
 *              token t of sequence b sits at position seq_lens[b] - T + t
 *              and sees rows 0 .. seq_lens[b] - T + t (within `window`)
 *   o          [B, T, h_q, d] fp32 or bf16; lse optional fp32 [B, h_q, T]
 *   window, alibi_slopes  as in gqa_prefill_fwd_ex (ALiBi distance measured
 *              between cache positions)
 *
 * T > S_max is GQA_ERR_SHAPE; a seq_lens entry outside [T, S_max] is clamped
 * into it and flagged GQA_ERR_BAD_LENGTH (that sequence's output is then
 * not meaningful).
 */
int gqa_prefill_kvcache_fwd(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* seq_lens, void* o, int o_dtype, float* lse, int B,
                            int T, int h_q, int g, int d, int S_max, float scale, int window,
                            const float* alibi_slopes, int32_t* status_dev, void* stream);

/*
 * gqa_decode_workspace_bytes -- device scratch bytes gqa_decode_fwd needs for
 * these sizes (split-KV partial outputs and their log-sum-exp values).
 * Returns 0 for sizes gqa_decode_fwd would reject.
 */
size_t gqa_decode_workspace_bytes(int B, int h_q, int g, int d, int S_max);

/*
 * gqa_decode_fwd -- one new query token per sequence attends over the KV
 * cache (the autoregressive decode step of the ijyty.com explainer,
 * section 2.1).
 *
 *   O[b,h,:] = sum_{j < seq_lens[b]} softmax_j(scale * q[b,h,:] . Kc[b,h/G,j,:]) Vc[b,h/G,j,:]
 *
 *   q          [B, h_q, d] bf16
 *   k_cache,
 *   v_cache    [B, g, S_max, d] bf16; rows at or past seq_lens[b] are never
 *              used in the result (they may hold anything, NaN included)
 *   seq_lens   device int32 [B], each in [0, S_max]; a sequence of length 0
 *              gives an all-zero output row and lse = -inf. Entries outside
 *              [0, S_max] are clamped and flagged GQA_ERR_BAD_LENGTH.
 *   o          [B, h_q, d] fp32 or bf16 per o_dtype
 *   lse        optional fp32 [B, h_q] (natural log), may be NULL
 *   workspace  device scratch of at least gqa_decode_workspace_bytes(...)
 *              bytes, 16-byte aligned, owned by the caller; its contents on
 *              entry do not matter and are garbage on exit. Calls that run
 *              concurrently on different streams need separate workspaces.
 */
int gqa_decode_fwd(const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* seq_lens, void* o, int o_dtype, float* lse,
                   int B, int h_q, int g, int d, int S_max, float scale,
                   void* workspace, size_t workspace_bytes,
                   int32_t* status_dev, void* stream);

/*
 * gqa_decode_fwd_ex -- gqa_decode_fwd with a sliding window (the query, at
 * position seq_lens[b] - 1, sees only the last `window` rows; 0 = all) and
 * optional ALiBi slopes (device fp32 [h_q]; slope_h * (seq_lens[b] - 1 - j)
 * is subtracted from the scaled score of row j). Same workspace as
 * gqa_decode_fwd; a negative window is GQA_ERR_SHAPE.
 */
int gqa_decode_fwd_ex(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* seq_lens, void* o, int o_dtype, float* lse, int B, int h_q,
                      int g, int d, int S_max, float scale, int window,
                      const float* alibi_slopes, void* workspace, size_t workspace_bytes,
                      int32_t* status_dev, void* stream);

/*
 * kv_cache_append -- write T new tokens per sequence behind its valid rows
 * and advance its length (the cache concatenation along the sequence axis,
 * ijyty.com explainer section 3.2; the cache keeps only g heads).
 *
 *   k_cache, v_cache  [B, g, S_max, d] bf16, updated in place
 *   seq_lens          device int32 [B], read then set to min(len + T, S_max)
 *   k_new, v_new      [B, T, g, d] bf16 (projection-output layout)
 *
 * Token t of sequence b is copied bit for bit into row seq_lens[b] + t of
 * every K/V head. Rows that would land at or past S_max are dropped and
 * GQA_ERR_CACHE_FULL is recorded in *status_dev (if given). Two launches are
 * queued: the row copy, then the length update. The update is a programmatic
 * dependent launch that may start once every row-copy block has read its
 * lengths, before the copied rows have landed; later work on the stream sees
 * both complete, as with any two launches.
 */
int kv_cache_append(void* k_cache, void* v_cache, int32_t* seq_lens,
                    const void* k_new, const void* v_new, int B, int g, int d,
                    int S_max, int T, int32_t* status_dev, void* stream);

/*
 * Paged KV cache with group-aligned pages (the PagedAttention integration of
 * the jsqmd.com survey, section 4.3: a page holds page_size tokens of one K/V
 * group, and the g group pages of one physical block are adjacent):
 *
 *   k_pool, v_pool  [num_pages, g, page_size, d] bf16
 *   block_table     device int32 [B, max_blocks]; entry i of sequence b is the
 *                   physical page of its logical rows i*page_size ..
 *                   (i+1)*page_size - 1 (entries past a sequence's length are
 *                   never read)
 *   page_size       a power of two in [16, 65536]; the logical capacity of a
 *                   sequence is page_size * max_blocks (< 2^31)
 *
 * An entry that is in use but outside [0, num_pages) reads zeros and is
 * flagged GQA_ERR_BAD_PAGE; sizes out of range are GQA_ERR_SHAPE.
 */

/* Workspace of gqa_decode_paged_fwd (0 for sizes it would reject). */
size_t gqa_decode_paged_workspace_bytes(int B, int h_q, int g, int d, int page_size,
                                        int max_blocks);

/*
 * gqa_decode_paged_fwd -- gqa_decode_fwd_ex over a paged cache: the same
 * result as gqa_decode_fwd_ex on the contiguous cache whose row j of
 * sequence b is row j % page_size of page block_table[b][j / page_size].
 * seq_lens entries are in [0, page_size * max_blocks].
 */
int gqa_decode_paged_fwd(const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_table, const int32_t* seq_lens, void* o,
                         int o_dtype, float* lse, int B, int h_q, int g, int d, int page_size,
                         int num_pages, int max_blocks, float scale, int window,
                         const float* alibi_slopes, void* workspace, size_t workspace_bytes,
                         int32_t* status_dev, void* stream);

/*
 * kv_cache_append_paged -- kv_cache_append into a paged cache: token t of
 * sequence b goes to logical row seq_lens[b] + t through the block table.
 * Rows past the capacity page_size * max_blocks are dropped and flagged
 * GQA_ERR_CACHE_FULL; lengths saturate at the capacity. Two launches.
 */
int kv_cache_append_paged(void* k_pool, void* v_pool, const int32_t* block_table,
                          int32_t* seq_lens, const void* k_new, const void* v_new, int B, int g,
                          int d, int page_size, int num_pages, int max_blocks, int T,
                          int32_t* status_dev, void* stream);

/*
 * kv_cache_append_rope -- kv_cache_append with the rotary position embedding
 * of the jsqmd.com attention survey (chapter 1, RoPE code; chapter 5 names
 * the fused-RoPE build option) applied on the way in, in one launch (plus
 * the length update):
 *   - key rows are rotated before they are stored, value rows are copied;
 *   - if q is given, the same tokens' query rows are rotated into q_out.
 * Token t of sequence b takes position p = seq_lens[b] + t (its cache row).
 * For each row x (d elements) and i < d/2:
 *     out[i]       = x[2i] * cos[p][i] - x[2i+1] * sin[p][i]
 *     out[d/2 + i] = x[2i] * sin[p][i] + x[2i+1] * cos[p][i]
 * evaluated in binary32 with each product, sum and difference rounded (no
 * fused multiply-add), then rounded to bf16 (nearest, ties to even).
 *
 *   k_cache, v_cache, seq_lens, k_new, v_new, B, g, d, S_max, T
 *                   as in kv_cache_append (k_new/v_new must not overlap the cache)
 *   q, q_out        device bf16 [B, T, h_q, d], both NULL or both given;
 *                   q_out == q rotates in place, otherwise the two must not
 *                   overlap. Query rows of tokens dropped for lack of room
 *                   are not written. h_q is ignored when q is NULL.
 *   rope_cos, rope_sin
 *                   device fp32 [rope_n_pos, d/2], row p = the cosines and
 *                   sines of position p; 16-byte aligned; rope_n_pos must be
 *                   >= S_max (every cache row has a table row)
 *
 * Errors as in kv_cache_append (GQA_ERR_CACHE_FULL / GQA_ERR_BAD_LENGTH in
 * *status_dev); sizes out of range are GQA_ERR_SHAPE.
 */
int kv_cache_append_rope(void* k_cache, void* v_cache, int32_t* seq_lens, const void* k_new,
                         const void* v_new, const void* q, void* q_out, const float* rope_cos,
                         const float* rope_sin, int rope_n_pos, int B, int h_q, int g, int d,
                         int S_max, int T, int32_t* status_dev, void* stream);

/*
 * kv_cache_append_paged_rope -- kv_cache_append_rope into a paged cache
 * (positions are logical rows; rope_n_pos >= page_size * max_blocks). A
 * block-table entry outside the pool for a stored row is GQA_ERR_BAD_PAGE.
 */
int kv_cache_append_paged_rope(void* k_pool, void* v_pool, const int32_t* block_table,
                               int32_t* seq_lens, const void* k_new, const void* v_new,
                               const void* q, void* q_out, const float* rope_cos,
                               const float* rope_sin, int rope_n_pos, int B, int h_q, int g,
                               int d, int page_size, int num_pages, int max_blocks, int T,
                               int32_t* status_dev, void* stream);

/*
 * gqa_selftest_bounded_wait -- checks the failure path the kernels share,
 * without a fault. Every wait inside the library's kernels is bounded (2 s);
 * when one runs out the kernel stops, frees what it holds and writes
 * GQA_ERR_TIMEOUT to its status word. This entry point launches one CTA that
 * waits, with the same code, on a barrier nothing ever arrives at, giving up
 * after limit_us microseconds (1 .. 2e6), so *status_dev (device int32,
 * required) becomes GQA_ERR_TIMEOUT unless it already held an error. The
 * device and the stream remain usable afterwards.
 */
int gqa_selftest_bounded_wait(int32_t* status_dev, int limit_us, void* stream);

/*
 * gqa_decode_fwd_noalloc -- gqa_decode_fwd for callers that cannot allocate.
 * The pages have no counterpart of this entry point; it exists for callers
 * that cannot hand over a workspace: plugin hosts that pass a library only
 * its inputs and outputs while their memory planner owns every other
 * allocation, and serving loops that must not call cudaMalloc after start-up
 * because it can synchronise the device.
 *
 * Same arguments, layouts and results as gqa_decode_fwd, minus the
 * workspace: the split-KV partials go to a scratch array built into the
 * library (gqa_decode_noalloc_scratch_bytes() bytes, 32 MiB), which every GPU
 * that loads the library holds until the process exits. The call allocates
 * nothing. Sizes whose gqa_decode_workspace_bytes exceeds the array are
 * rejected with GQA_ERR_SCRATCH_LIMIT before anything is queued (for
 * d = 128, h_q = 32, g = 8 the ragged B = 64, S_max = 8192 cache needs about
 * 16 MiB).
 *
 *  - The first call made while a device is current looks up the array's
 *    device address on that device (cudaGetSymbolAddress) and keeps it; make
 *    that first call before any stream capture on that device.
 *  - Every call shares the one array per device. The caller clears nothing:
 *    each call writes the partials it reads and zeroes the one counter word
 *    the split pass starts from. Calls that overlap on the GPU (different
 *    streams, or different host threads) race on it and give wrong results;
 *    serialise them.
 */
int gqa_decode_fwd_noalloc(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* seq_lens, void* o, int o_dtype, float* lse, int B,
                           int h_q, int g, int d, int S_max, float scale, int32_t* status_dev,
                           void* stream);

/* Size in bytes of the scratch array behind gqa_decode_fwd_noalloc. */
size_t gqa_decode_noalloc_scratch_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_B300_H */
