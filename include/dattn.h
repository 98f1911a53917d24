/*
 * dattn: split-KV decode attention over a paged KV cache (bf16, 8-bit FP8 E4M3 codes or
 * 4-bit integer codes, the quantized formats with one fp32 scale per row), for GB300
 * (sm_103a).
 *
 * The C ABI of libdattn.so. Every entry point takes plain pointers and sizes: no C++ and
 * no framework types. It validates its arguments on the host, then launches asynchronously
 * on the given CUDA stream. The library never allocates device memory, never frees it and
 * never synchronises. All buffers belong to the caller.
 *
 * The operation comes from the pages this library restates:
 *
 *  [IL] "Infinite-LLM: Efficient LLM Service for Long Context with DistAttention and
 *       Distributed KVCache". DistAttention splits the KV cache of one request into
 *       sub-blocks. Each sub-block j yields a MicroAttention triple over its seq_p keys
 *       (equations in 速读 and in "DistAttention 的等价数学变换"):
 *           m_j  = max_i s_i
 *           e_j  = sum_i exp(s_i - m_j)
 *           MA_j = sum_i exp(s_i - m_j) v_i        (unnormalised)
 *       The triples are then aggregated ("结果聚合与通信开销降低", Fig. 4b):
 *           m_g = max_j m_j,  e_g = sum_j e_j exp(m_j - m_g),
 *           out = sum_j MA_j exp(m_j - m_g) / e_g,
 *       which equals full softmax attention ("分布式注意力机制的通信挑战").
 *  [LS] "LoongServe: Efficiently Serving Long-Context Large Language Models with Elastic
 *       Sequence Parallelism", §4.2. In single- and multi-master distributed decoding, the
 *       master saves the new token's KV in its local pool, every instance computes local
 *       attention over its share of the KV, and the results are merged.
 *  [LV] "LLM长序列服务优化：LServe的块稀疏注意力技术". §2.2.2: 64-token physical pages hold
 *       16-token logical pages with per-channel k_max/k_min, and the page selection is
 *       reused over a window of decode steps. §3.1.2: the statistics are computed when the
 *       KV cache is written, a physical page is scored as the max over its logical pages,
 *       and the top-K pages are selected. §3.1.1: streaming heads attend sink tokens plus
 *       a local window. The streaming and retrieval heads run in one fused kernel.
 *       §3.2.1: the retrieval-head cache is paged and quantized at a configurable 2-8 bits,
 *       the streaming-head cache at 4 bits, with no scheme given; the 8-bit and 4-bit
 *       formats below are this library's reading of it.
 *
 * Here the "instances" are CTAs on one GPU. The KV of every (request, KV head) is split
 * into 16-token tiles. The tiles are spread evenly over num_splits CTAs, so each CTA
 * computes MicroAttention triples over a contiguous range of tiles. Triples of the same
 * (request, KV head) are merged in the same launch by whichever CTA finishes that head
 * last.
 *
 * Notation and conventions
 *  - B requests, Hq query heads, Hkv KV heads, g = Hq / Hkv query heads per KV head
 *    (query head h reads KV head h / g), d = head_dim, P = page_size tokens.
 *  - A logit is s_i = scale * (q . k_i). m values at this ABI are in natural-log units.
 *  - bf16 arrays are passed as dattn_bf16 (raw IEEE bfloat16 bits). Floats are fp32.
 *  - Device pointers are marked (device). Structs passed by pointer live in host memory.
 *  - Sequence length L_b = seq_lens[b]: tokens 0..L_b-1 of request b are valid. Token t
 *    lives in physical page block_table[b * max_pages_per_req + t / P], slot t % P.
 *  - Pool layout: k_pool and v_pool are [num_pages][Hkv][P][d] elements of the layout's
 *    kv_format (the 4-bit format packs two elements per byte: [num_pages][Hkv][P][d/2]
 *    bytes). Every (page, KV head) tile is one contiguous run.
 *  - The 8-bit format (kv_format = DATTN_KV_FP8_E4M3): every (token, KV head) row x of d
 *    values is stored as d one-byte codes plus one fp32 scale. The scales of the 16 tokens
 *    of logical page lp of (page, KV head) form one 128-byte run of kv_scale
 *    [num_pages][Hkv][P/16][2][16]: [..][lp][0][j] is the K scale and [..][lp][1][j] the V
 *    scale of token lp*16 + j of that page. scale = max_i |x_i| / 448
 *    and code_i = E4M3(x_i / scale), both divisions in IEEE fp32; E4M3 is the OCP 8-bit
 *    float (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest finite 448),
 *    rounded to nearest even and saturated to +-448. A row with scale 0 has +0 codes. The
 *    row's values are code_i * scale, and the attention runs over exactly these values.
 *    The query stays bf16; the statistics are still taken from the bf16 keys.
 *  - The 4-bit format (kv_format = DATTN_KV_INT4) [LV §3.2.1: streaming heads at 4 bits,
 *    retrieval heads at 2-8 configurable bits; the page names no scheme]: every (token, KV
 *    head) row x of d values is stored as d/2 bytes plus one fp32 scale in kv_scale, laid
 *    out as for the 8-bit format. scale = max_i |x_i| / 7 and code_i = x_i / scale rounded
 *    to the nearest integer, ties to even, in [-7, 7] (both divisions in IEEE fp32). Byte j
 *    of the row holds code_{2j} + 8 in its low nibble and code_{2j+1} + 8 in its high
 *    nibble. A row with scale 0 has code 0. The row's values are code_i * scale, and the
 *    attention runs over exactly these values.
 *  - The mixed format (kv_format = DATTN_KV_MIXED) [LV §3.2.1: one cache with 4-bit
 *    streaming heads and 2-8-bit retrieval heads]: every KV head h has its own format,
 *    head_format[h] = DATTN_KV_FP8_E4M3 or DATTN_KV_INT4, and its rows are stored exactly as
 *    in that format (codes and kv_scale as above). Of the Hkv heads, H8 are 8-bit and H4 are
 *    4-bit; a head's index within its own format is the number of earlier heads of that
 *    format. The pool is the 8-bit region [num_pages][H8][P][d] bytes followed by the 4-bit
 *    region [num_pages][H4][P][d/2] bytes (this replaces the [num_pages][Hkv][P][d] layout
 *    above); kv_scale keeps the [num_pages][Hkv][P/16][2][16] layout over all heads. One
 *    decode launch reads both regions.
 *  - Statistics layout: stats is [num_pages][Hkv][P/16][2][d]. Entry [..][lp][0][:] is
 *    k_max and [..][lp][1][:] is k_min of logical page lp, the 16 tokens
 *    lp*16..lp*16+15 of that physical page.
 *  - Device data errors (an unmapped page, a page id outside the pool, a length beyond
 *    the block table, a selected page beyond the length, a bounded wait that ran out) do
 *    not trap. The kernel skips the offending tile or token and ORs a DATTN_DEVERR_* bit
 *    into *dev_err when dev_err is not NULL. A skipped tile contributes nothing to the
 *    attention.
 *  - Workspace: calls that merge across CTAs need a caller-owned device workspace of at
 *    least dattn_workspace_size(...) bytes, 256-byte aligned. Its counter region must be
 *    all zero before the first use: allocate it zeroed or call dattn_workspace_init once.
 *    Every call leaves the counters at zero again. Calls that share one workspace must
 *    not run concurrently (use one workspace per stream).
 *  - Supported shapes: d in {64, 128}; P a multiple of 16 from 16 to 256; 1 <= g <= 8;
 *    Hkv <= 256; B (or C for dattn_partial) <= 4096; top_k <= 256.
 */
#ifndef DATTN_H
#define DATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t dattn_bf16;

typedef enum {
    DATTN_OK = 0,
    DATTN_ERR_INVALID_ARG = 1, /* a null pointer, a negative size or an inconsistent shape */
    DATTN_ERR_UNSUPPORTED = 2, /* a valid shape outside the supported set (see above) */
    DATTN_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned */
    DATTN_ERR_CUDA = 4         /* a CUDA runtime or driver call failed */
} dattn_status_t;

/* Bits OR-ed into the optional device error word. */
#define DATTN_DEVERR_UNMAPPED_PAGE 0x1  /* block-table entry < 0 for a needed page */
#define DATTN_DEVERR_PAGE_OOB 0x2       /* block-table entry >= num_pages */
#define DATTN_DEVERR_LEN_OOB 0x4        /* seq_len < 0, or beyond max_pages_per_req * P */
#define DATTN_DEVERR_TIMEOUT 0x8        /* a bounded pipeline wait ran out; output invalid */
#define DATTN_DEVERR_CHUNK_OOB 0x10     /* chunk_req or a chunk page index out of range */
#define DATTN_DEVERR_SELECT_OOB 0x20    /* a selected page lies beyond the request length */
#define DATTN_DEVERR_SMEM_ALIGN 0x40    /* a kernel's shared memory base was not 1024-byte aligned;
                                           that kernel computed nothing */

/* Head kinds of the block-sparse decode [LV §2.1.2, §3.1.1]. */
#define DATTN_HEAD_DENSE 0
#define DATTN_HEAD_RETRIEVAL 1
#define DATTN_HEAD_STREAMING 2

/* Element formats of the KV pool (dattn_kv_layout.kv_format). */
#define DATTN_KV_BF16 0      /* bf16 values */
#define DATTN_KV_FP8_E4M3 1  /* FP8 E4M3 codes with one fp32 scale per (token, KV head) row */
#define DATTN_KV_INT4 2      /* symmetric 4-bit codes, two per byte, one fp32 scale per row */
#define DATTN_KV_MIXED 3     /* per KV head: FP8 E4M3 or 4-bit rows (layout.head_format) */

/* Shape of the paged KV pool and the block table. A zero-initialised tail (kv_format 0,
 * NULL scales) is the bf16 pool. */
typedef struct dattn_kv_layout {
    int32_t num_pages;          /* physical pages in the pool */
    int32_t num_kv_heads;       /* Hkv */
    int32_t head_dim;           /* d: 64 or 128 */
    int32_t page_size;          /* P: tokens per physical page, a multiple of 16 */
    const int32_t *block_table; /* (device) [B][max_pages_per_req]; -1 = unmapped */
    int32_t max_pages_per_req;  /* row width of block_table */
    int32_t kv_format;          /* DATTN_KV_BF16, DATTN_KV_FP8_E4M3, DATTN_KV_INT4 or
                                   DATTN_KV_MIXED */
    float *kv_scale;            /* (device) fp32 [num_pages][Hkv][P/16][2][16], 16-byte aligned:
                                   the row scales of the 8-bit and 4-bit formats (ignored for
                                   bf16), written by dattn_kv_append; see the layout notes */
    const int8_t *head_format;  /* (host) [Hkv], read during the call, DATTN_KV_MIXED only:
                                   DATTN_KV_FP8_E4M3 or DATTN_KV_INT4 per KV head; NULL or
                                   another value is DATTN_ERR_INVALID_ARG */
} dattn_kv_layout;

/* Block-sparse decode settings [LV §2.2.2, §3.1.1, §3.1.2]. */
typedef struct dattn_sparse {
    const int8_t *head_kind;  /* (device) [Hkv]: DATTN_HEAD_* per KV head */
    int32_t sinks;            /* streaming heads: tokens [0, min(sinks, L)) */
    int32_t local;            /* streaming heads: tokens [max(sinks, L - local), L) */
    int32_t top_k;            /* retrieval heads: entries per row of selected */
    const int32_t *selected;  /* (device) [B][Hkv][top_k] request-relative physical page
                                 indices from dattn_page_select; -1 entries are ignored.
                                 A page must not appear twice in one row. */
    const int32_t *selected_phys; /* (device, nullable) [B][Hkv][top_k]: the pool pages of
                                 `selected` (block_table[b][selected[..]]), as
                                 dattn_page_select writes them. When given, the decode reads
                                 them instead of looking the pages up in the block table, which
                                 saves a dependent load before the first copy of a step. The
                                 block-table entries of selected pages must then not change
                                 while the selection is in use. */
} dattn_sparse;

/*
 * Append T new tokens per request to the paged pool [LS §4.2: the master saves the new
 * token's KV locally]. If stats is not NULL, also update the logical-page statistics
 * [LV §3.1.2: computed at KV-write time].
 *
 *   k_pool, v_pool (device) the pool in the layout's kv_format; for the 8-bit and 4-bit
 *                formats each row is quantized as described above and its scales go to
 *                layout->kv_scale; for the mixed format each KV head's rows are quantized in
 *                that head's format and go to its region.
 *   k_new, v_new (device) bf16 [B][T][Hkv][d]. Token t of request b is written at
 *                position seq_lens[b] + t.
 *   stats        (device, nullable) bf16 [num_pages][Hkv][P/16][2][d]. When a token
 *                opens a logical page (position % 16 == 0), that page's k_max and k_min
 *                are set to its key. Later tokens update them elementwise with strict
 *                comparison, so on a tie the earlier value stays.
 *   seq_lens     (device) int32 [B]. On entry, the current lengths; on exit, each is
 *                increased by T. When T > 49 the update runs as a second small kernel on
 *                the same stream.
 *   dev_err      (device, nullable) int32 error word, see DATTN_DEVERR_*. A token whose
 *                page is unmapped or out of range is not written.
 * Returns DATTN_OK or an error status; nothing is launched on error.
 */
dattn_status_t dattn_kv_append(const dattn_kv_layout *layout, void *k_pool,
                               void *v_pool, dattn_bf16 *stats, const dattn_bf16 *k_new,
                               const dattn_bf16 *v_new, int32_t B, int32_t T,
                               int32_t *seq_lens, int32_t *dev_err, void *stream);

/*
 * MicroAttention partials over explicit chunks of pages [IL, DistAttention 的等价数学变换].
 * Chunk c covers the request-relative pages
 * chunk_pages[chunk_page_indptr[c] .. chunk_page_indptr[c+1]) of request chunk_req[c].
 * Only tokens < seq_lens[chunk_req[c]] count. For every chunk c and query head h it writes
 *   m[c][h]  = max s_i (natural-log units),  e[c][h] = sum exp(s_i - m),
 *   MA[c][h][:] = sum exp(s_i - m) v_i.
 * An empty chunk gives m = -inf, e = 0, MA = 0.
 *
 *   k_pool, v_pool (device) the pool in the layout's kv_format
 *   q          (device) bf16 [B][Hq][d]
 *   seq_lens   (device) int32 [B]
 *   chunk_req  (device) int32 [C]
 *   chunk_page_indptr (device) int32 [C+1], non-decreasing, starting at 0. A chunk whose
 *              range is reversed, starts below 0, ends past chunk_page_indptr[C] or holds
 *              more than max_pages_per_req pages is flagged with DATTN_DEVERR_CHUNK_OOB and
 *              left empty; its pages are not read.
 *   chunk_pages (device) int32 [chunk_page_indptr[C]]
 *   m, e       (device) fp32 [C][Hq];  MA (device) fp32 [C][Hq][d]
 *   ws, ws_bytes  workspace, at least dattn_workspace_size(C, Hq, Hkv, d, 0, num_splits)
 *   num_splits number of CTAs the tiles are spread over; 0 = automatic
 */
dattn_status_t dattn_partial(const dattn_kv_layout *layout, const void *k_pool,
                             const void *v_pool, const dattn_bf16 *q, int32_t B,
                             int32_t Hq, float scale, const int32_t *seq_lens, int32_t C,
                             const int32_t *chunk_req, const int32_t *chunk_page_indptr,
                             const int32_t *chunk_pages, float *m, float *e, float *MA,
                             void *ws, size_t ws_bytes, int32_t num_splits, int32_t *dev_err,
                             void *stream);

/*
 * Log-sum-exp aggregation of chunk partials [IL, 结果聚合与通信开销降低]. For request b
 * and query head h it merges the chunks c in [chunk_indptr[b], chunk_indptr[b+1]):
 *   m_g = max m_c,  e_g = sum e_c exp(m_c - m_g),
 *   out = sum MA_c exp(m_c - m_g) / e_g,  MA_g = sum MA_c exp(m_c - m_g).
 * Chunks with m = -inf are empty and add nothing. If every chunk is empty, then
 * out = MA_g = 0, m_g = -inf and e_g = 0. (m_g, e_g, MA_g) is itself a partial, so
 * merges nest.
 *
 *   C            number of chunk rows in m, e and MA
 *   chunk_indptr (device) int32 [B+1]. A range outside [0, C] is clamped and flagged
 *                with DATTN_DEVERR_CHUNK_OOB.
 *   m, e (device) fp32 [C][Hq];  MA (device) fp32 [C][Hq][d]
 *   out  (device, nullable) fp32 [B][Hq][d]
 *   m_g, e_g (device, nullable) fp32 [B][Hq];  MA_g (device, nullable) fp32 [B][Hq][d]
 */
dattn_status_t dattn_merge(int32_t B, int32_t C, int32_t Hq, int32_t head_dim,
                           const int32_t *chunk_indptr, const float *m, const float *e,
                           const float *MA, float *out, float *m_g, float *e_g, float *MA_g,
                           int32_t *dev_err, void *stream);

/*
 * The aggregation of partials gathered from R ranks: the cross-GPU form of DistAttention
 * [IL, 结果聚合与通信开销降低: the instances send their partial results back and they are
 * aggregated; LS §4.2: in multi-master decoding every instance computes local attention
 * over its KV and the results are merged]. Rank r ran dattn_partial over its share of each
 * request's KV pages, one chunk per request, and an all-gather stacked the ranks' partials:
 *   m, e (device) fp32 [R][B][Hq];  MA (device) fp32 [R][B][Hq][d]
 * For request b and query head h the R partials [r][b][h] are merged exactly as dattn_merge
 * merges one request's chunks; a rank that holds none of the request's pages contributes an
 * empty partial (m = -inf), which adds nothing. R = 0 gives the empty result.
 *   out (device, nullable) fp32 [B][Hq][d];  m_g, e_g, MA_g (device, nullable) as dattn_merge
 */
dattn_status_t dattn_merge_gathered(int32_t B, int32_t R, int32_t Hq, int32_t head_dim,
                                    const float *m, const float *e, const float *MA, float *out,
                                    float *m_g, float *e_g, float *MA_g, int32_t *dev_err,
                                    void *stream);

/*
 * Fused single-launch decode: split-KV partials plus merge, dense or block-sparse.
 * Dense (sparse == NULL): every query head of request b attends tokens 0..L_b-1.
 * Block-sparse [LV §2.2.2, §3.1.1]: per KV head kind,
 *   DATTN_HEAD_DENSE      attends all tokens;
 *   DATTN_HEAD_RETRIEVAL  attends the tokens (< L_b) of the pages in sparse->selected;
 *   DATTN_HEAD_STREAMING  attends [0, min(sinks, L)) and [max(sinks, L - local), L).
 * num_splits CTAs (0 = automatic, from the SM count and the work size) each take an equal
 * share of the 16-token tiles of all (request, KV head) pairs. A head whose tiles span
 * several CTAs is merged by the last of them.
 *
 *   k_pool, v_pool (device) the pool in the layout's kv_format
 *   q        (device) bf16 [B][Hq][d];  seq_lens (device) int32 [B]
 *   out      (device) fp32 [B][Hq][d]
 *   m_g, e_g (device, nullable) fp32 [B][Hq]: the merged max (natural-log units) and sum
 *   ws, ws_bytes  workspace of at least dattn_workspace_size(B, Hq, Hkv, d, 0, num_splits)
 */
dattn_status_t dattn_decode(const dattn_kv_layout *layout, const void *k_pool,
                            const void *v_pool, const dattn_bf16 *q, int32_t B,
                            int32_t Hq, float scale, const int32_t *seq_lens,
                            const dattn_sparse *sparse, int32_t num_splits, void *ws,
                            size_t ws_bytes, float *out, float *m_g, float *e_g,
                            int32_t *dev_err, void *stream);

/*
 * Multi-query decode: T new query tokens per request attend the cache causally. This is the
 * step beside decode: [LS] "背景知识与设计动机" splits a long input into chunks processed
 * alongside decoding (chunked prefill), and a speculative or chunked step brings several new
 * tokens at once. The T new tokens of request b are the last T of its L_b = seq_lens[b]
 * tokens (append them first with dattn_kv_append). Query token t (0 <= t < T) attends tokens
 * 0 .. L_b - T + t; one that sees no token (L_b - T + t < 0) gives out = 0, m = -inf, e = 0.
 * The split, the partials and the merge are those of dattn_decode; with T = 1 this is
 * dattn_decode without block sparsity.
 *
 *   q        (device) bf16 [B][T][Hq][d]
 *   out      (device) fp32 [B][T][Hq][d];  m_g, e_g (device, nullable) fp32 [B][T][Hq]
 *   ws, ws_bytes  workspace of at least dattn_workspace_size(B, T * Hq, Hkv, d, 0, num_splits)
 * Besides the common limits it needs g * T <= 8 (the query heads and tokens of one KV head
 * share one tensor-core tile) and returns DATTN_ERR_UNSUPPORTED otherwise; T < 1 is
 * DATTN_ERR_INVALID_ARG.
 */
dattn_status_t dattn_decode_multi(const dattn_kv_layout *layout, const void *k_pool,
                                  const void *v_pool, const dattn_bf16 *q, int32_t B, int32_t T,
                                  int32_t Hq, float scale, const int32_t *seq_lens,
                                  int32_t num_splits, void *ws, size_t ws_bytes, float *out,
                                  float *m_g, float *e_g, int32_t *dev_err, void *stream);

/*
 * One decode step with its append, in one launch: exactly dattn_kv_append of one new token
 * per request (T = 1) followed by dattn_decode, for every pool format (a quantized pool
 * stores the new rows quantized exactly as dattn_kv_append does). [LS §4.2: the master saves
 * the new token's KV locally, then every instance attends over its KV including it.] The new
 * token of request b is written at position seq_lens[b] (and the logical-page statistics take
 * it in when stats is not NULL); the decode attends tokens 0 .. seq_lens[b] (the new one
 * included); on return seq_lens[b] has advanced by one. Outputs, pool, statistics, lengths
 * and error bits are those of the two separate calls. Saving the second launch and the wait
 * between them shortens a step by the append's latency.
 *
 *   k_pool, v_pool, stats, k_new, v_new  as for dattn_kv_append (bf16 [B][1][Hkv][d] new rows)
 *   q, scale, sparse, num_splits, out, m_g, e_g  as for dattn_decode
 *   seq_lens (device) int32 [B]: lengths before the step; advanced by one
 *   ws, ws_bytes  workspace of at least dattn_workspace_size(B, Hq, Hkv, d, 0, num_splits)
 */
dattn_status_t dattn_append_decode(const dattn_kv_layout *layout, void *k_pool, void *v_pool,
                                   dattn_bf16 *stats, const dattn_bf16 *k_new,
                                   const dattn_bf16 *v_new, const dattn_bf16 *q, int32_t B,
                                   int32_t Hq, float scale, int32_t *seq_lens,
                                   const dattn_sparse *sparse, int32_t num_splits, void *ws,
                                   size_t ws_bytes, float *out, float *m_g, float *e_g,
                                   int32_t *dev_err, void *stream);

/*
 * dattn_decode without a workspace argument: the same fused decode as dattn_decode, with its
 * scratch in a fixed 8 MiB device array inside the library instead of in caller memory.
 * The pages have no counterpart to this call; it exists for callers that cannot allocate
 * device memory. Examples: a plugin or custom op handed only its input and output
 * pointers, code running under a framework allocator that owns all device memory, and
 * latency-critical code that cannot risk the device synchronisation cudaMalloc may cause.
 * The call allocates nothing.
 *
 *  - Arguments, outputs and results are those of dattn_decode, minus ws and ws_bytes.
 *  - A problem whose dattn_workspace_size(B, Hq, Hkv, head_dim, 0, num_splits) exceeds
 *    8 MiB (8388608 bytes) is rejected with DATTN_ERR_WORKSPACE before any launch.
 *  - The first call on a device looks up the array's device address and caches it. Make
 *    that first call before any stream capture on that device.
 *  - All calls on a device share the one array, and it keeps the last call's contents. Each
 *    call clears the part that must start at zero, on its own stream. Calls that overlap on
 *    the GPU (unordered streams) race on the array and give wrong results.
 */
dattn_status_t dattn_decode_noalloc(const dattn_kv_layout *layout, const void *k_pool,
                                    const void *v_pool, const dattn_bf16 *q, int32_t B,
                                    int32_t Hq, float scale, const int32_t *seq_lens,
                                    const dattn_sparse *sparse, int32_t num_splits,
                                    float *out, float *m_g, float *e_g, int32_t *dev_err,
                                    void *stream);

/* Block-sparse prefill settings [LV §2.1.1, §2.1.2, §2.2.1]. Key and query blocks are 64
 * tokens: key block kb holds tokens 64*kb .. 64*kb + 63. */
typedef struct dattn_prefill_sparse {
    const int8_t *head_kind;     /* (device) [Hkv]: DATTN_HEAD_* per KV head */
    int32_t sink_blocks;         /* streaming heads: key blocks [0, sink_blocks) ... */
    int32_t local_blocks;        /* ... and the local_blocks key blocks ending at the query's */
    int32_t max_sel;             /* retrieval heads: entries per row of block_lists */
    int32_t qblock_stride;       /* rows of block_lists per (request, KV head) */
    const int32_t *block_lists;  /* (device) [B][Hkv][qblock_stride][max_sel]: row qb lists the
                                    key blocks the queries of block qb attend; -1 entries are
                                    ignored, and a block must not appear twice in one row */
} dattn_prefill_sparse;

/*
 * Block-sparse prefill of a chunk of Tq new tokens per request [LV §2.1.1: the KV history is
 * cut into fixed 64-token blocks and only the chosen blocks are loaded and computed; §2.1.2:
 * streaming heads keep a static Lambda pattern of the initial and the neighbouring blocks,
 * retrieval heads a set of blocks chosen at run time; §2.2.1: a block iterator walks the
 * chosen blocks without branches]. The chunk is the last Tq of the L_b = seq_lens[b] tokens
 * of request b (append it first with dattn_kv_append). Query token t, at position
 * p = L_b - Tq + t in query block qb = p / 64, attends the keys i <= p whose block
 * kb = i / 64 its KV head keeps for qb:
 *   sparse == NULL or DATTN_HEAD_DENSE: every kb <= qb (causal attention);
 *   DATTN_HEAD_STREAMING: kb < sink_blocks, or qb - local_blocks < kb <= qb;
 *   DATTN_HEAD_RETRIEVAL: the blocks listed in row qb of block_lists (blocks after qb add
 *                         nothing); a query that keeps no key gives out = 0, m = -inf, e = 0.
 * One CTA computes one 64-token query block of one query head over all its key blocks, so
 * no workspace is needed.
 *
 *   k_pool, v_pool (device) the pool, bf16 only (DATTN_ERR_UNSUPPORTED for the quantized
 *            formats)
 *   q        (device) bf16 [B][Tq][Hq][d];  seq_lens (device) int32 [B]
 *   out      (device) fp32 [B][Tq][Hq][d]
 *   m, e     (device, nullable) fp32 [B][Tq][Hq]: the row max (natural-log units) and sum,
 *            so a chunk's result merges with others by dattn_merge's equations
 * A seq_len below Tq, or a query block beyond qblock_stride, is flagged with
 * DATTN_DEVERR_LEN_OOB and that query block is skipped (its outputs are left untouched).
 */
dattn_status_t dattn_prefill(const dattn_kv_layout *layout, const void *k_pool,
                             const void *v_pool, const dattn_bf16 *q, int32_t B, int32_t Tq,
                             int32_t Hq, float scale, const int32_t *seq_lens,
                             const dattn_prefill_sparse *sparse, float *out, float *m, float *e,
                             int32_t *dev_err, void *stream);

/*
 * Page scoring and top-K selection for retrieval heads [LV §2.2.2, §3.1.2]. For every
 * request b and KV head h of kind DATTN_HEAD_RETRIEVAL:
 *   logical score  sigma(lp) = max over the g query heads j of
 *                  sum_d max(q_jd * kmax_d, q_jd * kmin_d),
 *                  evaluated in fp32 in a fixed order (deterministic). Each product of two
 *                  bf16 values is exact in fp32, so the evaluation is within
 *                  d * 2^-23 * sum_d |max(q_jd * kmax_d, q_jd * kmin_d)| of the exact score;
 *                  pages whose scores lie within that rounding may be ranked either way;
 *   physical score = max of sigma over its logical pages that hold a token < L_b;
 *   selection      the top_k physical pages by score, ties to the lower page index.
 * They are written in ascending page order to selected[b][h][0..top_k), padded with -1.
 * Rows of heads of other kinds are filled with -1. Call it once per reuse window and pass
 * the result to dattn_decode through dattn_sparse.selected.
 *
 *   stats    (device) bf16 [num_pages][Hkv][P/16][2][d], kept by dattn_kv_append
 *   q        (device) bf16 [B][Hq][d];  seq_lens (device) int32 [B]
 *   head_kind (device) int8 [Hkv];  selected (device) int32 [B][Hkv][top_k]
 *   selected_phys (device, nullable) int32 [B][Hkv][top_k]: the pool page of each selected
 *            page, block_table[b][selected[b][h][i]] (-1 beside -1 entries), for
 *            dattn_sparse.selected_phys
 *   ws, ws_bytes  workspace of at least dattn_workspace_size(B, Hq, Hkv, d, top_k, num_splits)
 * Besides the common limits it needs P/16 to be a power of two (P = 16, 32, 64, 128 or 256)
 * and returns DATTN_ERR_UNSUPPORTED otherwise.
 */
dattn_status_t dattn_page_select(const dattn_kv_layout *layout, const dattn_bf16 *stats,
                                 const dattn_bf16 *q, int32_t B, int32_t Hq,
                                 const int32_t *seq_lens, const int8_t *head_kind,
                                 int32_t top_k, int32_t *selected, int32_t *selected_phys,
                                 void *ws, size_t ws_bytes, int32_t num_splits,
                                 int32_t *dev_err, void *stream);

/*
 * Workspace bytes for dattn_partial (items = C, top_k = 0), dattn_decode (items = B,
 * top_k = 0) and dattn_page_select (items = B, top_k > 0) with the given num_splits
 * (0 = the automatic choice on the current device). Returns 0 for invalid arguments.
 */
size_t dattn_workspace_size(int32_t items, int32_t Hq, int32_t Hkv, int32_t head_dim,
                            int32_t top_k, int32_t num_splits);

/* Zero the workspace (cudaMemsetAsync on the stream). One call before first use suffices. */
dattn_status_t dattn_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* The automatic num_splits for a work size of total_tiles 16-token tiles on the current
 * device: SM count times resident CTAs per SM, capped so a CTA gets at least 16 tiles. */
int32_t dattn_auto_splits(int64_t total_tiles);

/* The balanced split: CTA c of G covers tiles [floor(c*W/G), floor((c+1)*W/G)). */
void dattn_split_range(int64_t total_tiles, int32_t num_splits, int32_t cta, int64_t *begin,
                       int64_t *end);

/* The CTA that owns tile t of W under the balanced split of G CTAs. */
int32_t dattn_split_owner(int64_t tile, int64_t total_tiles, int32_t num_splits);

/* Human-readable name of a status code. */
const char *dattn_status_string(dattn_status_t s);

/* Library version string, e.g. "dattn 0.1.0 sm_103a". */
const char *dattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DATTN_H */
