/*
 * ppa.h -- chunked-prefill attention over a paged KV cache, for NVIDIA GB300 (sm_103a).
 *
 * One batch of sequences is processed per call. Sequence b has c = context_lens[b] cached
 * tokens and n = cu_query_lens[b+1] - cu_query_lens[b] new query tokens, so s = c + n keys.
 * Query token j of sequence b sits at absolute position q = c + j. Key positions p < c are
 * read from the paged cache through the block table, one token at a time: physical page
 * block_table[b][p / P], slot p % P. Key positions p >= c are read from k_new / v_new, or,
 * with PPA_FLAG_KV_IN_CACHE, from the cache as well (after ppa_append_kv wrote them there).
 * Tiles of keys may therefore straddle page boundaries, and P may be any positive integer.
 * Sources: vLLM PR #54194 report (prefix-prefill tiles decoupled from the page size),
 * sections "功能与动机" and "关键源码片段" (context_attention_fwd, _paged_kv_cache_offsets).
 *
 * Mask: a query at q may attend to key k (0 <= k < s) iff base(q,k) OR mm(q,k).
 *   base: (causal ? k <= q : (window_right <= 0 || k - q < window_right))
 *         && (chunk_size > 0 ? k >= ((q / chunk_size) - chunk_lookback) * chunk_size
 *                            : (window_left <= 0 || q - k < window_left))
 *         with `causal` per sequence when ppa_dims.seq_causal is given
 *   mm:   some range [a, e] of the sequence with a < e has a <= q <= e' and a <= k <= e',
 *         with e' = min(e, s - 1), and, when PPA_FLAG_CLAMP_MM is set and window_left > 0,
 *         also q - k < window_left.
 * Sources: "[Kernel][Gemma4] Prune Triton sliding-window tiles for multimodal prefixes"
 * (PR #53147), sections "实现拆解" 1-2 and "关键源码片段" (compute_tile_loop_bounds); and
 * "[Kernel] Skip fully masked key blocks in windowed Triton prefill" (PR #50776), section
 * "关键源码片段" (separate left/right windows, 0 = off).
 *
 * Output: out[q, h] = sum_k softmax_k(sm_scale * <Q[q,h], K[k, h/G]>) V[k, h/G] over the
 * allowed keys, where G = num_q_heads / num_kv_heads (query heads g*G .. g*G+G-1 share KV
 * head g; PR #53147 "关键源码片段", BLOCK_M = BLOCK_Q * num_queries_per_kv).
 * Key tiles that hold no allowed pair are never loaded (PR #50776 "功能与动机"; PR #53147
 * "实现拆解" 2): a first stage computes the exact interval of live key tiles per query tile.
 *
 * Tensor layouts (row-major, element offsets in elements of the stated type):
 *   q            [total_q][num_q_heads][head_dim]            bf16
 *   k_new, v_new [total_q][num_kv_heads][head_dim]           bf16
 *   k_cache,
 *   v_cache      [num_pages][page_size][num_kv_heads][head_dim]  bf16 or fp8 e4m3fn (1 byte)
 *   block_table  [num_seqs][max_pages_per_seq]                int32, physical page ids
 *   cu_query_lens[num_seqs + 1]                              int32, cu[0] = 0, cu[B] = total_q
 *   context_lens [num_seqs]                                  int32, >= 0
 *   mm_ranges    [num_seqs][max_mm_ranges][2]                int32 {start, end}, end inclusive;
 *                                                            entries with start >= end are unused
 *   out          [total_q][num_q_heads][head_dim]            bf16
 * Only the first ceil(c / P) entries of a block-table row are ever read (ceil((c + n) / P)
 * with PPA_FLAG_KV_IN_CACHE, and by ppa_append_kv).
 *
 * Ownership and synchronisation: every pointer is a device pointer owned by the caller.
 * The library allocates nothing, never frees, never synchronises inside ppa_prefill, and
 * runs all work on `stream` (a cudaStream_t passed as void*; NULL = legacy default stream).
 * Argument errors found on the host return a status at once and launch nothing. Errors found
 * on the device (bad lengths, a page id outside [0, num_pages), an expired bounded wait) are
 * written to the caller's int32 `device_status` (first error wins). The kernels then skip
 * the affected work instead of faulting; ppa_read_status() reports the code.
 */
#ifndef PPA_H_
#define PPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PPA_OK = 0,
  PPA_ERR_INVALID = 1,     /* bad argument (host) or bad lengths found on the device */
  PPA_ERR_UNSUPPORTED = 2, /* head_dim / group size / dtype / path with no kernel in this build */
  PPA_ERR_CUDA = 3,        /* a CUDA runtime call failed (launch, copy, attribute) */
  PPA_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired; the kernel returned early */
  PPA_ERR_BAD_PAGE = 5     /* a block-table entry outside [0, num_pages); rows read as zero */
} ppa_status;

enum { PPA_KV_BF16 = 0, PPA_KV_FP8_E4M3 = 1 };

enum {
  PPA_FLAG_CAUSAL = 1u,   /* base mask is causal (k <= q); window_right is then ignored */
  PPA_FLAG_CLAMP_MM = 2u, /* multimodal keys also obey the left window (q - k < window_left) */
  PPA_FLAG_NO_PRUNE = 4u, /* testing: visit every key tile 0 .. ceil(s/TN)-1 and mask them */
  PPA_FLAG_FP8_INKERNEL = 8u, /* fp8 caches: widen e4m3 rows inside the attention kernel
                               * instead of dequantising the live cache tiles into workspace
                               * first; the workspace then needs no bf16 scratch (ignored for
                               * bf16 caches) */
  PPA_FLAG_KV_IN_CACHE = 16u  /* the new tokens' K/V are already in the cache at positions
                               * c .. c+n-1 (for instance written by ppa_append_kv): attention
                               * reads them from there and k_new / v_new are not read (NULL is
                               * allowed); block-table rows must then cover c + n positions */
};

typedef struct {
  int num_seqs;          /* B >= 0 */
  int total_q;           /* sum of query lengths, >= 0 */
  int num_q_heads;       /* Hq >= 1 */
  int num_kv_heads;      /* Hkv >= 1, Hq % Hkv == 0, Hq / Hkv <= 128 */
  int head_dim;          /* D: 64, 128 or 256 */
  int page_size;         /* P >= 1, any integer */
  int num_pages;         /* physical pages in each cache tensor, >= 1 */
  int max_pages_per_seq; /* block-table row length, >= 1 */
  int max_mm_ranges;     /* R >= 0; mm_ranges may be NULL when 0 */
  int window_left;       /* <= 0: unbounded on the left */
  int window_right;      /* <= 0: unbounded on the right (ignored when causal) */
  int kv_dtype;          /* PPA_KV_BF16 or PPA_KV_FP8_E4M3 */
  unsigned flags;        /* PPA_FLAG_* */
  float sm_scale;        /* softmax scale; <= 0 selects 1/sqrt(head_dim) */
  int chunk_size;        /* > 0: chunked-local attention, 0: off. The base mask's left edge is
                          * k >= ((q / chunk_size) - chunk_lookback) * chunk_size instead of the
                          * left window (window_left then only clamps multimodal ranges); the
                          * CHUNK_LOOKBACK branch of compute_tile_loop_bounds, "[Kernel][Gemma4]
                          * Prune Triton sliding-window tiles for multimodal prefixes",
                          * 关键源码片段, read per pair */
  int chunk_lookback;    /* >= 0: earlier chunks that stay visible (with chunk_size > 0) */
  int kv_split_tiles;    /* > 0: split-KV. A sequence whose new tokens fit one query tile
                          * (decode, speculative verification) and whose live keys span more
                          * than this many 128-key tiles is cut into segments of this many
                          * tiles, attended in parallel and merged by their log-sum-exps
                          * (the segmented mode the PR #53147 page names, tiles_per_segment).
                          * 0: off. -1: the library's tuned segment length (32 tiles). The
                          * workspace then holds the partial results. */
  const int32_t* seq_causal; /* NULL, or a device array of num_seqs int32: sequence b's base
                              * mask is causal iff seq_causal[b] != 0, overriding
                              * PPA_FLAG_CAUSAL (per-sequence causality, USE_PER_SEQ_CAUSAL on
                              * the multimodal-pruning page). Read on the device by ppa_plan,
                              * ppa_attend and the mask/count entry points. */
  int max_cache_tokens;  /* fp8 caches dequantised into workspace (no PPA_FLAG_FP8_INKERNEL):
                          * > 0 sizes the bf16 staging by this bound instead of by every
                          * block-table slot: at least the number of cached positions the
                          * batch's queries may attend to, summed over sequences (the sum of
                          * context_lens always suffices; windows make it smaller). Only the
                          * key tiles those positions fall in are staged. If they need more
                          * room on the device, the call stores PPA_ERR_INVALID and computes
                          * nothing. 0: room for every block-table slot. */
} ppa_dims;

/* Bytes of device workspace ppa_prefill needs for `dims` (query-tile table and work list; with
 * multimodal ranges (max_mm_ranges > 0) also 8 bytes per query token: each row's allowed key
 * interval, written by ppa_plan so that the attention kernel does not rescan the ranges).
 * For an fp8 cache without PPA_FLAG_FP8_INKERNEL it also holds the bf16 scratch that the live
 * cache key tiles are dequantised into before the attention kernel runs: tiles of 128
 * positions for K and for V (2 * 128 * num_kv_heads * head_dim * 2 bytes per tile), as many
 * as floor(max_cache_tokens / 128) + 2 * num_seqs when max_cache_tokens > 0 (the live
 * positions of a sequence are consecutive, so they touch at most that many tiles), else
 * num_seqs * ceil(max_pages_per_seq * page_size / 128), never more than the latter; plus a
 * table of num_seqs * ceil(max_pages_per_seq * page_size / 128) int32 and a bitmap.
 * If that bf16 staging does not fit the int32 row range, it is dropped and the fp8 path widens
 * in the kernel, as with the flag.
 * Returns 0 if dims is NULL or invalid. The caller allocates it; contents need no
 * initialisation and may be reused across calls on the same stream. */
size_t ppa_workspace_bytes(const ppa_dims* dims);

/* The attention forward pass. Pointers as in the layout table above; k_scale / v_scale are
 * device pointers to one fp32 each (the per-tensor dequantisation scales), required when
 * kv_dtype is PPA_KV_FP8_E4M3 and ignored otherwise. k_new / v_new must be non-NULL unless
 * PPA_FLAG_KV_IN_CACHE is set (then they are not read). q, k_new, v_new, k_cache, v_cache
 * and out must be 16-byte aligned. Launches two stages on `stream`: ppa_plan (the
 * live-tile bounds and work list) and ppa_attend (the persistent attention kernel). */
ppa_status ppa_prefill(const ppa_dims* dims, const void* q, const void* k_new, const void* v_new,
                       const void* k_cache, const void* v_cache, const int32_t* block_table,
                       const int32_t* cu_query_lens, const int32_t* context_lens,
                       const int32_t* mm_ranges, const float* k_scale, const float* v_scale,
                       void* out, void* workspace, int32_t* device_status, void* stream);

/* The two stages of ppa_prefill, callable separately so that one plan serves every layer of
 * a batch (the lengths, ranges and mask parameters do not change between layers).
 *
 * ppa_plan (stage 1): validates the lengths on the device, computes every query tile's
 * live key-tile interval and the work list (heaviest tiles first) into `workspace`, and,
 * with multimodal ranges, every query token's allowed key interval.
 *
 * ppa_attend (stage 2): the attention kernel over the work list in `workspace`. The
 * workspace must hold a plan made by ppa_plan for the same dims and the same
 * cu_query_lens / context_lens / mm_ranges contents; the plan is left intact, so any number
 * of ppa_attend calls may follow one ppa_plan on the same stream. Calls that share a
 * workspace must not overlap in time (they share its work-stealing counter). */
ppa_status ppa_plan(const ppa_dims* dims, const int32_t* cu_query_lens,
                    const int32_t* context_lens, const int32_t* mm_ranges, void* workspace,
                    int32_t* device_status, void* stream);

ppa_status ppa_attend(const ppa_dims* dims, const void* q, const void* k_new, const void* v_new,
                      const void* k_cache, const void* v_cache, const int32_t* block_table,
                      const int32_t* cu_query_lens, const int32_t* context_lens,
                      const int32_t* mm_ranges, const float* k_scale, const float* v_scale,
                      void* out, void* workspace, int32_t* device_status, void* stream);

/* KV append: writes the new tokens' K/V into the paged cache, where the cache-sourced path
 * (PPA_FLAG_KV_IN_CACHE; the k=None path of the PR #54194 report, 实现拆解 item 4) reads
 * them. The pages print no append code; this is its plain reading. New token j of sequence
 * b (row cu_query_lens[b] + j of k_new / v_new) is written to position
 * c = context_lens[b] + j of the sequence: page block_table[b][c / page_size], slot
 * c % page_size, all KV heads. A bf16 cache takes the values unchanged. An fp8 cache takes, per
 * element, the E4M3 code nearest to value / scale (the quotient in fp32; ties to the even code;
 * magnitudes past 448 saturate to 448; NaN stays NaN), with k_scale / v_scale device
 * pointers to one fp32 each. Nothing else in the caches changes.
 * Host-side errors (NULL or misaligned pointers, invalid dims) return before any launch. On
 * the device, a sequence with invalid lengths, or whose new positions pass its block-table
 * row, writes nothing and sets PPA_ERR_INVALID in *device_status; a page id outside
 * [0, num_pages) skips that token and sets PPA_ERR_BAD_PAGE. k_new, v_new, k_cache and
 * v_cache must be 16-byte aligned. Launches one kernel on `stream`. */
ppa_status ppa_append_kv(const ppa_dims* dims, const void* k_new, const void* v_new,
                         void* k_cache, void* v_cache, const int32_t* block_table,
                         const int32_t* cu_query_lens, const int32_t* context_lens,
                         const float* k_scale, const float* v_scale, int32_t* device_status,
                         void* stream);

/* Size of the scratch ppa_prefill_noalloc keeps in a static device array: 2 MiB. The scratch a
 * batch needs is ppa_workspace_bytes(): about 36 + 4 * num_kv_heads bytes per query tile plus 16
 * bytes per sequence, so 2 MiB holds, for example, about 30,000 query tiles at 8 KV heads
 * (more with multimodal ranges or split-KV, whose extra scratch counts too). */
#define PPA_NOALLOC_WORKSPACE_BYTES (2u << 20)

/* ppa_prefill for callers that cannot allocate device memory: no workspace argument.
 * The paged-attention pages have no counterpart of this entry point; it exists for callers
 * such as a plugin inside a host framework that owns the whole device memory pool and gives
 * its plugins no allocator, or a runtime that forbids device allocation after start-up to
 * keep a fixed memory footprint. The scratch ppa_prefill would take from `workspace` lives
 * instead in one file-scope device array of PPA_NOALLOC_WORKSPACE_BYTES, which every GPU that
 * loads the library holds until the process exits. This call allocates and frees nothing.
 *   - Inputs, `out` and `device_status` are the caller's, exactly as for ppa_prefill.
 *   - fp8 caches are widened inside the attention kernel (as with PPA_FLAG_FP8_INKERNEL)
 *     and kv_split_tiles is ignored: the dequantisation staging and the split partials do
 *     not fit the fixed scratch. The output is the same attention either way.
 *   - A batch whose ppa_workspace_bytes() (for those settings) exceeds
 *     PPA_NOALLOC_WORKSPACE_BYTES is rejected with PPA_ERR_UNSUPPORTED before anything is
 *     launched (use ppa_prefill for it).
 *   - The first call on each device looks up that device's address of the array (with the
 *     device current) and caches it; make that first call before any stream capture.
 *   - All calls on a device share the one array. Calls whose work overlaps on the GPU (other
 *     streams, other host threads without ordering) race on it and give wrong results; calls
 *     ordered on one stream are safe. Each call rewrites every scratch word it reads, so
 *     leftovers of the previous call need no clearing. */
ppa_status ppa_prefill_noalloc(const ppa_dims* dims, const void* q, const void* k_new,
                               const void* v_new, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, const int32_t* cu_query_lens,
                               const int32_t* context_lens, const int32_t* mm_ranges,
                               const float* k_scale, const float* v_scale, void* out,
                               int32_t* device_status, void* stream);

/* The tile shape ppa_prefill uses for `dims`: tq query tokens per query tile (so tq * G <= 128
 * rows) and tn keys per key tile. Writes 0 to both if dims is invalid. */
void ppa_query_tiles(const ppa_dims* dims, int* tq, int* tn);

/* Stage 1 alone, for testing: for every (sequence, query tile of tq tokens) in order, writes
 * {lo, hi} (int32 pairs) such that key tiles lo .. hi-1 of width tn are exactly those holding
 * an allowed pair (PR #53147 "关键源码片段", compute_tile_loop_bounds; we use the first query
 * row for the window edge). bounds_out must hold 2 * sum_b ceil(n_b / tq) ints. */
ppa_status ppa_tile_bounds(const ppa_dims* dims, int tq, int tn, const int32_t* cu_query_lens,
                           const int32_t* context_lens, const int32_t* mm_ranges,
                           int32_t* bounds_out, int32_t* device_status, void* stream);

/* Testing: the allowed-pair bitmap of sequence `seq` as the attention kernel evaluates it:
 * bit (k % 32) of word bitmap[j * words_per_row + k / 32] is set iff query token j may attend
 * to key k. Rows j < min(n, max_rows) are written, words beyond ceil(s/32) are zeroed. */
ppa_status ppa_debug_mask(const ppa_dims* dims, int seq, const int32_t* cu_query_lens,
                          const int32_t* context_lens, const int32_t* mm_ranges,
                          uint32_t* bitmap_out, int max_rows, int words_per_row, void* stream);

/* Number of allowed (query token, key) pairs summed over the batch, for one head; written
 * to the device uint64 *count_out. Live-pair FLOPs are 4 * D * Hq * count. */
ppa_status ppa_live_pairs(const ppa_dims* dims, const int32_t* cu_query_lens,
                          const int32_t* context_lens, const int32_t* mm_ranges,
                          unsigned long long* count_out, void* stream);

/* Number of cached context tokens (positions k < c) that at least one query of their sequence
 * may attend to, summed over the batch, written to the device uint64 *count_out. These are
 * the cache rows one prefill pass must read at least once (one KV head); the algorithmic HBM
 * bytes of a pass count each of them once per KV head for K and for V. */
ppa_status ppa_live_kv_tokens(const ppa_dims* dims, const int32_t* cu_query_lens,
                              const int32_t* context_lens, const int32_t* mm_ranges,
                              unsigned long long* count_out, void* stream);

/* Testing: decodes n fp8 e4m3fn codes to bf16 bit patterns with the attention kernel's own
 * conversion (exact; NaN codes give a bf16 NaN). */
ppa_status ppa_debug_e4m3_to_bf16(const uint8_t* codes, uint16_t* bf16_out, int n, void* stream);

/* Testing the bounded device-side waits without a fault. Every wait inside the attention
 * kernels is bounded; when one runs out, the kernel stores PPA_ERR_TIMEOUT in *device_status,
 * every warp leaves its loop, the copies still in flight are waited for (bounded again), the
 * tensor-core operations retire, TMEM is freed and the kernel returns, so the context stays
 * usable and the next call on the stream runs normally. This entry point runs ppa_prefill
 * (same arguments) with every such wait limited to wait_limit_us microseconds (> 0), and
 * with the query loader of the CTA that takes the plan's first work item never loading that
 * item's query tiles nor fetching further work: the waits for them run out. The output is then unspecified. Head dims 64 and 128 (the
 * single-CTA kernel) only; head_dim 256 returns PPA_ERR_UNSUPPORTED. The pages have no
 * counterpart of this entry point: it exercises the library's own failure path. */
ppa_status ppa_debug_prefill_stalled(const ppa_dims* dims, const void* q, const void* k_new,
                                     const void* v_new, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* cu_query_lens,
                                     const int32_t* context_lens, const int32_t* mm_ranges,
                                     const float* k_scale, const float* v_scale, void* out,
                                     void* workspace, int32_t* device_status,
                                     unsigned wait_limit_us, void* stream);

/* Synchronises `stream`, returns the code stored in *device_status and clears it to 0.
 * Returns PPA_ERR_CUDA if the synchronisation or the copy fails. */
ppa_status ppa_read_status(int32_t* device_status, void* stream);

/* Static text for a status code. */
const char* ppa_status_string(ppa_status status);

/* Library version (major * 10000 + minor * 100 + patch). 0.2.0 added ppa_append_kv, the
 * PPA_FLAG_FP8_INKERNEL and PPA_FLAG_KV_IN_CACHE flags, and the ppa_dims fields chunk_size,
 * chunk_lookback and seq_causal. 0.3.0 inserted kv_split_tiles before seq_causal and appended
 * max_cache_tokens to ppa_dims (layout changes: callers built against 0.2 must rebuild), and
 * added kv_split_tiles = -1, ppa_prefill_noalloc and ppa_debug_prefill_stalled. */
#define PPA_VERSION 300
int ppa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PPA_H_ */
