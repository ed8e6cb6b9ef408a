/*
 * se.h -- C ABI of the attention-scored sparse KV library (single GPU, sm_103a).
 *
 * One data-parallel path shared by sparse-inference serving methods: window
 * queries score the cached keys, each KV head keeps its top entries, retained
 * entries are compacted into fresh pages, Quest-style pages are selected per
 * query, and decode attention runs over the resulting view.
 *
 * Sources (page title -- section):
 *   SparseEngine -- "How it works": hooks finish_step (H2O chunk eviction with
 *       accumulated attention scores, SnapKV selection/eviction after the last
 *       prompt chunk) and build_decode_selection (Quest page selection); the
 *       CacheManager owns layout, position mapping and allocate / write /
 *       update / free; physical eviction rewrites the retained slot mapping and
 *       the context length and returns slots to the allocator; logical
 *       selection only changes what attention reads; View = BuildView(C, I),
 *       o = Attention(q, View).
 *   SparseEngine -- "How it differs": prefix-cache pruning of an application
 *       span [L, R): a policy mask picks positions to keep, applied to idle
 *       blocks only, logical prefix untouched, resident set R' = (R \ T) U I.
 *   KARA -- Method 1 (sliding-window bidirectional scoring of the
 *       compressible window), Method 2 (Token2Chunk), Method 3 (KvLLM on a
 *       paged KV cache, periodic compression of the trailing block).
 *
 * Conventions for every call
 *   - All pointers are device pointers to caller-owned memory unless a
 *     parameter says "host".  The library never allocates device memory;
 *     calls that need scratch space take a caller-provided workspace whose
 *     size the matching *_workspace_size() query returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Argument errors the host can see (NULL pointers,
 *     unsupported shapes, too small a workspace) are returned synchronously
 *     and nothing is launched.
 *   - Errors only the device can see (a free list too short, uneven per-head
 *     counts, an index out of range) are written to the cache's device status
 *     word with first-writer-wins semantics; the call still returns SE_OK.
 *     Every state-changing call checks before it writes, so a call that
 *     reports a device error leaves the cache as it found it.
 *   - Calls on one stream that touch the same cache must not overlap with
 *     calls on another stream.
 */
#ifndef SE_H
#define SE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SE_OK = 0,
  SE_ERR_INVALID_ARG = 1,   /* host: bad pointer / size / mode          */
  SE_ERR_UNSUPPORTED = 2,   /* host: shape or dtype outside this build   */
  SE_ERR_OUT_OF_PAGES = 3,  /* device: free list shorter than needed     */
  SE_ERR_UNEVEN = 4,        /* device: KV heads of a sequence would end
                               with different resident counts            */
  SE_ERR_BUSY = 5,          /* reserved                                  */
  SE_ERR_TIMEOUT = 6,       /* device: a bounded wait gave up            */
  SE_ERR_BOUNDS = 7,        /* device: an index argument out of range    */
  SE_ERR_CUDA = 8           /* host: a CUDA launch or query failed       */
} se_status;

typedef enum { SE_BF16 = 0, SE_F32 = 1 } se_dtype;

/*
 * Paged KV cache descriptor (SparseEngine "How it works": CacheManager
 * state; KARA Method 3: paged KV).  Everything is caller-owned device memory.
 *
 *   k_pool, v_pool  [num_pages][Hkv][page_size][D] of dtype ("HND" pages:
 *                   one (page, head) is one contiguous page_size x D block)
 *   block_table     [B][max_pages_per_seq] int32 physical page of each block
 *                   of a sequence, -1 = none
 *   slot_map        [B][Hkv][max_pages_per_seq*page_size] int32 logical
 *                   position held by each resident slot, -1 past ctx_len
 *   ctx_len         [B] int32 resident entries per KV head (equal for all
 *                   heads of a sequence)
 *   logical_len     [B] int32 logical prefix length (eviction never changes it)
 *   free_list       [num_pages] int32 stack of free page ids, free_list[0 ..
 *                   *free_top) valid, top at the end
 *   free_top        [1] int32
 *   page_refcount   [num_pages] int32 or NULL; a page with count > 1 is busy
 *                   (shared or in flight)
 *   status          [1] int32 device error word, 0 = no error; the caller
 *                   clears it
 *
 * Query heads h map to KV head h / (Hq / Hkv).  Supported: D in {64, 128},
 * page_size 16 (or any power of two <= 64), dtype bf16 or fp32.
 */
typedef struct {
  void* k_pool;
  void* v_pool;
  int32_t* block_table;
  int32_t* slot_map;
  int32_t* ctx_len;
  int32_t* logical_len;
  int32_t* free_list;
  int32_t* free_top;
  int32_t* page_refcount;
  int32_t* status;
  int32_t B, Hq, Hkv, D, page_size, num_pages, max_pages_per_seq;
  int32_t dtype; /* se_dtype */
} se_paged_kv;

/* ------------------------------------------------------------------------ */
/* 1. Window scoring                                                          */
/* ------------------------------------------------------------------------ */
/*
 * se_score_window -- SparseEngine "How it works" (SnapKV / H2O scores at the
 * end of prefill) and KARA Method 1 (bidirectional window scoring).
 *
 * For every sequence b and KV head g, with A_h = softmax_j(q . k_j / sqrt(D))
 * taken over the resident slots j in [attn_lo[b], attn_hi[b]) visible to the
 * query, writes
 *     scores[(b*Hkv + g)*scores_stride + j] (+)= sum_{h in g} sum_q A_h[q, j]
 * for j in [out_lo[b], out_hi[b]) (a sub-range of the attention range).
 * Other entries of `scores` are not touched.
 *
 *   q_win     [B][w][Hq][D] window queries (cache dtype)
 *   q_pos     [B][w] int32 logical positions of the window queries
 *   causal    1: query at position t sees slots whose slot_map <= t;
 *             0: every query sees the whole attention range
 *   accumulate 1: add to scores; 0: overwrite
 *   n_max     host: upper bound of attn_hi[b] - attn_lo[b] over b (sizes the
 *             grid; entries past the real range are masked)
 *   workspace se_score_window_workspace_size(kv, w, n_max) bytes, zeroed
 *             before its first use.  Its start is a control block (per
 *             (sequence, KV head) counters of the one-launch form, below)
 *             that every call leaves zero again, so a workspace is zeroed
 *             once and reused; calls that share a workspace must not
 *             overlap on the GPU.  Its first 8 bytes may hold a limit in
 *             nanoseconds for the kernels' bounded waits (0: 2 s; both the
 *             tensor-core forms read it); a wait that runs out sets
 *             SE_ERR_TIMEOUT in kv->status, records where it was in bytes
 *             [12, 16) (nonzero; the caller reads and clears it) and the
 *             launch winds down -- copies and MMAs in flight are still
 *             waited for, up to 2 s -- without writing further scores.
 * A query that sees no key adds nothing.
 *
 * bf16 with D = 128 runs on the tensor cores: a sweep of row statistics,
 * then a sweep of column sums (two or three launches, each key read twice);
 * fp32 and D = 64 on the CUDA cores.
 */
se_status se_score_window(const se_paged_kv* kv, const void* q_win, int32_t w,
                          const int32_t* q_pos, const int32_t* attn_lo,
                          const int32_t* attn_hi, const int32_t* out_lo,
                          const int32_t* out_hi, int32_t causal, int32_t accumulate,
                          int32_t n_max, float* scores, int64_t scores_stride,
                          void* workspace, size_t workspace_bytes, void* stream);
size_t se_score_window_workspace_size(const se_paged_kv* kv, int32_t w, int32_t n_max);

/*
 * se_score_window_one_launch -- the same scores as se_score_window (same
 * arguments, same workspace size, same control block), with both sweeps in
 * one cooperative launch of one CTA per SM: the keys are cut into waves that
 * fit L2, the column sums of a wave follow its row statistics two waves
 * later, and the rows' softmax denominators are merged across CTAs inside
 * the launch, so every key is read from HBM once.  Needs bf16, D = 128,
 * w * Hq / Hkv <= 256, B <= 128 and key ranges of at least eight 128-key
 * tiles (n_max); otherwise returns SE_ERR_UNSUPPORTED without launching.
 * The workspace's bytes [16, 20) count its calls (they tag each call's
 * merged rows); bytes [64, 64 + 4 B Hkv) are per-(sequence, KV head) tile
 * counters that every call leaves at zero.
 */
se_status se_score_window_one_launch(const se_paged_kv* kv, const void* q_win, int32_t w,
                                     const int32_t* q_pos, const int32_t* attn_lo,
                                     const int32_t* attn_hi, const int32_t* out_lo,
                                     const int32_t* out_hi, int32_t causal, int32_t accumulate,
                                     int32_t n_max, float* scores, int64_t scores_stride,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* 2. Selection                                                               */
/* ------------------------------------------------------------------------ */
typedef enum {
  SE_SELECT_TOPK = 0,       /* pooled top-k + forced range (SnapKV, H2O prefill, Quest) */
  SE_SELECT_KARA_CHUNK = 1, /* Token2Chunk (KARA Method 2)                               */
  SE_SELECT_EVICT_ONE = 2   /* H2O: lowest running score outside the recent window       */
} se_select_mode;

typedef struct {
  int32_t mode;          /* se_select_mode                                          */
  int32_t pool_kernel;   /* TOPK: odd avg-pool kernel, 1 = none                     */
  int32_t k;             /* TOPK: entries kept besides the forced range;
                            KARA_CHUNK: number of discrete candidates               */
  int32_t chunk_budget;  /* KARA_CHUNK: compressible entries retained               */
  float chunk_coef;      /* KARA_CHUNK: chunk score (s_a+s_b)/2 - coef*(b-a)        */
  int32_t budget;        /* EVICT_ONE: evict only while ctx_len > budget            */
  int32_t recent;        /* EVICT_ONE: positions >= logical_len - recent are kept   */
  int32_t n_max;         /* host: upper bound of cand_hi - cand_lo (TOPK, KARA)     */
} se_select_params;

/*
 * se_topk_select -- SparseEngine "How it works" (per-KV-head retention from
 * attention scores; Quest page top-k), KARA Method 1-2, H2O eviction.
 *
 *   scores    [B][Hkv][scores_stride] fp32, indexed by resident slot (TOPK,
 *             KARA_CHUNK) or running scores (EVICT_ONE)
 *   cand_lo/cand_hi [B] candidate slot range; force_lo/force_hi [B] forced
 *             range, kept unconditionally and never a candidate
 *   keep_idx  TOPK / KARA_CHUNK: [B][Hkv][keep_stride] kept slots, ascending;
 *             n_keep[b] = their count (same for every head).
 *             EVICT_ONE: [B][Hkv] victim slot or -1; n_keep may be NULL.
 * TOPK ranks candidates by (avg-pooled score desc, slot asc) -- pooling over
 * [cand_lo, cand_hi) with zero padding -- and keeps the first k (the device
 * ranks by the fp32 window sum, which orders as the mean does).
 * KARA_CHUNK keeps the top-k candidates, adds chunk interiors between
 * consecutive candidates by (chunk score desc, start asc) while they fit
 * chunk_budget, then tops up with the best remaining tokens to exactly
 * chunk_budget.  EVICT_ONE: among slots with position < logical_len - recent,
 * the lowest score (ties: the higher position) when ctx_len > budget.
 */
se_status se_topk_select(const se_paged_kv* kv, const float* scores, int64_t scores_stride,
                         const se_select_params* params, const int32_t* cand_lo,
                         const int32_t* cand_hi, const int32_t* force_lo,
                         const int32_t* force_hi, int32_t* keep_idx, int32_t keep_stride,
                         int32_t* n_keep, void* stream);

/* ------------------------------------------------------------------------ */
/* 3. Physical compaction and prefix pruning                                  */
/* ------------------------------------------------------------------------ */
typedef enum { SE_COMPACT_FRESH_PAGES = 0, SE_COMPACT_MOVE_LAST = 1 } se_compact_mode;

/*
 * se_compact_evict -- SparseEngine "How it works": physical eviction updates
 * the retained slot mapping and the context length and returns slots to the
 * allocator.
 *
 * FRESH_PAGES: keep_idx [B][Hkv][keep_stride] ascending slots in
 *   [first_slot[b], ctx_len[b]), n_keep[b] per head.  Slots below
 *   first_slot[b] stay; from page first_slot[b]/page_size on, the sequence is
 *   rewritten into pages popped from the free list (stack top first, by
 *   ascending sequence then block); the old pages are pushed afterwards in the
 *   same order (a busy page loses one reference instead).  New ctx_len =
 *   first_slot + n_keep; slot_map follows the entries; positions past the new
 *   length become -1.  max_keep (host) bounds n_keep for grid sizing.
 *   A sequence with first_slot[b] = ctx_len[b] and n_keep[b] = 0 is left
 *   untouched (no page moves), so one call can compact a subset of sequences.
 * MOVE_LAST: keep_idx [B][Hkv] victim slot per head (-1 on every head = no
 *   eviction for that sequence): the last resident entry moves into the
 *   victim slot, ctx_len - 1, a page left empty is pushed to the free list.
 *
 * aux (optional) [B][Hkv][aux_stride] fp32 per-slot metadata moved with the
 * entries (H2O running scores); vacated slots get 0.
 * Device errors: SE_ERR_OUT_OF_PAGES, SE_ERR_UNEVEN, SE_ERR_BOUNDS.
 * Workspace: se_compact_evict_workspace_size bytes, zeroed before its first
 * use (MOVE_LAST keeps a count of finished CTAs there that every completed
 * call leaves at zero); calls that share a workspace must not overlap on the
 * GPU.
 */
se_status se_compact_evict(const se_paged_kv* kv, int32_t mode, const int32_t* keep_idx,
                           int32_t keep_stride, const int32_t* n_keep,
                           const int32_t* first_slot, int32_t max_keep, float* aux,
                           int64_t aux_stride, void* workspace, size_t workspace_bytes,
                           void* stream);
size_t se_compact_evict_workspace_size(const se_paged_kv* kv, int32_t max_keep);

/*
 * se_compact_decode -- SnapKV's step after the last prompt chunk (SparseEngine
 * "How it works": physical eviction into fresh pages, then attention over the
 * retained entries through the AttentionView) in one pass over the kept
 * entries.  The cache ends as after se_compact_evict(FRESH_PAGES) with the
 * same keep_idx, keep_stride, n_keep, first_slot, max_keep and aux, and
 * o [B][Hq][D] (cache dtype) holds single-query attention of q [B][Hq][D]
 * over every entry of the compacted sequences, as se_sparse_decode_attn with
 * the dense view computes it after the compaction.  Each kept K/V row is
 * read from HBM once: the kernel stages it in shared memory, copies it to its
 * fresh page and attends over it there.
 *
 * max_entries (host) must be at least every compacted length first_slot[b] +
 * n_keep[b]; a longer sequence is refused on the device (SE_ERR_BOUNDS, cache
 * untouched).  The one-pass kernel runs one cluster of k CTAs per (sequence,
 * KV head), k a power of two up to 16 with at most 512 entries per CTA and at
 * most 152 x 4 CTAs in all; other shapes (and devices where such a cluster
 * does not fit) run the compaction and then the decode attention, with the
 * same results.
 * Workspace: se_compact_decode_workspace_size bytes, zeroed before its first
 * use (the decode part keeps per-unit counters there that every completed
 * call leaves at zero).  Device errors as se_compact_evict(FRESH_PAGES); after
 * one, o is undefined.
 */
se_status se_compact_decode(const se_paged_kv* kv, const int32_t* keep_idx, int32_t keep_stride,
                            const int32_t* n_keep, const int32_t* first_slot, int32_t max_keep,
                            float* aux, int64_t aux_stride, const void* q, void* o,
                            int32_t max_entries, void* workspace, size_t workspace_bytes,
                            void* stream);
size_t se_compact_decode_workspace_size(const se_paged_kv* kv, int32_t max_keep,
                                        int32_t max_entries);

/*
 * se_prune_span -- SparseEngine "How it differs": sparse prefix-cache pruning.
 * For each sequence, T = positions in [L[b], R[b]) and I = {t in T :
 * mask[b*mask_stride + t - L[b]] != 0}; the resident set of every head
 * becomes (Res \ T) U (I n Res), entries inside busy pages (page_refcount > 1)
 * stay whatever the mask says, and logical_len is unchanged.  The sequence is
 * then rewritten as se_compact_evict(FRESH_PAGES) does, from the first slot
 * (over all heads) whose position is >= L[b].  n_busy (optional) [B] receives
 * the number of busy pages in the rewritten region.  Token ids are not
 * needed: the logical prefix is the untouched logical_len / positions.
 * Device errors: SE_ERR_UNEVEN (heads would keep different counts),
 * SE_ERR_OUT_OF_PAGES.
 */
se_status se_prune_span(const se_paged_kv* kv, const int32_t* L, const int32_t* R,
                        const uint8_t* mask, int32_t mask_stride, int32_t* n_busy,
                        float* aux, int64_t aux_stride, void* workspace,
                        size_t workspace_bytes, void* stream);
size_t se_prune_span_workspace_size(const se_paged_kv* kv);

/* ------------------------------------------------------------------------ */
/* 4. Quest page selection                                                    */
/* ------------------------------------------------------------------------ */
/*
 * se_quest_build_meta -- per-page elementwise key min / max (the persistent
 * metadata kept beside the KV state, SparseEngine "How it works").
 * kmin, kmax [num_pages][Hkv][D] (cache dtype); written for every resident
 * page of every sequence, over its resident slots only.
 */
se_status se_quest_build_meta(const se_paged_kv* kv, void* kmin, void* kmax, void* stream);

/*
 * se_quest_page_select -- SparseEngine "How it works" (build_decode_selection:
 * Quest's query-dependent page selection).  For sequence b, KV group g and
 * full block i < nblocks-1:
 *     U = sum_{h in g} sum_d max(q[b,h,d]*kmax[p,g,d], q[b,h,d]*kmin[p,g,d])
 * with p = block_table[b][i]; keeps the top `top_pages` blocks by (U desc,
 * block asc) plus the last block.  page_idx [B][Hkv][top_pages+1] block
 * indices ascending, -1 padded; n_sel (optional) [B] their count.
 * q [B][Hq][D] (cache dtype).  max_blocks (host) bounds nblocks.
 */
se_status se_quest_page_select(const se_paged_kv* kv, const void* kmin, const void* kmax,
                               const void* q, int32_t top_pages, int32_t max_blocks,
                               int32_t* page_idx, int32_t* n_sel, void* workspace,
                               size_t workspace_bytes, void* stream);
size_t se_quest_page_select_workspace_size(const se_paged_kv* kv, int32_t max_blocks);

/*
 * se_quest_decode_step -- one Quest decode step in a single launch
 * (SparseEngine "What it is" / "How it works": Quest page selection, then
 * attention over the selected pages).  Results equal se_quest_page_select
 * followed by se_sparse_decode_attn over the page view: per (b, g) the page
 * bound U over full pages 0 .. nb-2 (nb = ceil(ctx_len / page_size)), the
 * top `top_pages` by (U desc, page asc) plus page nb-1, and single-query
 * attention of q over the tokens of those pages.
 * kmin, kmax [num_pages][Hkv][D] (from se_quest_build_meta or kept current by
 * se_append_kv); q, o [B][Hq][D].  page_idx [B][Hkv][top_pages + 1] (optional)
 * receives the selected pages ascending, -1 padded; n_sel [B] (optional) the
 * count.  No workspace: each (b, g) runs on one cluster of 8 CTAs.
 * Supports bf16, D = 128, Hq / Hkv in {1, 2, 4, 8}, top_pages <= 255 and up
 * to 16384 full pages per sequence; otherwise SE_ERR_UNSUPPORTED (host) or
 * SE_ERR_BOUNDS on the device status (longer context, bad page id).
 */
se_status se_quest_decode_step(const se_paged_kv* kv, const void* kmin, const void* kmax,
                               const void* q, int32_t top_pages, void* o, int32_t* page_idx,
                               int32_t* n_sel, void* stream);

/* ------------------------------------------------------------------------ */
/* 5. Decode attention over a view                                            */
/* ------------------------------------------------------------------------ */
typedef enum { SE_VIEW_DENSE = 0, SE_VIEW_PAGES = 1, SE_VIEW_TOKENS = 2 } se_view;

/*
 * se_sparse_decode_attn -- SparseEngine "How it works": View = BuildView(C, I),
 * o = Attention(q, View).  For query head h of KV group g,
 *     o[b,h] = sum_j softmax_j(q[b,h] . k_j / sqrt(D)) v_j
 * over the view's entries of (b, g):
 *   DENSE   every resident slot [0, ctx_len[b])
 *   PAGES   sel [B][Hkv][sel_stride]: n_sel block indices (-1 = skip); the
 *           resident slots of those blocks
 *   TOKENS  sel [B][Hkv][sel_stride]: n_sel resident slots (-1 = skip)
 * q, o [B][Hq][D] (cache dtype; o rounded from fp32).
 * acc_scores (optional) [B][Hkv][acc_stride] fp32: += sum_{h in g} of this
 * step's softmax weight of each viewed slot (H2O running scores).
 * max_entries (host) bounds the entries of one (b, g) view.
 * workspace se_sparse_decode_attn_workspace_size(kv, max_entries) bytes,
 * zeroed before its first use: it holds per-(b, g) counters of the CTAs that
 * finished, which every call that completes leaves at zero again (zero it
 * anew after a call that set a device error).  Calls that share a workspace
 * must not overlap on the GPU.
 */
se_status se_sparse_decode_attn(const se_paged_kv* kv, const void* q, int32_t view,
                                const int32_t* sel, int32_t sel_stride, int32_t n_sel,
                                int32_t max_entries, void* o, float* acc_scores,
                                int64_t acc_stride, void* workspace, size_t workspace_bytes,
                                void* stream);
size_t se_sparse_decode_attn_workspace_size(const se_paged_kv* kv, int32_t max_entries);

/*
 * se_sparse_decode_attn_static -- the same decode attention as
 * se_sparse_decode_attn, for callers that cannot allocate device memory at
 * the point where they call it: code that runs inside a framework's own
 * allocator-free region (plugins of an inference engine that owns every
 * buffer, hooks that run while a memory pool is locked), embedded runtimes
 * with a fixed memory budget, or callers without a device allocator at all.
 * The pages have no counterpart of this call; it is a deployment variant.
 *
 * Instead of a caller-provided workspace it uses one scratch array of
 * SE_DECODE_STATIC_SCRATCH_BYTES (16 MiB) that the library defines in
 * device memory; every GPU that loads the library holds that array until the
 * process exits.  Arguments are those of se_sparse_decode_attn without the
 * workspace; the caller still owns q, o, sel and acc_scores.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture on the device.
 *   - Calls share the array, which keeps the previous call's contents.
 *     Nothing in it needs to start at zero (each call writes every value it
 *     reads first), but calls that overlap on the GPU -- on different
 *     streams, or on one stream from different host threads without ordering
 *     -- race on it.  Serialize them.
 *   - Returns SE_ERR_UNSUPPORTED, launching nothing, when the call needs more
 *     scratch than the array holds (se_sparse_decode_attn_workspace_size
 *     gives the amount for the same arguments).
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define SE_DECODE_STATIC_SCRATCH_BYTES (16u << 20)
se_status se_sparse_decode_attn_static(const se_paged_kv* kv, const void* q, int32_t view,
                                       const int32_t* sel, int32_t sel_stride, int32_t n_sel,
                                       int32_t max_entries, void* o, float* acc_scores,
                                       int64_t acc_stride, void* stream);

/* ------------------------------------------------------------------------ */
/* Helpers                                                                    */
/* ------------------------------------------------------------------------ */
/*
 * se_append_kv -- SparseEngine "How it works" (CacheManager write): n_new
 * tokens per sequence at slots ctx_len[b] .. ctx_len[b] + n_new - 1 with
 * positions logical_len[b] onward (a decode step is n_new = 1, a prefill
 * chunk is n_new > 1).  Blocks that were empty take fresh pages popped from
 * the free-list top in ascending (b, block) order.  Both lengths grow by
 * n_new.  k_new, v_new [B][n_new][Hkv][D] in the cache dtype (device).
 * aux (optional, [B][Hkv][aux_stride] fp32) gets 0 at the new slots.  kmin,
 * kmax (optional, both or neither) [num_pages][Hkv][D] Quest page bounds kept
 * current: a fresh page starts from its keys, an existing page widens.
 * Host errors: SE_ERR_INVALID_ARG (null buffers, n_new < 0, workspace too
 * small).  Device errors (nothing written): SE_ERR_BOUNDS (a sequence would
 * exceed max_pages_per_seq pages), SE_ERR_OUT_OF_PAGES.
 * Workspace: se_append_kv_workspace_size bytes, zeroed before its first use
 * (it holds a count of finished CTAs that every completed call leaves at
 * zero); calls that share a workspace must not overlap on the GPU.
 */
se_status se_append_kv(const se_paged_kv* kv, const void* k_new, const void* v_new,
                       int32_t n_new, float* aux, int64_t aux_stride, void* kmin, void* kmax,
                       void* workspace, size_t workspace_bytes, void* stream);
size_t se_append_kv_workspace_size(const se_paged_kv* kv);

/*
 * se_release_seqs -- CacheManager "free" of whole sequences (SparseEngine
 * "How it differs": an idle chain's row is reclaimed when capacity is
 * needed).  Every sequence b with mask[b] != 0 (device int32 [B]) gives back
 * all its pages: pushed onto the free list in ascending (sequence, block)
 * order, except pages whose reference count is above one, which only lose
 * this sequence's reference.  Counts are judged as they were before the
 * call: release sequences that share pages in separate calls.  Block table
 * and slot map rows become -1, ctx_len and logical_len 0.
 * Device error (nothing written): SE_ERR_BOUNDS for a page id >= num_pages.
 */
se_status se_release_seqs(const se_paged_kv* kv, const int32_t* mask, void* workspace,
                          size_t workspace_bytes, void* stream);
size_t se_release_seqs_workspace_size(const se_paged_kv* kv);

/*
 * Chain index -- SparseEngine "How it differs" (Chain Cache): ties each
 * session (chain_id) to the sequence row of the paged cache holding its
 * retained KV and to its logical token prefix.  Host memory and host work
 * only; every call on one index is serialised internally.
 *   se_chain_acquire  for a request's tokens (host int32 [n_tokens]): resumes
 *       the idle chain whose prefix is the longest prefix of the tokens (ties:
 *       most recently used) -- *reuse_len = that prefix's length, prefill only
 *       tokens[reuse_len:] -- or starts a chain on the lowest free row, or on
 *       the row of the least recently used idle chain, which is dropped
 *       (*reclaimed_row = that row, else -1: release its pages with
 *       se_release_seqs first).  SE_ERR_BUSY when every row serves a request.
 *   se_chain_finish   the request on chain_id ended; its logical prefix is now
 *       tokens (prompt and generated tokens); the chain becomes idle.
 *   se_chain_drop     forgets an idle chain; *row = its row (now free).
 * Invalid handles, ids or busy chains: SE_ERR_INVALID_ARG.
 */
typedef struct se_chain_index se_chain_index;
se_chain_index* se_chain_index_create(int32_t n_rows);
void se_chain_index_destroy(se_chain_index* idx);
se_status se_chain_acquire(se_chain_index* idx, const int32_t* tokens, int64_t n_tokens,
                           int64_t* chain_id, int32_t* row, int64_t* reuse_len,
                           int32_t* reclaimed_row);
se_status se_chain_finish(se_chain_index* idx, int64_t chain_id, const int32_t* tokens,
                          int64_t n_tokens);
se_status se_chain_drop(se_chain_index* idx, int64_t chain_id, int32_t* row);
int32_t se_chain_count(se_chain_index* idx);

/* Human-readable name of a status code (static string). */
const char* se_status_string(int32_t status);

/* Library version: major*10000 + minor*100 + patch. */
int32_t se_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SE_H */
