/*
 * quest.h - C ABI of libquest.so, Quest's decode-time hot path on GB300 (sm_103a).
 *
 * Quest (Tang et al., ICML 2024) keeps the whole paged KV cache, summarises every page
 * by the per-dimension minimum and maximum of its keys, scores each page against the
 * current query with an upper bound on q.k, keeps the K best pages per head, and runs
 * exact attention over those pages only.  Sources, cited below by title:
 *   [Guide]   "Guide to Quest: Query-Aware KV Cache Sparsity for LLMs"
 *   [Summary] "Quest: Query-Aware Sparsity for Efficient Long-Context LLM Inference"
 *             (Tang 2024 paper summary page)
 *   [Project] the sourcepulse project page of the published implementation
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer in quest_cache_t and every tensor argument is a DEVICE pointer owned
 *   by the caller.  The library allocates no memory and keeps no state except a
 *   thread-local error string.  All tensors are dense, row-major, 16-byte aligned.
 * - fp16 means IEEE binary16.  head_dim must be 128, page_size 16 or 32, and
 *   num_q_heads / num_kv_heads (the group size G) one of 1, 2, 4, 8.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream)
 *   and return a status code.  A non-zero code from the host-side checks means nothing
 *   was launched.  quest_last_error() describes the last failure of this thread.
 * - Faults that only the device can see (a block-table entry outside [0, num_phys), a
 *   sequence length outside [0, max_pages * page_size], an inter-CTA wait that ran out)
 *   never trap: the kernel skips the offending page, records the first such fault in the
 *   workspace status word and finishes.  quest_read_status() synchronises the stream,
 *   returns that code and clears it.  Outputs of a call that recorded a fault are
 *   unspecified; re-initialise the workspace (quest_workspace_init) after one.
 * - The workspace is caller-owned device scratch of quest_workspace_size() bytes.  It
 *   must be zeroed once before first use (quest_workspace_init) and is then reused
 *   across calls: its counters return to zero at the end of each call.  Calls that share
 *   one workspace must be ordered (same stream, or events); concurrent calls need
 *   separate workspaces.
 */
#ifndef QUEST_H
#define QUEST_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QUEST_VERSION 1

/* Status codes. */
#define QUEST_OK 0
#define QUEST_ERR_INVALID_ARG 1   /* null / misaligned pointer, negative size, bad top_k  */
#define QUEST_ERR_UNSUPPORTED 2   /* head_dim != 128, page_size not 16/32, G not 1/2/4/8,
                                     max_pages above QUEST_MAX_PAGES                        */
#define QUEST_ERR_WORKSPACE 3     /* workspace null or smaller than quest_workspace_size() */
#define QUEST_ERR_CUDA 4          /* a CUDA runtime call failed (message in last_error)    */
#define QUEST_ERR_TIMEOUT 5       /* device: a bounded inter-CTA wait ran out              */
#define QUEST_ERR_BAD_PAGE 6      /* device: block-table entry outside [0, num_phys)       */
#define QUEST_ERR_BAD_LENGTH 7    /* device: seq_len outside [0, max_pages * page_size], or
                                     an append into a row with no room                      */
#define QUEST_ERR_BAD_SELECTION 8 /* device: quest_sparse_decode got a page index outside
                                     [0, N_b) or a count outside [0, min(top_k, N_b)]        */

/* Largest block-table row (pages per sequence) the selection kernels hold on chip. */
#define QUEST_MAX_PAGES 16384

typedef void* quest_stream_t; /* cudaStream_t */

/*
 * One layer's paged KV cache ([Guide] Implementation step 1: physical K/V pages,
 * per-page key min/max, block table and per-sequence page counts; here lengths are
 * kept in tokens).
 *   k_pool, v_pool : fp16 [num_phys][num_kv_heads][page_size][128]; token t of sequence
 *                    b lives in physical page block_table[b][t / page_size], slot
 *                    t % page_size.  One (page, kv head) chunk is contiguous.
 *   meta           : fp16 [batch][num_kv_heads][max_pages][2][128]: for logical page p of
 *                    sequence b and kv head g, the per-dimension key minimum (row 0) and
 *                    maximum (row 1) over the tokens present ([Guide] Solution step 1).
 *                    Boxes are kept per sequence in logical page order (not per physical
 *                    page) so that scoring streams them contiguously without the block
 *                    table.
 *   block_table    : int32 [batch][max_pages], logical page -> physical page.  Entries at
 *                    or past ceil(seq_len / page_size) are never read, except the page a
 *                    call's new tokens go to (quest_append, quest_prefill, the decode
 *                    calls that append).
 *   seq_lens       : int32 [batch], tokens present; written by quest_append,
 *                    quest_prefill and the decode calls that append.
 */
typedef struct quest_cache {
    int32_t batch;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t page_size;
    int32_t max_pages;
    int32_t num_phys;
    void* k_pool;
    void* v_pool;
    void* meta;
    const int32_t* block_table;
    int32_t* seq_lens;
} quest_cache_t;

/* Optional launch tuning (pass NULL for defaults).  Results do not depend on it beyond
 * floating-point rounding of the split-K merge. */
typedef struct quest_opts {
    int32_t pages_per_split;  /* selected pages per decode work item (default: about 8 work
                                 items per (sequence, kv head), at least 16 pages; dense
                                 decode: at least 8)                                         */
    int32_t score_tile_pages; /* pages per scoring work item (default 128)                */
    int32_t max_ctas;         /* one-launch kernels: cap on persistent CTAs (cluster kernel:
                                 clusters; stream kernel: CTAs) (0 = all that fit)          */
    int32_t debug_flags;      /* QUEST_DEBUG_* (0 in normal use)                          */
    int64_t wait_limit_ns;    /* bound on any inter-CTA wait (default 1e9 ns)             */
    int32_t reserved;         /* must be 0                                                */
    int32_t trace_capacity;   /* one-launch kernels: records `trace` can hold             */
    uint64_t* trace;          /* one-launch kernels: optional device timeline, NULL = off;
                                 zero it before the call.  Record i is trace[1 + 2i] =
                                 %globaltimer ns, trace[2 + 2i] = smid << 48 | cta << 32 |
                                 event << 24 | item; unused records stay 0.  CTA c owns
                                 records [64c, 64c + 64) (cluster kernel) or
                                 [256c, 256c + 256) (stream kernel).                        */
    int32_t cluster_size;     /* fused kernel: CTAs per (sequence, kv head) cluster, 1..16;
                                 0: the largest size up to 8 at which every pair's cluster
                                 is resident at once (1 when there are more pairs than SMs
                                 can hold)                                                  */
    int32_t sink_pages;       /* quest_topk / quest_decode*: the first sink_pages pages of   */
    int32_t local_pages;      /* a sequence longer than top_k pages, and its last
                                 local_pages pages, are always kept; the other
                                 top_k - sink_pages - local_pages slots go to the best of
                                 the rest ([Guide] Solution step 3, third bullet;
                                 Implementation step 2).  0 and 0 (the default): plain
                                 top-K.  Needs sink_pages, local_pages >= 0 and
                                 sink_pages + local_pages <= top_k (QUEST_ERR_INVALID_ARG) */
    int32_t gqa_union;        /* the union form of the group-level selection ([Guide] Best
                                 Practices step 2): each query head keeps its top_k pages and
                                 the kv head keeps their union, in selection rows of
                                 min(G * top_k, max_pages) entries.  quest_topk: scores are
                                 per query head ([batch][num_q_heads][max_pages],
                                 quest_estimate_heads).  quest_decode / quest_decode_step: run
                                 as a chain (the new token first, then every query head's
                                 bounds, the union, the sparse decode over it; size the
                                 workspace with the same opts); the one-launch paths and
                                 quest_decode_layers answer QUEST_ERR_UNSUPPORTED.  Not with
                                 sink / local pages (QUEST_ERR_INVALID_ARG).                  */
    int32_t path;             /* quest_decode*: QUEST_PATH_* (quest_decode_layers: see there).
                                 The chain
                                 computes the same step as separate kernels: estimate, top-K
                                 and sparse decode, or, for MHA rows of at most 4096 pages
                                 whose decode work items fit on the GPU about twice over,
                                 estimate and a sparse decode whose work items each take
                                 their pair's top-K; the estimate writes
                                 the new token's row and box as it scores that page, and the
                                 sparse decode advances the lengths at its end (selection
                                 kept in the workspace unless idx_out / count_out are
                                 given).                                                     */
} quest_opts_t;

/* Values of quest_opts_t.path.
 *   FUSED  : one launch of the cluster kernel, a thread-block cluster per (sequence, kv
 *            head) pair.
 *   CHAIN  : separate estimate, top-K and sparse-decode kernels, back to back (for short
 *            MHA rows with few pairs the top-K runs inside the sparse decode's work items).
 *   STREAM : one persistent launch of the stream kernel, one CTA per SM, every CTA working
 *            on every pair: pairs are scored in order over the whole GPU, each pair is
 *            selected as soon as its last page is scored while later pairs still stream,
 *            and the kept pages of every pair are decoded by every CTA.  Needs every CTA
 *            resident at once (cooperative launch), batch <= 1024 and top_k <= 2048.
 * AUTO (0) takes the one-launch cluster kernel for short rows (max_pages below 1024) when
 * every (sequence, kv head) pair of the call gets a cluster of at least 2 CTAs, all
 * resident at once with 2 CTAs per SM: there the step's fixed cost dominates and one
 * launch pays it once.  Otherwise (longer rows, more pairs, or a CTA needing more than
 * half an SM's shared memory) it takes the chain, whose scoring, top-K and decode kernels
 * spread over the whole GPU.  AUTO always takes the one-launch kernel when cluster_size,
 * trace or debug_flags is set, and the chain when no cluster of the one-launch kernel fits
 * in shared memory.  quest_decode_path() tells which one a call takes. */
#define QUEST_PATH_AUTO 0
#define QUEST_PATH_FUSED 1
#define QUEST_PATH_CHAIN 2
#define QUEST_PATH_STREAM 3

/* The path (QUEST_PATH_FUSED, _CHAIN or _STREAM) that quest_decode / quest_decode_step
 * (n_layers = 1) or quest_decode_layers (n_layers layers) take for this cache, top_k and
 * opts, or minus a QUEST_ERR_* status on invalid arguments.  Queries the device's occupancy
 * for the one-launch kernel; launches nothing. */
int quest_decode_path(const quest_cache_t* cache, int32_t top_k, const quest_opts_t* opts,
                      int32_t n_layers);

/* Kernel launches of one quest_decode or quest_decode_step call for this cache, top_k and
 * opts: 1 on the one-launch paths; on the chain 3 (estimate, top-K, sparse decode), or 2
 * when the sparse decode's work items take the top-K themselves (few pairs: see
 * QUEST_PATH_CHAIN); with gqa_union 3, and one more for quest_decode_step (its append).
 * Minus a QUEST_ERR_* status on invalid arguments; launches nothing. */
int quest_decode_launches(const quest_cache_t* cache, int32_t top_k, const quest_opts_t* opts);

/* quest_decode only (one-launch paths): never publish the selection, so that every
 * decode work item's bounded wait runs out and the call reports QUEST_ERR_TIMEOUT.  For
 * testing the timeout path; outputs are then unspecified. */
#define QUEST_DEBUG_WITHHOLD_SELECTION 1

/* Bytes of workspace the calls below need for this cache, top_k and opts; 0 if the
 * arguments are invalid (see quest_last_error). */
size_t quest_workspace_size(const quest_cache_t* cache, int32_t top_k, const quest_opts_t* opts);

/* Zero `ws_bytes` bytes of workspace on `stream` (cudaMemsetAsync). */
int quest_workspace_init(void* ws, size_t ws_bytes, quest_stream_t stream);

/*
 * Bounding boxes after prefill.  [Guide] Solution step 1 (min-max key bounding box
 * equations) and Implementation step 1 (min/max along the page's token axis): for every
 * sequence b, page p < ceil(seq_lens[b] / P) and kv head, meta[...][0][i] = min and
 * meta[...][1][i] = max of k[t][i] over the tokens t < seq_lens[b] of that page (a
 * partial last page is boxed over its valid tokens).  Exact (fp16 min/max).  Reads the
 * keys of every present token once.
 */
int quest_build_meta(const quest_cache_t* cache, void* ws, size_t ws_bytes,
                     quest_stream_t stream);

/*
 * Decode-time append.  [Guide] Solution step 1: a page's box is built as the page fills,
 * in prefill and in generation alike.  k_new, v_new: fp16 [batch][num_kv_heads][128].
 * For each sequence b the token goes to position L = seq_lens[b] (page L / P, which the
 * caller must have mapped in block_table, slot L % P); slot 0 starts the page's box,
 * any other slot widens it; then seq_lens[b] becomes L + 1.  A sequence with no room
 * (L + 1 > max_pages * P) or an unmapped page is skipped and reported.
 */
int quest_append(const quest_cache_t* cache, const void* k_new, const void* v_new, void* ws,
                 size_t ws_bytes, quest_stream_t stream);

/*
 * Chunked prefill with the boxes formed in the same pass.  [Guide] Solution step 1: the
 * box is formed as pages fill during prompt prefill.  k, v: fp16
 * [batch][n_tokens][num_kv_heads][128], token j of sequence b going to position
 * L_b + j (L_b = seq_lens[b]; every page it reaches must be mapped in block_table).
 * Each touched page's box becomes the per-dimension min / max over its old box (when the
 * page already held tokens) and its new keys: the same boxes as n_tokens quest_append
 * calls, or as quest_build_meta after the whole prompt, bit for bit.  Then seq_lens[b]
 * becomes L_b + n_tokens.  Reads the chunk once, writes it once plus the touched boxes.
 * A sequence with no room (L_b + n_tokens > max_pages * P) or a page outside
 * [0, num_phys) is reported (QUEST_ERR_BAD_LENGTH / QUEST_ERR_BAD_PAGE in the status)
 * and its length is left unchanged.  n_tokens = 0 does nothing.
 */
int quest_prefill(const quest_cache_t* cache, const void* k, const void* v, int32_t n_tokens,
                  void* ws, size_t ws_bytes, quest_stream_t stream);

/*
 * Query-aware criticality.  [Guide] Solution step 2, the upper-bound inequality:
 *   score[b][g][p] = sum_i max(q_i * Kmin_i, q_i * Kmax_i)
 * for the query heads h of kv head g (h / G == g), taking the maximum over those G
 * heads (selection per kv head).  The 1/sqrt(d) factor of the page's formula is left
 * out: a positive constant that cannot change the ranking.  Products are exact in fp32,
 * the sum is fp32.  q: fp16 [batch][num_q_heads][128].  scores: fp32
 * [batch][num_kv_heads][max_pages]; pages at or past ceil(seq_len / P) get -inf.
 */
int quest_estimate(const quest_cache_t* cache, const void* q, float* scores, void* ws,
                   size_t ws_bytes, quest_stream_t stream);

/*
 * The same bound per query head, without the maximum over its group: scores is fp32
 * [batch][num_q_heads][max_pages] (-inf at and past ceil(seq_len / P)).  Input of the
 * union form of the group-level selection ([Guide] Best Practices step 2; quest_topk with
 * opts->gqa_union).
 */
int quest_estimate_heads(const quest_cache_t* cache, const void* q, float* scores, void* ws,
                         size_t ws_bytes, quest_stream_t stream);

/*
 * Top-K page selection.  [Guide] Solution step 3; [Summary] Summary (the K best-scoring
 * pages).  For each (b, g) keeps K_b = min(top_k, N_b) pages, N_b = ceil(seq_len / P):
 * the pages with the largest scores, equal scores going to the lower page index.  If
 * N_b <= top_k every page is kept.  idx: int32 [batch][num_kv_heads][top_k], the kept
 * logical pages in ASCENDING page order, -1 after the first K_b; count: int32
 * [batch][num_kv_heads] = K_b.  Selection is an exact radix select on the fp32 scores.
 * opts (may be NULL): sink_pages / local_pages force the first and last pages in.
 */
int quest_topk(const quest_cache_t* cache, const float* scores, int32_t top_k, int32_t* idx,
               int32_t* count, void* ws, size_t ws_bytes, const quest_opts_t* opts,
               quest_stream_t stream);

/*
 * Attention over the kept pages.  [Summary] Summary: exact attention is computed only
 * over the Top-K pages; [Guide] Solution step 3 and Implementation step 3.  For query
 * head h (kv head g = h / G):
 *   out[b][h] = sum_t softmax_t(q.k_t / sqrt(128)) v_t,  lse[b][h] = log sum_t exp(q.k_t / sqrt(128))
 * over every token t < seq_len of the pages idx[b][g][0..count-1].  Split-K over the
 * kept pages with a log-sum-exp merge; fp32 arithmetic on fp16 data.  out: fp16
 * [batch][num_q_heads][128]; lse: fp32 [batch][num_q_heads] or NULL.  No kept token:
 * out = 0, lse = -inf.
 */
int quest_sparse_decode(const quest_cache_t* cache, const void* q, const int32_t* idx,
                        const int32_t* count, int32_t top_k, void* out, float* lse, void* ws,
                        size_t ws_bytes, const quest_opts_t* opts, quest_stream_t stream);

/*
 * The whole decode step: quest_estimate, quest_topk and quest_sparse_decode as one call
 * ([Guide] Best Practices step 3 suggests fusing the bound estimation with the page
 * gather).  On the one-launch path (opts->path, quest_decode_path) a thread-block cluster
 * per (sequence, kv head) pair does all of it: every CTA of the cluster scores a share of
 * the pair's boxes and passes its keys to the cluster's first CTA over distributed shared
 * memory, that CTA selects the pages (waits are bounded), every CTA attends over a share
 * of the kept pages, and the first CTA merges the shares.  On the chain path the three
 * kernels run back to back.  Same results as the three calls, up to the rounding of the
 * split-K merge.  idx_out / count_out (layouts of quest_topk) receive the selection if
 * non-NULL.
 */
int quest_decode(const quest_cache_t* cache, const void* q, int32_t top_k, void* out,
                 float* lse, int32_t* idx_out, int32_t* count_out, void* ws, size_t ws_bytes,
                 const quest_opts_t* opts, quest_stream_t stream);

/*
 * One whole decode step: the append of quest_append (k_new, v_new: fp16
 * [batch][num_kv_heads][128]) folded into quest_decode.  Whatever scores the new token's
 * page (a CTA of the pair's cluster, or the chain's estimate kernel) widens (or opens)
 * that page's box, writes the token's K/V rows and scores the page with the updated box;
 * selection and attention then cover seq_len + 1 tokens; seq_lens[b] becomes seq_len + 1
 * at the end of the step (a sequence with no room or an unmapped page is reported and
 * keeps its length).  Results equal quest_append followed by quest_decode.
 */
int quest_decode_step(const quest_cache_t* cache, const void* q, const void* k_new,
                      const void* v_new, int32_t top_k, void* out, float* lse, int32_t* idx_out,
                      int32_t* count_out, void* ws, size_t ws_bytes, const quest_opts_t* opts,
                      quest_stream_t stream);

/*
 * Every layer of one decode step in one call.  [Guide] Evaluation (end-to-end latency
 * table): a whole token step runs the sparse decode in every layer, which is where the
 * end-to-end gains are measured.  The same fused step as quest_decode_step (or
 * quest_decode when k_new is NULL) for n_layers layers that share the batch, the block
 * table and the lengths, each with its own K/V pools, boxes, query, new token and output.
 * With the one-launch kernel the (layer, sequence, kv head) pairs are the work units of
 * one persistent launch, so one pair's selection overlaps other pairs' streaming.
 * opts.path as for quest_decode, the rule counting every layer's pairs; the chain writes
 * every layer's new token first, advances the lengths once, then runs each layer's
 * estimate, top-K and sparse decode.  cache: the shared shape, block_table and seq_lens
 * (its k_pool / v_pool / meta are not used).  layers: host array of n_layers
 * (1..QUEST_MAX_LAYERS) quest_layer_t, read during the call only; pointers as in
 * quest_decode_step.  k_new / v_new: given for every
 * layer (each layer appends at slot seq_len[b]; seq_lens advance once, at the end) or for
 * none.  No idx_out.  ws: as quest_decode for this cache and top_k.
 */
#define QUEST_MAX_LAYERS 32
typedef struct {
    void* k_pool;        /* fp16 [num_phys][num_kv_heads][page_size][128] */
    void* v_pool;
    void* meta;          /* fp16 [batch][num_kv_heads][max_pages][2][128] */
    const void* q;       /* fp16 [batch][num_q_heads][128] */
    const void* k_new;   /* fp16 [batch][num_kv_heads][128] or NULL */
    const void* v_new;
    void* out;           /* fp16 [batch][num_q_heads][128] */
    float* lse;          /* fp32 [batch][num_q_heads] or NULL */
} quest_layer_t;

int quest_decode_layers(const quest_cache_t* cache, const quest_layer_t* layers, int32_t n_layers,
                        int32_t top_k, void* ws, size_t ws_bytes, const quest_opts_t* opts,
                        quest_stream_t stream);

/*
 * Full-context attention over every token (every page kept): the library's own dense
 * baseline ([Summary] Key points compare Quest's attention with a dense kernel).
 */
int quest_dense_decode(const quest_cache_t* cache, const void* q, void* out, float* lse,
                       void* ws, size_t ws_bytes, const quest_opts_t* opts,
                       quest_stream_t stream);

/*
 * quest_decode for callers that cannot allocate device memory.  The papers have no
 * counterpart to this call; it exists for callers that are handed their tensors but may
 * not obtain device memory themselves (an extension hosted by a runtime that owns the
 * allocator, an engine that forbids allocation while serving, a binding with no device
 * allocator), so they cannot pass quest_decode a workspace.  Same arguments and results as
 * quest_decode without ws / ws_bytes / opts (defaults are used).  The scratch is a 16 MiB
 * array in the library's own device memory (present on every GPU that loads the library,
 * until the process exits); a cache / top_k whose quest_workspace_size() exceeds 16 MiB is
 * rejected with QUEST_ERR_WORKSPACE.  Nothing is allocated.
 * - Every call looks up that array's address on the current device (not a stream
 *   operation), so a device reset that rebuilds the context leaves no stale address.
 * - Every call, on every stream, shares the one array: calls that may overlap on the GPU
 *   race and give wrong results.  Each call clears the part that must start at zero.
 * - status_out (nullable, device int32[4]) receives the device status word and its three
 *   detail words (see quest_read_status) once the call's work is done, in stream order
 *   (QUEST_OK and zeros for batch 0).  The array is private to the library and the next
 *   call clears it: with status_out NULL a device-side error (an unmapped page, a wait
 *   that ran out) of this call is lost.
 */
int quest_decode_static(const quest_cache_t* cache, const void* q, int32_t top_k, void* out,
                        float* lse, int32_t* idx_out, int32_t* count_out, int32_t* status_out,
                        quest_stream_t stream);

/*
 * Synchronise `stream`, return the device status recorded in the workspace (QUEST_OK
 * or a QUEST_ERR_* code) and clear it.  detail (nullable, 3 ints) receives the first
 * fault's sequence, logical page and a kernel-specific code.
 */
int quest_read_status(void* ws, size_t ws_bytes, quest_stream_t stream, int32_t* detail);

/* Text of the last failure on this thread ("" if none). */
const char* quest_last_error(void);

/* Name of a status code. */
const char* quest_status_string(int code);

int quest_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QUEST_H */
