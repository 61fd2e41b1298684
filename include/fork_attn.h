/*
 * fork_attn.h -- C ABI of libforkattn.so: decode attention over a branching, paged KV cache
 * on one NVIDIA B300 (sm_103a).
 *
 * What the calls compute (sources are the pages' titles and sections):
 *
 *   - Octopus (zicq.com, "Octopus以共享KV DAG重构多智能体强化学习"), section "Zero-Copy Radix
 *     Forking": branches fork from a radix prefix of physical KV pages; a fork adds a cursor,
 *     not a copy, and the shared pages are read-only.  Here a fork is two branches whose
 *     segment lists name the same segments (or segments over the same physical pages).
 *   - Octopus, section "Attention-Only KV Mounting": a thread attends to a sibling's
 *     terminal KV block in place.  Here a mount is a segment whose pages belong to a sibling,
 *     listed in the mounting branch's segment list.
 *   - AKV (news.farwalk.ai, "清华与港中文开源 AKV"), section "AKV 如何工作？": Drop removes
 *     entries from later attention and keeps positions; Append adds new tokens.  Here a drop
 *     is a cleared bit in the branch's visibility bits; the query tokens of a branch are its
 *     last n_q logical tokens (their K/V are already appended).
 *   - Agentrix (gitlink.org.cn, "Agentrix：面向智能体的内存管理系统设计与实现"), section
 *     "初赛基础与决赛演进", CUDA ForkAttention: the cached pages are split into a common part
 *     and private parts, many queries reuse one read of the common KV, and per-branch results
 *     are merged.  Here: the planner groups page runs by reader set, the kernels read every
 *     visible physical page once per KV head and row group, and a log-sum-exp merge joins
 *     the partial results.
 *
 * Result, for branch b with logical sequence of length n_b and query token i (position
 * p = n_b - n_q_b + i), query head h, KV head g = h / (Hq / Hkv), and visible set
 * V = { j <= p : vis_b[j] = 1 }:
 *     s_j = scale * <q[b,i,h], K[slot(j), g]>
 *     lse[b,i,h] = ln sum_{j in V} exp(s_j)                     (natural log, scale included)
 *     out[b,i,h] = sum_{j in V} exp(s_j - lse) * V[slot(j), g]
 * An empty V gives out = 0 and lse = -inf.
 *
 * Conventions common to every call:
 *   - Every function returns an int status: FA_OK (0) or a negative FA_ERR_*; none aborts.
 *     fork_attn_strerror() names a status.
 *   - Host pointers are marked [host], device pointers [device].  The library never
 *     allocates device memory: the caller owns every device buffer (inputs, outputs, plan
 *     buffer and scratch) and keeps it alive while work that uses it may run.
 *   - A stream argument is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Only head_dim = 128 and page_size = 16 are built; other values return
 *     FA_ERR_UNSUPPORTED.
 */
#ifndef FORK_ATTN_H
#define FORK_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    FA_OK = 0,
    FA_ERR_NULL = -1,          /* a required pointer is NULL                                  */
    FA_ERR_INVALID = -2,       /* malformed descriptor or dims (see fork_attn_plan_create)   */
    FA_ERR_UNSUPPORTED = -3,   /* head_dim / page_size / GQA shape not built                  */
    FA_ERR_RANGE = -4,         /* an index (page id, segment id, offset) is out of range     */
    FA_ERR_ALIGN = -5,         /* a device pointer is not 16-byte aligned                    */
    FA_ERR_NOT_UPLOADED = -6,  /* fork_attn_decode before fork_attn_plan_upload               */
    FA_ERR_CUDA = -7,          /* a CUDA runtime / driver call failed                         */
    FA_ERR_NOMEM = -8,         /* host allocation failed                                      */
    FA_ERR_BUFFER_SMALL = -9,  /* a caller buffer is smaller than fork_attn_plan_sizes says   */
    FA_ERR_DEVICE = -10,       /* a kernel reported a fault through the plan's error word     */
    FA_ERR_SCRATCH_LIMIT = -11 /* the plan needs more than fork_attn_decode_static_scratch's  */
                               /* built-in device array holds (FA_STATIC_SCRATCH_BYTES)        */
};

enum { FA_BF16 = 0, FA_F32 = 1 };

/* Problem dimensions.  num_q_heads % num_kv_heads == 0 (GQA group G = num_q_heads /
 * num_kv_heads, query head h reads KV head h / G).  scale multiplies q.k (1/sqrt(128) in the
 * workloads).  out_dtype selects the element type of `out` in fork_attn_decode. */
typedef struct {
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;   /* must be 128 */
    int32_t page_size;  /* must be 16  */
    float scale;
    int32_t out_dtype;  /* FA_BF16 or FA_F32 */
} fa_dims;

/* A segment: `len` consecutive tokens, starting at slot `tok_begin` of the listed page
 * page_ids[page_off]; token t sits in page page_ids[page_off + (tok_begin + t) / page_size],
 * slot (tok_begin + t) % page_size. */
typedef struct {
    int32_t page_off;   /* index into page_ids of the segment's first page   */
    int32_t tok_begin;  /* 0 .. page_size-1                                  */
    int32_t len;        /* >= 1                                              */
} fa_segment;

/* The branching cache, all in [host] memory owned by the caller and read only during
 * fork_attn_plan_create.  Branch b's logical sequence is the concatenation of segments
 * branch_segs[branch_seg_off[b] .. branch_seg_off[b+1]) in list order; a segment may be
 * listed by many branches (a fork or a mount) and even twice by one (it then counts twice). */
typedef struct {
    const int32_t *page_ids;        /* [num_page_ids] physical page per listed page          */
    int64_t num_page_ids;
    const fa_segment *segs;         /* [num_segs]                                            */
    int32_t num_segs;
    const int32_t *branch_seg_off;  /* [num_branches + 1], branch_seg_off[0] = 0, ascending  */
    const int32_t *branch_segs;     /* segment ids                                           */
    int32_t num_branches;           /* >= 1                                                  */
    const int32_t *branch_q_off;    /* [num_branches + 1] query tokens per branch (CSR);     */
                                    /* NULL = one query token per branch.  1 <= n_q <= n_b.   */
    const uint32_t *vis_bits;       /* visibility bits, bit j%32 of word vis_word_off[b] +   */
    const int64_t *vis_word_off;    /* j/32 for logical index j of branch b; 1 = visible.    */
                                    /* Both NULL = everything visible.                        */
    int64_t num_vis_words;          /* length of vis_bits (bounds vis_word_off[b] + n_b/32)  */
    int64_t num_pages_pool;         /* physical page ids must lie in [0, num_pages_pool);    */
                                    /* (num_pages_pool + 1) x num_kv_heads < 2^31             */
} fa_desc;

/* Planner knobs; pass NULL to fork_attn_plan_create for the defaults (all fields 0). */
typedef struct {
    int32_t chunk_pages;    /* max pages per work chunk (0 = chosen from the SM count)      */
    int32_t num_sms;        /* SMs to plan for (0 = 148)                                     */
    int32_t tensor_min_rows;/* reader-set rows at which a run goes to the tcgen05 kernel    */
                            /* (0 = default; < 0 = never)                                    */
    int32_t tensor_ctas;    /* persistent CTAs of the tcgen05 kernel (0 = from the planner's */
                            /* split of SMs between it and the row kernels)                  */
    int32_t tensor_chunk_pages; /* max pages per tcgen05 chunk, rounded up to whole 8-page   */
                            /* tiles (0 = chosen by the planner)                             */
    int32_t representatives;/* 1: the query tokens are representative queries for key       */
                            /* scoring: each sees its branch's whole visible list (no causal */
                            /* limit; n_q may exceed n_b), and the plan can also drive       */
                            /* fork_attn_score / fork_attn_topk.  0: decode queries          */
    int32_t reserved[2];    /* must be 0                                                     */
} fa_plan_opts;

/* Counters of a plan, for measurement.  unique_visible_slots: distinct physical token slots
 * visible to at least one query (a slot read by many branches counts once); touched_pages:
 * distinct physical pages holding such a slot.  One slot of one KV head is 2 x 128 x 2 bytes
 * of K and V. */
typedef struct {
    int64_t unique_visible_slots;
    int64_t touched_pages;
    int64_t listed_visible_slots;  /* sum over branches of visible entries (copy-context)   */
    int64_t num_chunks;
    int64_t num_items_rows;        /* work items of the mma.sync row kernels                */
    int64_t num_items_tensor;      /* work items of the tcgen05 kernel                      */
    int64_t kv_bytes_rows;         /* K+V bytes read by the row kernel (all heads)           */
    int64_t kv_bytes_tensor;       /* K+V bytes read by the tcgen05 kernel                   */
    int64_t partial_rows;          /* fp32 partial (out, lse) rows in scratch                */
    int64_t merge_rows;            /* (query token, head) rows merged by the merge kernel   */
    int64_t total_q;
    int64_t unique_slots_rows;     /* distinct visible physical slots read by the row kernel */
    int64_t unique_slots_tensor;   /* distinct visible physical slots read by tcgen05 kernel */
    int64_t flops_rows;            /* algorithmic flops of the row kernel: 4 x 128 per       */
    int64_t flops_tensor;          /* (query row, KV head, visible slot causally before it)  */
    int64_t num_items_row8;        /* of num_items_rows: items with <= 8 rows (own kernel)   */
    int64_t unique_slots_row8;     /* visible slots of the chunks that kernel reads          */
    int64_t unique_slots_row32;    /* the same for the row kernel of up to 32 rows (a chunk  */
                                   /* whose row groups go to both counts in both)            */
    int64_t tensor_ctas;           /* persistent CTAs the tcgen05 kernel is launched with    */
    int64_t items_skipped;         /* (row group, chunk) pairs left out (any KV head): every */
                                   /* row's query token lies before the chunk's first slot   */
                                   /* (prefill-shaped plans); items read only up to the last */
                                   /* page some row of the group can see                     */
} fa_plan_stats;

typedef struct fa_plan fa_plan; /* opaque; owned by the library */

/* Builds a plan on the host: validates dims and descriptor, finds runs of physical pages
 * with the same reader set, skips pages no reader sees, cuts runs into chunks, assigns
 * partial-result rows and packs per-chunk visibility words.  Errors: FA_ERR_NULL,
 * FA_ERR_INVALID (bad CSR, n_q outside [1, n_b], empty branch, bad scale/out_dtype, a
 * negative planner knob or a non-zero reserved field),
 * FA_ERR_RANGE (segment id, page offset or page id out of range, bit array too short),
 * FA_ERR_UNSUPPORTED (head_dim != 128, page_size != 16, Hq % Hkv != 0, G > 32),
 * FA_ERR_NOMEM.  *out_plan is set only on FA_OK. */
int fork_attn_plan_create(const fa_dims *dims, const fa_desc *desc, const fa_plan_opts *opts,
                          fa_plan **out_plan);

/* Byte sizes of the two device buffers the caller must provide to fork_attn_plan_upload:
 * plan_bytes for the plan arrays, scratch_bytes for fp32 partial results (may be 0). */
int fork_attn_plan_sizes(const fa_plan *plan, size_t *plan_bytes, size_t *scratch_bytes);

/* Fills *stats [host]. */
int fork_attn_plan_stats(const fa_plan *plan, fa_plan_stats *stats);

/* Copies the plan arrays into dev_plan_buf [device, 256-byte aligned, >= plan_bytes] on
 * `stream` and records both buffers in the plan for later decodes.  dev_scratch_buf
 * [device, 256-byte aligned, >= scratch_bytes] may be NULL when scratch_bytes is 0.  The
 * host copy is synchronous with respect to the host.  Errors: FA_ERR_NULL, FA_ERR_ALIGN,
 * FA_ERR_BUFFER_SMALL, FA_ERR_CUDA. */
int fork_attn_plan_upload(fa_plan *plan, void *dev_plan_buf, size_t plan_buf_bytes,
                          void *dev_scratch_buf, size_t scratch_buf_bytes, void *stream);

/* Runs the decode on `stream`: no allocation, no host synchronisation.
 *   q       [device] bf16 [total_q][num_q_heads][128]; total_q = branch_q_off[B]; query token
 *           i of branch b is row branch_q_off[b] + i.
 *   k_pages [device] bf16 [num_pages_pool][num_kv_heads][16][128]
 *   v_pages [device] same layout as k_pages
 *   out     [device] out_dtype [total_q][num_q_heads][128]
 *   lse     [device] fp32 [total_q][num_q_heads]  (natural log)
 * All device pointers must be 16-byte aligned.  Inputs are only read.  The plan's device
 * buffers hold the work counters of the persistent tcgen05 kernel and the fp32 partials, so
 * two decodes of one plan must not overlap on the GPU (one stream, or order them); decodes
 * of different plans may.  Errors: FA_ERR_NULL, FA_ERR_ALIGN, FA_ERR_NOT_UPLOADED,
 * FA_ERR_CUDA (launch failure). */
int fork_attn_decode(const void *q, const void *k_pages, const void *v_pages,
                     const fa_plan *plan, void *out, float *lse, void *stream);

/* The same decode with its kernels run one after the other on `stream`, each timed alone:
 * `events` [host] (may be NULL) is an array of 2*n_events cudaEvent_t handles (as void*),
 * [start, stop] recorded on `stream` around the row kernel of at most 8 stacked rows, the row
 * kernel of up to 32, the tcgen05 kernel and the merge kernel, in that order (an absent kernel
 * records start = stop).  n_events must be 0 or 4.
 *
 * fork_attn_decode itself runs the kernels overlapped, all on `stream`: the tcgen05 kernel
 * first, then the row kernels as programmatic dependent launches (they start once every
 * tcgen05 CTA has started, and take the SMs it leaves and frees), then the merge as an
 * ordinary launch after all of them, with no helper stream or event; an event recorded
 * between those kernels would order them (and so serialise them), which is why this call
 * runs them one by one instead. */
int fork_attn_decode_timed(const void *q, const void *k_pages, const void *v_pages,
                           const fa_plan *plan, void *out, float *lse, void *stream,
                           void **events, int32_t n_events);

/* Reads the device error word of the plan's last decode on `stream` (synchronising it) into
 * *device_error [host] and clears it.  A non-zero word means a kernel gave up (an expired wait
 * or a failed check) and the outputs of that decode are not valid.  After
 * fork_attn_plan_upload or fork_attn_decode(_timed) the word is the one in the plan buffer;
 * after fork_attn_decode_static_scratch it is the one in the library's built-in device array
 * on the device that call ran on (make that device current), which the next
 * fork_attn_decode_static_scratch of any plan on that device overwrites.  Nothing is
 * allocated.  Errors: FA_ERR_NULL, FA_ERR_NOT_UPLOADED (the plan was never uploaded nor run
 * through fork_attn_decode_static_scratch), FA_ERR_CUDA, FA_ERR_DEVICE (the word was set). */
int fork_attn_check(fa_plan *plan, int32_t *device_error, void *stream);

/* Size of the device array used by fork_attn_decode_static_scratch: 32 MiB. */
#define FA_STATIC_SCRATCH_BYTES (32u << 20)

/* A decode for callers that cannot allocate device memory at all: an engine plugin whose
 * host owns every device allocation and hands it only the input and output tensors, or code
 * that must not touch the allocator while it runs (a latency-critical loop, or a region
 * where the allocator is locked).  The source pages have no counterpart of this call; it
 * exists only so that such callers can run the same plan.
 *
 * The caller passes the same inputs and outputs as to fork_attn_decode and a plan from
 * fork_attn_plan_create; the plan does not need fork_attn_plan_upload.  Instead of caller
 * buffers, the plan arrays and the fp32 partial results live in one device array of
 * FA_STATIC_SCRATCH_BYTES that the library defines at file scope: every GPU that loads the
 * library holds it until the process exits.  Each call copies the plan arrays into the array
 * (cudaMemcpyAsync from host memory, on `stream`; this also clears the device error word)
 * and then runs the same kernels as fork_attn_decode.  Nothing is allocated: no cudaMalloc,
 * no cudaFree, no allocating library routine.
 *
 * The first call on a device (made current by the caller) looks up the array's device
 * address with cudaGetSymbolAddress.  Every call on a device shares the one array and leaves the last call's contents in it:
 * two calls whose work overlaps on the GPU (different streams, or different host threads)
 * race on it, so serialise them.  fork_attn_check on the same plan reads and clears the
 * device error word this call wrote (word 0 of the array), until another call overwrites it.
 *
 * Errors: FA_ERR_NULL, FA_ERR_ALIGN (as fork_attn_decode), FA_ERR_SCRATCH_LIMIT when
 * plan_bytes + scratch_bytes of fork_attn_plan_sizes exceed FA_STATIC_SCRATCH_BYTES (checked
 * before any CUDA call), FA_ERR_CUDA. */
int fork_attn_decode_static_scratch(const void *q, const void *k_pages, const void *v_pages,
                                    const fa_plan *plan, void *out, float *lse, void *stream);

/* ---- Physical compaction with optional repositioning ----
 * AgentKV blog (rit.work), "Как AgentKV выбирает и освобождает записи кэша": the kept entries
 * of a cache are packed into fresh pages, so the freed pages can go back to the allocator and
 * later decodes read fewer bytes.  AKV (news.farwalk.ai), "AKV 如何工作？": Repos rewrites the
 * kept keys to positions 0..r-1 with a RoPE rotation, values unchanged.
 *
 * For each listed branch, the entries visible in its bits (all of them without bits) are
 * copied in logical order to destination pages: the n-th kept entry of the branch to slot
 * n % page_size of the branch's (n / page_size)-th destination page.  V is copied as is; K too
 * unless reposition != 0, in which case the key of the entry at logical index j is rotated
 * by the position change d = n - j: for i < head_dim / 2 with theta_i =
 * rope_base^(-2 i / head_dim), the pair (x_i, x_{i + head_dim/2}) becomes
 * (x_i cos(d theta_i) - x_{i+h} sin(d theta_i), x_{i+h} cos(d theta_i) + x_i sin(d theta_i))
 * (rotate-half pairing), computed in fp32 and rounded to bf16 (nearest even).
 *
 * share_prefix != 0 keeps a fork's sharing: the listed branches' common prefix -- the first
 * P logical entries, where every listed branch has the same physical slot and the same
 * visibility bit at each of them -- is packed once, and each branch's entries after it go
 * to pages of the branch's own.  Entry n of every branch is still the n-th kept one, with the
 * same position change, so each branch reads [the shared run's r_s entries] then [its own
 * r - r_s entries], two segments that both start at slot 0 of a page. */
typedef struct {
    int32_t num_kv_heads;
    int32_t head_dim;     /* 128 */
    int32_t page_size;    /* 16 */
    int32_t reposition;   /* 0: keys copied; 1: keys rotated from position j to n (Repos) */
    double rope_base;     /* > 1; used when reposition != 0 */
    int32_t share_prefix; /* 0: every branch packed on its own; 1: common prefix packed once */
    int32_t reserved;     /* must be 0 */
} fa_compact_dims;

typedef struct fa_compact fa_compact; /* opaque; owned by the library */

/* Plans the compaction of branches[0 .. num_branches) of `desc` (host arrays, read here
 * only).  Destination pages are dst_page_ids [host], consumed branch after branch, each branch
 * from a fresh page (ceil(r / page_size) pages for r kept entries); with share_prefix the
 * shared run's ceil(r_s / page_size) pages come first, then each branch's ceil((r - r_s) /
 * page_size).  They must not be pages of
 * any listed branch (the gather runs in place in the same pool) and must not hold anything
 * another reader still needs.  Errors: FA_ERR_NULL, FA_ERR_INVALID (branch index, bad CSR or
 * segment, too few destination pages, a destination page listed twice or read by a listed
 * branch, rope_base <= 1 with reposition, share_prefix not 0 or 1, reserved != 0),
 * FA_ERR_RANGE (page id, segment id or bit word out of range; a pool of more than 2^27
 * pages), FA_ERR_UNSUPPORTED (head_dim != 128, page_size != 16), FA_ERR_NOMEM.  *out is set
 * only on FA_OK. */
int fork_attn_compact_create(const fa_compact_dims *dims, const fa_desc *desc,
                             const int32_t *branches, int32_t num_branches,
                             const int32_t *dst_page_ids, int64_t num_dst_pages,
                             fa_compact **out);

/* kept_tokens [host, num_branches] (may be NULL): r per listed branch.  work_bytes (may be
 * NULL): the size of the device work buffer of fork_attn_compact_upload. */
int fork_attn_compact_sizes(const fa_compact *c, int64_t *kept_tokens, size_t *work_bytes);

/* shared_kept (may be NULL): r_s, the kept entries of the shared run (0 without
 * share_prefix).  prefix_len (may be NULL): P, the common prefix's length in logical entries
 * (0 without share_prefix). */
int fork_attn_compact_shared(const fa_compact *c, int64_t *shared_kept, int64_t *prefix_len);

/* Copies the plan's slot lists into dev_work [device, 256-byte aligned, >= work_bytes] on
 * `stream` (from the plan's host memory: keep the plan until the stream has passed the copy).
 * Errors: FA_ERR_NULL, FA_ERR_ALIGN, FA_ERR_BUFFER_SMALL, FA_ERR_CUDA. */
int fork_attn_compact_upload(fa_compact *c, void *dev_work, size_t work_bytes, void *stream);

/* Runs the gather on `stream`: k_pages, v_pages [device, 16-byte aligned] bf16
 * [num_pages_pool][num_kv_heads][16][128] are read at the kept slots and written at the
 * destination slots.  No allocation, no host synchronisation; running it again rewrites the
 * same destinations.  Errors: FA_ERR_NULL, FA_ERR_ALIGN, FA_ERR_NOT_UPLOADED, FA_ERR_CUDA. */
int fork_attn_compact_run(const fa_compact *c, void *k_pages, void *v_pages, void *stream);

/* Frees the compaction plan (not the caller's device buffers). */
int fork_attn_compact_destroy(fa_compact *c);

/* Joins the results of one problem split into parts that each saw a disjoint share of every
 * branch's visible entries (for instance one range of logical positions per GPU, each part
 * decoded with the other entries' visibility bits cleared): part_out [device, fp32,
 * n_parts x rows x head_dim (128)] and part_lse [device, fp32, n_parts x rows], part k's rows
 * at k * rows; rows = total_q x Hq.  Per row, the log-sum-exp merge of the parts in order
 * (Agentrix (gitlink.org.cn), "初赛基础与决赛演进": per-branch results are merged):
 *     L = max_k lse_k + ln sum_k exp(lse_k - max_k lse_k),   out = sum_k exp(lse_k - L) out_k,
 * a part with lse = -inf contributing nothing; a row no part saw gets out = 0, lse = -inf.
 * out [device, rows x 128, bf16 (RNE) or fp32 by out_dtype], lse [device, fp32, rows], on
 * `stream`; no allocation, no synchronisation.  Errors: FA_ERR_NULL, FA_ERR_INVALID (n_parts
 * < 1, rows < 0, bad out_dtype), FA_ERR_ALIGN (part_out, out not 16-byte aligned),
 * FA_ERR_CUDA. */
int fork_attn_merge_parts(const float *part_out, const float *part_lse, int32_t n_parts,
                          int64_t rows, void *out, int32_t out_dtype, float *lse, void *stream);

/* ---- Key scoring by representative queries, and top-k keep ----
 * AgentKV blog (rit.work), "Как AgentKV выбирает и освобождает записи кэша": the recent
 * queries of every phase are merged into one set of representatives (32 in the main
 * experiments), every key is scored by the mean attention the representatives give it, and
 * the entries with the largest scores are kept.  For branch b of a plan made with
 * fa_plan_opts.representatives = 1, its n_q query tokens are its representatives r < R, and
 * for each of its visible entries j
 *     score(j) = 1 / (R Hq) * sum over r < R, h < Hq of exp(s_{r,h,j} - lse_{r,h}),
 * s_{r,h,j} = scale <q_{r,h}, K[slot(j), h / G]>, lse_{r,h} over the branch's visible entries
 * (no causal limit).  Three calls on one stream:
 *   1. fork_attn_score_lse(q, k, plan, lse, stream): the lse of every representative row
 *      [device, fp32, total_q x Hq] (the decode's kernels with no V, no P V and no output
 *      rows; fork_attn_decode on the same plan gives the same lse and the outputs too);
 *   2. fork_attn_score(q, k, plan, lse, scores, stream): scores [device, fp32,
 *      total_entries]: branch b's entries at entry_off[b] + j, entry_off the running sum of
 *      the branches' list lengths n_b; an entry the branch does not see is NaN.  Uses the
 *      plan's scratch (per-KV-head scores) and sets the plan's error word (fork_attn_check);
 *   3. fork_attn_topk(plan, scores, keep_k, keep_bits, stream): keep_k [device, int32,
 *      num_branches]; keep_bits [device, uint32, total_words]: branch b's new visibility bits,
 *      bit j % 32 of word word_off[b] + j / 32 (word_off the running sum of ceil(n_b / 32)),
 *      set for the k_b visible entries with the largest scores, equal scores keeping the
 *      smaller j (all visible entries when k_b >= their number, none when k_b <= 0).
 * q, k_pages, lse: as fork_attn_decode's (16-byte aligned), the same plan, uploaded; the
 * lse pass writes the plan's scratch partials and its error word.  Errors:
 * FA_ERR_NULL, FA_ERR_INVALID (not a representatives plan), FA_ERR_NOT_UPLOADED,
 * FA_ERR_ALIGN, FA_ERR_CUDA.  fork_attn_plan_create refuses a representatives plan with
 * n_q x G > 256 for a branch (FA_ERR_UNSUPPORTED). */
int fork_attn_score_lse(const void *q, const void *k_pages, const fa_plan *plan, float *lse,
                        void *stream);
int fork_attn_score(const void *q, const void *k_pages, const fa_plan *plan, const float *lse,
                    float *scores, void *stream);
int fork_attn_topk(const fa_plan *plan, const float *scores, const int32_t *keep_k,
                   uint32_t *keep_bits, void *stream);
/* total_entries / total_words (either may be NULL): the sizes of scores and keep_bits. */
int fork_attn_score_sizes(const fa_plan *plan, int64_t *total_entries, int64_t *total_words);

/* Frees the host plan.  Device buffers stay owned by the caller. */
int fork_attn_plan_destroy(fa_plan *plan);

/* A static string for a status code. */
const char *fork_attn_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* FORK_ATTN_H */
