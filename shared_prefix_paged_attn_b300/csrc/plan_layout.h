// Device-visible plan arrays, written by the host planner (plan.cpp) and read by the kernels.
// Plain structs of int32 so that one host blob can be copied to the device as is.
#pragma once
#include <stdint.h>

namespace fa {

constexpr int kHeadDim = 128;
constexpr int kPageSize = 16;
constexpr int kRowsMax = 32;      // rows of one row-kernel work item (two m16 tiles)
constexpr int kTcRows = 128;      // rows of one tcgen05 work item (one M = 128 tile)
constexpr int kAlign = 256;       // byte alignment of every array in the plan blob
constexpr int kMaxChunkPages = 256;  // longest chunk the planner cuts (the tcgen05 kernel's limit)

// A chunk: consecutive physical pages chunk_pages[page_off .. page_off + n_pages) that every
// one of its readers sees as consecutive logical positions.  Its readers ("occurrences")
// are occs[occ_off .. occ_off + n_occ).
struct Chunk {
    int32_t page_off;
    int32_t n_pages;
    int32_t occ_off;
    int32_t n_occ;
};

// One reader of one chunk (host side only): branch `branch` sees slot s of the chunk's page
// k at logical position lpos0 + 16 k + s.  mask_off: word offset of its visibility words
// (bit 16 k + s), or -1 when every slot of the chunk is valid and visible to it.
// prow_base: its first fp32 partial row, or -1 when the occurrence is the branch's only one
// and writes `out` directly.  Partial row of (query token i, head-in-group jh, KV head g):
// prow_base + (i * G + jh) * Hkv + g.
struct Occ {
    int32_t branch;
    int32_t lpos0;
    int32_t mask_off;
    int32_t prow_base;
    int32_t pos_off;  // representative plans: its pages' score positions at occ_pos[pos_off ..]
};

// A work item: one chunk, one KV head, and a row group = rows[row_off .. row_off + n_rows)
// (row groups are shared by every KV head of a chunk).  n_pages: the chunk's first pages that
// the item reads -- all of them, unless no row of the group can see past some page (a row's
// query token lies before the rest of the chunk: prefill-shaped plans, where every token of a
// branch is a query); the kernels stop there.
struct Item {
    int32_t chunk;
    int32_t head;
    int32_t row_off;
    int32_t n_rows;
    int32_t n_pages;
    int32_t pad[3];
};

// One stacked query row of a row group: a (reader, query token, query head in the GQA group).
// For KV head g: its q / out / lse row is qrow0 + g * G, its partial row prow0 + g (prow0 = -1:
// a direct write).  climit: chunk tokens t <= climit are causally visible.  mask_off: the
// reader's visibility words for the chunk, -1 = all visible.
struct RowRec {
    int32_t qrow0;
    int32_t climit;
    int32_t mask_off;
    int32_t prow0;
};

// Per branch: its query rows start at q_begin (token index into q/out), n_q of them, the
// first at logical position qpos0.  Its partial rows (one base per occurrence, in chunk
// order) are merge_bases[merge_off .. merge_off + n_merge); n_merge <= 1 with a direct write
// means nothing to merge, n_merge == 0 means no visible entry at all.
struct Branch {
    int32_t q_begin;
    int32_t n_q;
    int32_t qpos0;
    int32_t merge_off;
    int32_t n_merge;
    int32_t direct;
    int32_t pad[2];
};

// Per query token, what the merge kernel needs: its branch's partial-row bases
// merge_bases[merge_off .. merge_off + n_merge), whether its only chunk wrote `out` directly,
// its index i among the branch's query tokens, and its logical position pos.  The first
// kMergeInline bases, with the first logical position of each one's chunk, are also held
// here, so that a token with that many partials or fewer needs one load of this record
// before it loads the partials themselves.  The merge skips a partial whose chunk starts
// after pos (merge_lpos, parallel to merge_bases): the token sees nothing of that chunk, and
// the planner may have left the item that would have written the partial out.
constexpr int kMergeInline = 5;
struct QMerge {
    int32_t merge_off;
    int32_t n_merge;
    int32_t direct;
    int32_t i;
    int32_t pos;
    int32_t base[kMergeInline];
    int32_t lpos[kMergeInline];
    int32_t pad;
};
static_assert(sizeof(QMerge) == 64, "one 64-byte record per query token");

// Byte offsets of the arrays inside the device plan buffer.  The first 256 bytes are a
// header of int32 words, zero in the uploaded plan: [0] the device error word, [1] [2] the
// work counter and exit count of the persistent tcgen05 kernel (its last CTA puts both back
// to zero), [3] the work counter of the scoring kernel (set to zero before each launch); the
// other words are unused and stay zero.
//
// Plans of representative queries (for key scoring) also hold: every work item once more in
// one list (score_items), cut into units of at most kScoreUnitTiles 128-key tiles (score_units:
// item, first tile, tiles, 0), for every reader of every chunk page the score index of the
// page's slot 0 for that reader (occ_pos: entry_off[branch] + the logical position of slot 0,
// pages in chunk order, one run per occurrence), each row's occurrence run in it (row_pos),
// and per branch the offsets of its entries (entry_off) and of its keep-bit words (word_off).
// A chunk's pages need not be logically adjacent (a run may step over pages its readers do
// not see), so the positions are listed per page.
struct Layout {
    int64_t chunk_pages, chunks, items_rows, items_tc, items_r8, rows, branches, q_merge, merge_bases,
        merge_lpos, mask_words, score_items, score_units, occ_pos, row_pos, entry_off, word_off, total;
    int32_t n_chunk_pages, n_chunks, n_items_rows, n_items_tc, n_items_r8, n_rows, n_branches, total_q,
        n_merge_bases, n_mask_words, n_score_items, n_score_units;
    int64_t total_entries, total_words;
};

// Tiles of one unit of the scoring kernel's work queue.
constexpr int kScoreUnitTiles = 16;

// Device error word bits (header word 0), and which kernel set them.
enum : int32_t {
    kErrTimeout = 1,   // a bounded wait expired
    kErrBounds = 2,    // a checked index was out of range
    kErrTc = 4,        // ... in the tcgen05 kernel
    kErrRow8 = 8,      // ... in the row kernel for <= 8 rows
    kErrRow = 16,      // ... in the row kernel for <= 32 rows
    kErrScore = 32,    // ... in the key-scoring kernel
    kErrMerge = 64,    // ... in the merge kernel
};

}  // namespace fa
