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

// A chunk: consecutive physical pages chunk_pages[page_off .. page_off + n_pages) that every
// one of its readers sees as consecutive logical positions.  Its readers ("occurrences")
// are occs[occ_off .. occ_off + n_occ).
struct Chunk {
    int32_t page_off;
    int32_t n_pages;
    int32_t occ_off;
    int32_t n_occ;
};

// One reader of one chunk: branch `branch` sees slot s of the chunk's page k at logical
// position lpos0 + 16 k + s.  mask_off: word offset of its visibility words (bit 16 k + s),
// or -1 when every slot of the chunk is valid and visible to it.  prow_base: first fp32
// partial row of this occurrence for KV head 0 (rows of head g start at prow_base +
// g * n_q * G), or -1 when the occurrence is the branch's only one and writes `out` directly.
struct Occ {
    int32_t branch;
    int32_t lpos0;
    int32_t mask_off;
    int32_t prow_base;
};

// A work item: one chunk, one KV head, and a row group = entries ents[ent_off ..
// ent_off + n_ent), together n_rows = sum(ni) * G rows.
struct Item {
    int32_t chunk;
    int32_t head;
    int32_t ent_off;
    int32_t n_ent;
    int32_t n_rows;
    int32_t pad[3];
};

// Query tokens i0 .. i0 + ni - 1 of occurrence `occ`.
struct Ent {
    int32_t occ;
    int32_t i0;
    int32_t ni;
    int32_t pad;
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

// Byte offsets of the arrays inside the device plan buffer.  The first 256 bytes hold the
// device error word (int32 at offset 0).
struct Layout {
    int64_t chunk_pages, chunks, occs, items_rows, items_tc, ents, branches, q_branch,
        merge_bases, mask_words, total;
    int32_t n_chunk_pages, n_chunks, n_occs, n_items_rows, n_items_tc, n_ents, n_branches,
        total_q, n_merge_bases, n_mask_words;
};

// Device error word bits.
enum : int32_t {
    kErrTimeout = 1,   // a bounded wait expired
    kErrBounds = 2,    // a checked index was out of range
};

}  // namespace fa
