// Kernel parameter block shared by the decode kernels (passed by value as a grid constant).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include "../../include/fork_attn.h"
#include "plan_layout.h"

namespace fa {

struct DecodeParams {
    CUtensorMap kmap;  // K pages viewed as [pages][Hkv][16][128] bf16, box 64 x 16, 128B swizzle
    CUtensorMap vmap;  // same for V
    CUtensorMap kmap_page;  // K as [pages][Hkv][2 halves][16][64]: one box = a whole page-head
    CUtensorMap vmap_page;  // V the same way
    const __nv_bfloat16 *q;
    void *out;
    float *lse;
    float *part_o;    // [partial_rows][128] fp32
    float *part_lse;  // [partial_rows] fp32, natural log
    const int32_t *chunk_pages;
    const Chunk *chunks;
    const Item *items;     // row-kernel work items
    const Item *items_tc;  // tcgen05-kernel work items
    const Item *items_r8;  // work items of the row kernel for <= 8 rows
    const RowRec *rows;
    const Branch *branches;
    const QMerge *q_merge;
    const int32_t *merge_bases;
    const int32_t *merge_lpos;  // first logical position of each partial's chunk
    const uint32_t *mask_words;
    int32_t *err;
    int32_t Hq, Hkv, G, out_dtype;
    float scale_log2;  // scale * log2(e): scores are kept in base 2 inside the kernels
    int32_t n_items;
    int32_t n_items_tc;
    int32_t n_items_r8;
    int32_t tc_ctas;  // persistent CTAs of the tcgen05 kernel
    int32_t pool_pages;  // page index one past the pool: TMA reads it as zeros
    int32_t total_rows;  // total_q * Hq
    int32_t n_partial_rows;  // rows of part_o / part_lse
    int32_t n_mask_words;    // words of mask_words
    int32_t lse_only;        // 1: only each row's lse (no V, no P V; partial O rows are zeros, out unused)
};

// Checked build (FORK_ATTN_CHECKED): every page id and row record the kernels take from the
// plan buffer is tested against the pool and the plan's arrays before it is used.  One out of
// range sets kErrBounds and the kernel's bit in the error word and is replaced by an index in
// range (the result is then garbage, but no access leaves its buffer).  The plain build
// trusts the planner, which validated the descriptors.
#ifdef FORK_ATTN_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// A page id for a plain load (fallback: page 0).
__device__ __forceinline__ int32_t checked_page(const DecodeParams &p, int32_t page, int32_t kbit) {
    if (kChecked && (page < 0 || page >= p.pool_pages)) {
        atomicOr(p.err, kErrBounds | kbit);
        return 0;
    }
    return page;
}

// A row record: its q/out row, its partial row (-1: direct) and its visibility words (-1:
// none) for a chunk of n_pages pages.
__device__ __forceinline__ void checked_row(const DecodeParams &p, int32_t &qrow, int32_t &prow, int32_t &mask_off,
                                            int32_t n_pages, int32_t kbit) {
    if (!kChecked) return;
    bool bad = false;
    if (qrow < 0 || qrow >= p.total_rows) { qrow = 0; bad = true; }
    if (prow < -1 || prow >= p.n_partial_rows) { prow = -1; bad = true; }
    if (mask_off < -1 || (mask_off >= 0 && int64_t(mask_off) + (n_pages + 1) / 2 > p.n_mask_words)) {
        mask_off = -1;
        bad = true;
    }
    if (bad) atomicOr(p.err, kErrBounds | kbit);
}

}  // namespace fa
