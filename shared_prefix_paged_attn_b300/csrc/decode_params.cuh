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
};

}  // namespace fa
