// Host-side plan object shared by the planner (plan.cpp) and the launcher (decode.cu).
#pragma once
#include <stdint.h>

#include <vector>

#include "../../include/fork_attn.h"
#include "plan_layout.h"

struct fa_plan {
    fa_dims dims;
    int32_t G;                    // query heads per KV head
    int64_t num_pages_pool;
    fa::Layout lay;
    std::vector<uint8_t> blob;    // host copy of the device plan buffer (lay.total bytes)
    int64_t partial_rows;         // fp32 partial rows (each 128 floats + 1 lse)
    bool representatives;         // a plan of representative queries (key scoring)
    bool merge_wide;              // few merged rows, most partials in rows of more than kMergeInline
    fa_plan_stats stats;
    int32_t tc_ctas;              // persistent CTAs of the tcgen05 kernel (<= SMs)
    // set by fork_attn_plan_upload
    void *dev_plan;
    void *dev_scratch;
    bool uploaded;
    // device error word of the plan's last decode: word 0 of dev_plan after an upload or a
    // fork_attn_decode, word 0 of the built-in static array after a
    // fork_attn_decode_static_scratch (read and cleared by fork_attn_check)
    mutable int32_t *err_word;
};

namespace fa {
inline int64_t scratch_lse_offset(int64_t partial_rows) {
    // partial O: partial_rows x 128 fp32, then partial lse: partial_rows fp32 (256-aligned)
    return ((partial_rows * kHeadDim * 4 + kAlign - 1) / kAlign) * kAlign;
}
inline int64_t scratch_bytes(int64_t partial_rows) {
    if (partial_rows == 0) return 0;
    return scratch_lse_offset(partial_rows) + ((partial_rows * 4 + kAlign - 1) / kAlign) * kAlign;
}
// A scoring plan's scratch holds, after the partials, the per-KV-head key scores:
// Hkv x total_entries fp32.
inline int64_t score_part_offset(const fa_plan *p) { return scratch_bytes(p->partial_rows); }
inline int64_t plan_scratch_bytes(const fa_plan *p) {
    const int64_t sc = p->representatives ? int64_t(p->dims.num_kv_heads) * p->lay.total_entries * 4 : 0;
    return scratch_bytes(p->partial_rows) + ((sc + kAlign - 1) / kAlign) * kAlign;
}
}  // namespace fa
