// Host planner for fork decode attention over a branching, paged KV cache.
//
// Agentrix (gitlink.org.cn), section "初赛基础与决赛演进", CUDA ForkAttention: the cache is
// split by the pages actually shared into a common part and private parts, the common KV is
// read once for many queries, and per-branch results are merged.  Octopus (zicq.com),
// section "Packed DAG-GRPO", notes that real speed depends on page layout, block-table
// organisation, occupancy and branch imbalance; the planner is where those are decided.
//
// Steps:
//   1. validate the dims and the descriptor (every index is range-checked here, once);
//   2. walk every branch's segments and emit one record per (physical page, reader), where a
//      reader is a branch at a given logical offset; the record carries the 16 visibility
//      bits of that page for that reader (slot in the segment and not dropped);
//   3. group records by physical page: a page's reader set is all of its records;
//   4. chain pages into runs: page p' follows p when every reader of p reads p' at the next
//      16 logical positions and nobody else reads p' (equal reader sets), or, for pages that
//      lie before every reader's query tokens, when the same readers read p' further on;
//      pages that no reader sees at all are skipped;
//   5. cut runs into chunks (long enough that fp32 partial results stay a few percent of the
//      KV bytes, short enough for occupancy: up to 128 pages for the row kernels while a full
//      wave of row items remains, whole 8-page tiles for the tcgen05 kernel), pack per-reader
//      visibility words, give every (chunk, reader) its partial rows (or a direct write when
//      it is the branch's only one);
//   6. emit work items = chunk x KV head x row group and the per-branch merge lists;
//   7. choose the tcgen05 kernel's persistent CTA count by replaying its work counter beside
//      the row work streaming on the SMs left and freed.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <queue>
#include <vector>

#include "plan_internal.h"

namespace {

using fa::kPageSize;

// Time of one 128-token tile of a tcgen05 work item on B300 (microseconds), for the CTA split.
constexpr double kTcTileUs = 2.2;

struct Rec {
    int32_t page;
    int32_t branch;
    int32_t lpos0;  // logical position of the page's slot 0 for this reader
    uint32_t vis;   // 16 bits: slot in the segment and visible
};

struct Input {
    const fa_dims *d;
    const fa_desc *s;
    int32_t G;
    std::vector<int64_t> n_b;
    std::vector<int32_t> q_off;
    bool reps = false;  // representative queries: each sees its branch's whole list
    // logical position of branch b's query token i: the last n_q positions of the branch, or,
    // for representative queries, past the end of the list (no causal limit)
    int64_t qpos(int32_t b, int64_t i) const {
        return reps ? n_b[b] - 1 : n_b[b] - (q_off[b + 1] - q_off[b]) + i;
    }
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t align_up(int64_t a) { return ceil_div(a, fa::kAlign) * fa::kAlign; }

int validate(Input &in) {
    const fa_dims *d = in.d;
    const fa_desc *s = in.s;
    if (d->head_dim != fa::kHeadDim || d->page_size != kPageSize) return FA_ERR_UNSUPPORTED;
    if (d->num_q_heads < 1 || d->num_kv_heads < 1) return FA_ERR_INVALID;
    if (d->num_q_heads % d->num_kv_heads) return FA_ERR_UNSUPPORTED;
    in.G = d->num_q_heads / d->num_kv_heads;
    if (in.G > fa::kRowsMax) return FA_ERR_UNSUPPORTED;
    if (!(d->scale > 0.0f) || !std::isfinite(d->scale)) return FA_ERR_INVALID;
    if (d->out_dtype != FA_BF16 && d->out_dtype != FA_F32) return FA_ERR_INVALID;
    if (s->num_branches < 1 || s->num_pages_pool < 1 || s->num_segs < 0 || s->num_page_ids < 0)
        return FA_ERR_INVALID;
    if (s->num_pages_pool > (int64_t(1) << 31) - 1) return FA_ERR_RANGE;
    // the kernels address a page-head as page x Hkv + head in int32, one page past the pool too
    if ((s->num_pages_pool + 1) * int64_t(d->num_kv_heads) > (int64_t(1) << 31) - 1) return FA_ERR_RANGE;
    if (!s->branch_seg_off || !s->branch_segs) return FA_ERR_NULL;
    if ((s->num_segs > 0 && !s->segs) || (s->num_page_ids > 0 && !s->page_ids)) return FA_ERR_NULL;
    if ((s->vis_bits == nullptr) != (s->vis_word_off == nullptr)) return FA_ERR_INVALID;
    for (int64_t i = 0; i < s->num_page_ids; ++i)
        if (s->page_ids[i] < 0 || s->page_ids[i] >= s->num_pages_pool) return FA_ERR_RANGE;
    for (int32_t i = 0; i < s->num_segs; ++i) {
        const fa_segment &g = s->segs[i];
        if (g.len < 1) return FA_ERR_INVALID;
        if (g.tok_begin < 0 || g.tok_begin >= kPageSize || g.page_off < 0) return FA_ERR_RANGE;
        if (g.page_off + ceil_div(int64_t(g.tok_begin) + g.len, kPageSize) > s->num_page_ids)
            return FA_ERR_RANGE;
    }
    const int32_t B = s->num_branches;
    if (s->branch_seg_off[0] != 0) return FA_ERR_INVALID;
    in.n_b.assign(B, 0);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t e0 = s->branch_seg_off[b], e1 = s->branch_seg_off[b + 1];
        if (e1 <= e0) return FA_ERR_INVALID;  // an empty branch has no query token
        for (int32_t e = e0; e < e1; ++e) {
            const int32_t sg = s->branch_segs[e];
            if (sg < 0 || sg >= s->num_segs) return FA_ERR_RANGE;
            in.n_b[b] += s->segs[sg].len;
        }
        if (in.n_b[b] > (int64_t(1) << 30)) return FA_ERR_INVALID;
    }
    in.q_off.assign(B + 1, 0);
    for (int32_t b = 0; b < B; ++b) {
        const int64_t nq = s->branch_q_off ? int64_t(s->branch_q_off[b + 1]) - s->branch_q_off[b] : 1;
        if (s->branch_q_off && s->branch_q_off[0] != 0) return FA_ERR_INVALID;
        if (nq < 1 || (!in.reps && nq > in.n_b[b])) return FA_ERR_INVALID;
        if (in.reps && nq * in.G > 2 * fa::kTcRows) return FA_ERR_UNSUPPORTED;
        in.q_off[b + 1] = int32_t(in.q_off[b] + nq);
        if (int64_t(in.q_off[b]) + nq > (int64_t(1) << 30)) return FA_ERR_INVALID;
    }
    if (s->vis_bits) {
        if (s->num_vis_words < 0) return FA_ERR_INVALID;
        for (int32_t b = 0; b < B; ++b) {
            const int64_t w0 = s->vis_word_off[b];
            if (w0 < 0 || w0 + ceil_div(in.n_b[b], 32) > s->num_vis_words) return FA_ERR_RANGE;
        }
    }
    return FA_OK;
}

struct Builder {
    Input &in;
    std::vector<Rec> recs;            // in (branch, logical) order
    std::vector<int64_t> branch_rec;  // CSR into recs per branch
    std::vector<int32_t> by_page;     // record ids sorted by (page, branch, lpos0)
    std::vector<int32_t> group_start, group_count, group_of_page;
    std::vector<uint32_t> group_union;

    explicit Builder(Input &i) : in(i) {}

    bool visible(int32_t b, int64_t j) const {
        const fa_desc *s = in.s;
        if (!s->vis_bits) return true;
        const uint32_t w = s->vis_bits[s->vis_word_off[b] + (j >> 5)];
        return (w >> (j & 31)) & 1u;
    }

    void emit_records() {
        const fa_desc *s = in.s;
        branch_rec.assign(s->num_branches + 1, 0);
        for (int32_t b = 0; b < s->num_branches; ++b) {
            int64_t L = 0;
            for (int32_t e = s->branch_seg_off[b]; e < s->branch_seg_off[b + 1]; ++e) {
                const fa_segment &g = s->segs[s->branch_segs[e]];
                const int64_t n_pages = ceil_div(int64_t(g.tok_begin) + g.len, kPageSize);
                for (int64_t k = 0; k < n_pages; ++k) {
                    const int32_t page = s->page_ids[g.page_off + k];
                    const int64_t lo = (k == 0) ? g.tok_begin : 0;
                    const int64_t hi = std::min<int64_t>(kPageSize, g.tok_begin + int64_t(g.len) - kPageSize * k);
                    const int64_t lpos0 = L + kPageSize * k - g.tok_begin;
                    uint32_t vis = 0;
                    for (int64_t sl = lo; sl < hi; ++sl)
                        if (visible(b, lpos0 + sl)) vis |= 1u << sl;
                    if (!recs.empty() && int64_t(recs.size()) > branch_rec[b] &&
                        recs.back().page == page && recs.back().lpos0 == lpos0) {
                        recs.back().vis |= vis;  // a segment boundary inside one page
                    } else {
                        recs.push_back(Rec{page, b, int32_t(lpos0), vis});
                    }
                }
                L += g.len;
            }
            branch_rec[b + 1] = int64_t(recs.size());
        }
    }

    void group_by_page() {
        const int32_t n = int32_t(recs.size());
        by_page.resize(n);
        for (int32_t i = 0; i < n; ++i) by_page[i] = i;
        std::sort(by_page.begin(), by_page.end(), [&](int32_t a, int32_t b) {
            const Rec &x = recs[a], &y = recs[b];
            if (x.page != y.page) return x.page < y.page;
            if (x.branch != y.branch) return x.branch < y.branch;
            return x.lpos0 < y.lpos0;
        });
        group_of_page.assign(in.s->num_pages_pool, -1);
        for (int32_t i = 0; i < n;) {
            int32_t j = i;
            uint32_t u = 0;
            while (j < n && recs[by_page[j]].page == recs[by_page[i]].page) u |= recs[by_page[j++]].vis;
            group_of_page[recs[by_page[i]].page] = int32_t(group_start.size());
            group_start.push_back(i);
            group_count.push_back(j - i);
            group_union.push_back(u);
            i = j;
        }
    }

    // p1 continues p0 when the reader lists match with every logical offset advanced by 16.
    bool chains(int32_t g0, int32_t g1) const {
        if (group_count[g0] != group_count[g1]) return false;
        for (int32_t t = 0; t < group_count[g0]; ++t) {
            const Rec &a = recs[by_page[group_start[g0] + t]];
            const Rec &b = recs[by_page[group_start[g1] + t]];
            if (a.branch != b.branch || int64_t(b.lpos0) != int64_t(a.lpos0) + kPageSize) return false;
        }
        return true;
    }

    // Every reader of page group g sees all of the page before its branch's first query token:
    // no causal cut can fall inside it.
    bool pre_query(int32_t g) const {
        if (in.reps) return true;  // no causal limit at all
        for (int32_t t = 0; t < group_count[g]; ++t) {
            const Rec &a = recs[by_page[group_start[g] + t]];
            if (int64_t(a.lpos0) + kPageSize > in.qpos(a.branch, 0)) return false;
        }
        return true;
    }

    // p1 may join p0's run although not logically adjacent: the same readers, each reading p1
    // entirely after p0 (their order is kept) and entirely before its queries.
    bool jumps(int32_t g0, int32_t g1) const {
        if (group_count[g0] != group_count[g1]) return false;
        for (int32_t t = 0; t < group_count[g0]; ++t) {
            const Rec &a = recs[by_page[group_start[g0] + t]];
            const Rec &b = recs[by_page[group_start[g1] + t]];
            if (a.branch != b.branch || int64_t(b.lpos0) < int64_t(a.lpos0) + kPageSize) return false;
        }
        return pre_query(g1);
    }

    // Runs follow one branch's pages in logical order.  A page joins the run when every
    // reader reads it right after the previous one, or -- while the whole run lies before
    // every reader's queries -- when it has the same readers further on (attention over such
    // tokens does not depend on their order or position, so a chunk may gather the visible
    // pieces around dropped ones; the kernels' causal test then never cuts it).  Pages nobody
    // sees are skipped.
    std::vector<std::vector<int32_t>> build_runs() {
        std::vector<std::vector<int32_t>> runs;
        std::vector<char> assigned(group_start.size(), 0);
        for (int32_t b = 0; b < in.s->num_branches; ++b) {
            for (int64_t r = branch_rec[b]; r < branch_rec[b + 1]; ++r) {
                const int32_t g = group_of_page[recs[r].page];
                if (assigned[g]) continue;
                assigned[g] = 1;
                if (group_union[g] == 0) continue;  // no reader sees this page: never read it
                std::vector<int32_t> run{g};
                bool all_pre = pre_query(g), jumped = false;
                int64_t cur = r;
                for (int64_t nx_i = r + 1; nx_i < branch_rec[b + 1]; ++nx_i) {
                    const Rec &nx = recs[nx_i];
                    const int32_t g1 = group_of_page[nx.page];
                    if (group_union[g1] == 0) continue;  // unseen pages leave no gap in a chunk
                    if (assigned[g1]) break;
                    const bool adjacent = int64_t(nx.lpos0) == int64_t(recs[cur].lpos0) + kPageSize &&
                                          nx_i == cur + 1 && chains(run.back(), g1);
                    const bool pre1 = pre_query(g1);
                    if (adjacent && (!jumped || pre1)) {
                        // plain continuation
                    } else if (all_pre && jumps(run.back(), g1)) {
                        jumped = true;
                    } else {
                        break;
                    }
                    all_pre = all_pre && pre1;
                    assigned[g1] = 1;
                    run.push_back(g1);
                    cur = nx_i;
                }
                runs.push_back(std::move(run));
            }
        }
        return runs;
    }
};

struct Emit {
    std::vector<int32_t> chunk_pages;
    std::vector<fa::Chunk> chunks;
    std::vector<fa::Occ> occs;
    std::vector<fa::Item> items_rows, items_tc, items_r8;
    std::vector<fa::RowRec> rows;
    std::vector<fa::Branch> branches;
    std::vector<fa::QMerge> q_merge;
    std::vector<int32_t> merge_bases;
    std::vector<int32_t> merge_lpos;  // first logical position of each partial's chunk
    // representative queries only (key scoring)
    std::vector<fa::Item> score_items;
    std::vector<int32_t> score_units, occ_pos, row_pos, entry_off, word_off;  // units: (item, tile0, tiles, 0)
    std::vector<uint32_t> mask_words;
};

int build_plan(Input &in, const fa_plan_opts &opts, fa_plan *plan) {
    Builder bd(in);
    bd.emit_records();
    bd.group_by_page();
    std::vector<std::vector<int32_t>> runs = bd.build_runs();

    const fa_desc *s = in.s;
    const int32_t B = s->num_branches, G = in.G, Hkv = in.d->num_kv_heads;
    Emit em;
    fa_plan_stats &st = plan->stats;
    std::memset(&st, 0, sizeof st);

    // representative queries: every run on the tcgen05 kernel, so that a branch's rows of one
    // chunk (n_q x G <= 256) always sit in one row group, which the scoring pass needs
    const int32_t tmin = in.reps ? 1
                                 : opts.tensor_min_rows < 0 ? 0 : (opts.tensor_min_rows > 0 ? opts.tensor_min_rows : 64);
    auto run_rows = [&](const std::vector<int32_t> &run) {  // stacked rows of a run's readers
        const int32_t g0 = run[0];
        int64_t rows = 0;
        for (int32_t t = 0; t < bd.group_count[g0]; ++t) {
            const Rec &rd = bd.recs[bd.by_page[bd.group_start[g0] + t]];
            rows += int64_t(in.q_off[rd.branch + 1] - in.q_off[rd.branch]) * G;
        }
        return rows;
    };
    // Chunk size of the row kernels' runs: longer chunks mean fewer per-item prologues and
    // fewer partials to merge, as long as enough items are left to fill every SM with row
    // CTAs at the end of the decode (one wave: three CTAs on each of 148 SMs).  The largest of
    // 128, 96, 64 pages that keeps that many row items (measured on B300: the long-context
    // rolling-drop decode 221 -> 213 us at 128 pages; the flat-fork one, with 256 items at
    // 64 pages, lost 8% at 128).
    int32_t base_pages = 64;
    if (opts.chunk_pages > 0) {
        base_pages = opts.chunk_pages;
    } else {
        const int64_t want = 3 * 148;
        for (int32_t cand : {128, 96}) {
            int64_t items = 0;
            for (const auto &run : runs) {
                const int64_t rows = run_rows(run);
                if (tmin > 0 && rows >= tmin) continue;
                const int64_t target = std::min<int64_t>(std::max<int64_t>(cand, 2 * rows), fa::kMaxChunkPages);
                items += std::max<int64_t>(1, ceil_div(int64_t(run.size()), target)) *
                         ceil_div(std::max<int64_t>(rows, 1), fa::kRowsMax) * Hkv;
            }
            if (items >= want) {
                base_pages = cand;
                break;
            }
        }
    }
    // key scoring: branch b's entries are scores[entry_off[b] .. + n_b), its keep bits the
    // words word_off[b] .. + ceil(n_b / 32)
    if (in.reps) {
        int64_t e = 0, wsum = 0;
        for (int32_t b = 0; b < B; ++b) {
            em.entry_off.push_back(int32_t(e));
            em.word_off.push_back(int32_t(wsum));
            e += in.n_b[b];
            wsum += ceil_div(in.n_b[b], 32);
            if (e > (int64_t(1) << 31) - 1 || e * Hkv > (int64_t(1) << 40)) return FA_ERR_UNSUPPORTED;
        }
        em.entry_off.push_back(int32_t(e));
        em.word_off.push_back(int32_t(wsum));
    }

    std::vector<char> chunk_tc;  // per chunk: its items go to the tcgen05 kernel
    std::vector<int64_t> chunk_slots;  // per chunk: visible slots of its pages (any reader)
    std::vector<int32_t> occ_count(B, 0);
    for (const auto &run : runs) {
        const int32_t g0 = run[0];
        const int32_t n_read = bd.group_count[g0];
        const int64_t rows = run_rows(run);
        // fp32 partial rows cost rows * 1 KiB (write + read) per chunk and KV head; a chunk of
        // n pages carries n * 8 KiB of K+V, so n >= 2 * rows keeps partials near 6% of KV.
        int64_t target = std::max<int64_t>(base_pages, 2 * rows);
        if (opts.chunk_pages > 0) target = opts.chunk_pages;
        target = std::min<int64_t>(target, fa::kMaxChunkPages);
        const bool tc_run = tmin > 0 && rows >= tmin;
        if (tc_run && opts.tensor_chunk_pages > 0)
            target = std::min<int64_t>(fa::kMaxChunkPages, ceil_div(opts.tensor_chunk_pages, 8) * 8);
        const int64_t n = int64_t(run.size());
        const int64_t n_ch = std::max<int64_t>(1, ceil_div(n, target));
        // tcgen05 chunks are whole 128-token tiles (8 pages) except the last one of a run
        const int64_t tc_len = ceil_div(ceil_div(n, n_ch), 8) * 8;
        int64_t pos = 0;
        for (int64_t c = 0; pos < n; ++c) {
            const int64_t len = tc_run ? std::min(tc_len, n - pos) : n / n_ch + (c < n % n_ch ? 1 : 0);
            fa::Chunk ch;
            ch.page_off = int32_t(em.chunk_pages.size());
            ch.n_pages = int32_t(len);
            ch.occ_off = int32_t(em.occs.size());
            ch.n_occ = n_read;
            int64_t slots_c = 0;
            for (int64_t k = 0; k < len; ++k) {
                const int32_t g = run[pos + k];
                em.chunk_pages.push_back(bd.recs[bd.by_page[bd.group_start[g]]].page);
                st.unique_visible_slots += __builtin_popcount(bd.group_union[g]);
                (tc_run ? st.unique_slots_tensor : st.unique_slots_rows) += __builtin_popcount(bd.group_union[g]);
                slots_c += __builtin_popcount(bd.group_union[g]);
                st.touched_pages += 1;
                for (int32_t t = 0; t < n_read; ++t) {
                    const Rec &rd = bd.recs[bd.by_page[bd.group_start[g] + t]];
                    st.listed_visible_slots += __builtin_popcount(rd.vis);
                    // QK^T and P V: 2 x 128 multiply-adds per (query row, KV head, visible slot
                    // at or before the query token's position); query tokens from the first
                    // one whose position is past the page's last slot see all of its slots
                    const int64_t nq = in.q_off[rd.branch + 1] - in.q_off[rd.branch];
                    const int64_t qpos0 = in.qpos(rd.branch, 0);
                    const int64_t i_full = in.reps ? 0 : std::min<int64_t>(nq, std::max<int64_t>(0, int64_t(rd.lpos0) + kPageSize - 1 - qpos0));
                    int64_t pairs = (nq - i_full) * __builtin_popcount(rd.vis);
                    for (int64_t i = std::max<int64_t>(0, int64_t(rd.lpos0) - qpos0); i < i_full; ++i) {
                        const int64_t cut = qpos0 + i - rd.lpos0;  // slots s <= cut are causally visible
                        if (cut >= 0) pairs += __builtin_popcount(rd.vis & ((2u << cut) - 1u));
                    }
                    (tc_run ? st.flops_tensor : st.flops_rows) += pairs * G * Hkv * 4 * fa::kHeadDim;
                }
            }
            for (int32_t t = 0; t < n_read; ++t) {
                const Rec &rd = bd.recs[bd.by_page[bd.group_start[run[pos]] + t]];
                fa::Occ oc;
                oc.branch = rd.branch;
                oc.lpos0 = rd.lpos0;
                oc.prow_base = 0;  // assigned below
                bool all = true;
                for (int64_t k = 0; k < len && all; ++k)
                    all = bd.recs[bd.by_page[bd.group_start[run[pos + k]] + t]].vis == 0xFFFFu;
                if (all) {
                    oc.mask_off = -1;
                } else {
                    oc.mask_off = int32_t(em.mask_words.size());
                    for (int64_t k = 0; k < len; k += 2) {
                        uint32_t w = bd.recs[bd.by_page[bd.group_start[run[pos + k]] + t]].vis;
                        if (k + 1 < len) w |= bd.recs[bd.by_page[bd.group_start[run[pos + k + 1]] + t]].vis << 16;
                        em.mask_words.push_back(w);
                    }
                }
                oc.pos_off = -1;
                if (in.reps) {  // every page's slot-0 score index for this reader
                    oc.pos_off = int32_t(em.occ_pos.size());
                    for (int64_t k = 0; k < len; ++k) {
                        const Rec &rk = bd.recs[bd.by_page[bd.group_start[run[pos + k]] + t]];
                        em.occ_pos.push_back(int32_t(em.entry_off[rk.branch] + rk.lpos0));
                    }
                    if (em.occ_pos.size() > size_t(INT32_MAX)) return FA_ERR_UNSUPPORTED;
                }
                em.occs.push_back(oc);
                occ_count[rd.branch] += 1;
            }
            em.chunks.push_back(ch);
            chunk_tc.push_back(tc_run ? 1 : 0);
            chunk_slots.push_back(slots_c);
            pos += len;
        }
    }

    // partial rows: a branch read by a single occurrence writes `out` directly
    em.branches.resize(B);
    std::vector<std::vector<int32_t>> per_branch(B), per_branch_lpos(B);
    int64_t prow = 0;
    for (size_t o = 0; o < em.occs.size(); ++o) {
        const int32_t b = em.occs[o].branch;
        if (occ_count[b] == 1) {
            em.occs[o].prow_base = -1;
        } else {
            em.occs[o].prow_base = int32_t(prow);
            per_branch[b].push_back(int32_t(prow));
            per_branch_lpos[b].push_back(em.occs[o].lpos0);
            prow += int64_t(in.q_off[b + 1] - in.q_off[b]) * G * Hkv;
            if (prow > (int64_t(1) << 31) - 1) return FA_ERR_UNSUPPORTED;
        }
    }
    // partials merged in all, and those in rows of more than kMergeInline partials (the
    // merge kernel's long path): when those are most of them and the rows are few, the merge
    // keeps more of a row's partial loads in flight (measured on B300: the flat-fork merge,
    // 512 rows of 18 partials, 11.3 -> 9.9 us and the kv-DAG one, 1024 rows, 13.7 -> 12.1 us;
    // the rolling-drop one, 4096 rows, unchanged, and the multi-tree one, 65536 rows, 69 ->
    // 81 us for want of resident warps)
    int64_t merged_all = 0, merged_long = 0;
    for (int32_t b = 0; b < B; ++b) {
        fa::Branch &br = em.branches[b];
        std::memset(&br, 0, sizeof br);
        br.q_begin = in.q_off[b];
        br.n_q = in.q_off[b + 1] - in.q_off[b];
        br.qpos0 = int32_t(in.qpos(b, 0));
        br.merge_off = int32_t(em.merge_bases.size());
        br.n_merge = int32_t(per_branch[b].size());
        br.direct = occ_count[b] == 1;
        em.merge_bases.insert(em.merge_bases.end(), per_branch[b].begin(), per_branch[b].end());
        em.merge_lpos.insert(em.merge_lpos.end(), per_branch_lpos[b].begin(), per_branch_lpos[b].end());
        for (int32_t i = 0; i < br.n_q; ++i) {
            fa::QMerge qm;
            std::memset(&qm, 0, sizeof qm);
            qm.merge_off = br.merge_off;
            qm.n_merge = br.n_merge;
            qm.direct = br.direct;
            qm.i = i;
            qm.pos = int32_t(in.qpos(b, i));
            for (int32_t k = 0; k < std::min(br.n_merge, fa::kMergeInline); ++k) {
                qm.base[k] = per_branch[b][k];
                qm.lpos[k] = per_branch_lpos[b][k];
            }
            em.q_merge.push_back(qm);
        }
        if (occ_count[b] != 1) {
            st.merge_rows += int64_t(br.n_q) * in.d->num_q_heads;
            merged_all += int64_t(br.n_q) * br.n_merge;
            if (br.n_merge > fa::kMergeInline) merged_long += int64_t(br.n_q) * br.n_merge;
        }
    }

    // work items: chunk x KV head x row group (row groups shared by every head); row groups
    // hold <= 32 rows for the row kernel and <= 256 rows (two M = 128 tiles) for tcgen05
    const int32_t Hq = in.d->num_q_heads;
    for (size_t c = 0; c < em.chunks.size(); ++c) {
        const fa::Chunk &ch = em.chunks[c];
        const bool tc = chunk_tc[c] != 0;
        const int32_t max_rows = tc ? 2 * fa::kTcRows : fa::kRowsMax;
        const int32_t q_per_piece = std::max(1, max_rows / G);
        std::vector<std::pair<int32_t, int32_t>> groups;  // (row_off, n_rows)
        int32_t cur_off = int32_t(em.rows.size()), cur_rows = 0;
        for (int32_t t = 0; t < ch.n_occ; ++t) {
            const fa::Occ &oc = em.occs[ch.occ_off + t];
            const fa::Branch &br = em.branches[oc.branch];
            for (int32_t i0 = 0; i0 < br.n_q; i0 += q_per_piece) {
                const int32_t ni = std::min(q_per_piece, br.n_q - i0);
                if (cur_rows + ni * G > max_rows) {
                    groups.push_back({cur_off, cur_rows});
                    cur_off = int32_t(em.rows.size());
                    cur_rows = 0;
                }
                for (int32_t i = i0; i < i0 + ni; ++i)
                    for (int32_t jh = 0; jh < G; ++jh) {
                        fa::RowRec r;
                        r.qrow0 = (br.q_begin + i) * Hq + jh;
                        r.climit = int32_t(in.qpos(oc.branch, i) - oc.lpos0);
                        r.mask_off = oc.mask_off;
                        r.prow0 = oc.prow_base < 0 ? -1 : oc.prow_base + (i * G + jh) * Hkv;
                        em.rows.push_back(r);
                        if (in.reps) em.row_pos.push_back(oc.pos_off);
                    }
                cur_rows += ni * G;
            }
        }
        if (cur_rows) groups.push_back({cur_off, cur_rows});
        if (!tc) {  // the visible slots each row kernel must read (once per launch)
            bool r8 = false, r32 = false;
            for (const auto &gr : groups) (gr.second <= 8 ? r8 : r32) = true;
            if (r8) st.unique_slots_row8 += chunk_slots[c];
            if (r32) st.unique_slots_row32 += chunk_slots[c];
        }
        // pages each row group can see: up to its largest causal limit.  A group whose rows all
        // lie before the chunk sees nothing of it and gets no item at all -- unless a row of
        // it writes `out` directly (its branch's only chunk, no merge to fill the row in): then
        // one page, which every row sees nothing of (out 0, lse -inf)
        std::vector<int32_t> group_pages(groups.size());
        for (size_t gi = 0; gi < groups.size(); ++gi) {
            int32_t lim = -1;
            bool direct = false;
            for (int32_t r = groups[gi].first; r < groups[gi].first + groups[gi].second; ++r) {
                lim = std::max(lim, em.rows[r].climit);
                direct = direct || em.rows[r].prow0 < 0;
            }
            group_pages[gi] = lim < 0 ? (direct ? 1 : 0)
                                      : int32_t(std::min<int64_t>(ch.n_pages, int64_t(lim) / kPageSize + 1));
        }
        for (int32_t h = 0; h < Hkv; ++h) {
            for (size_t gi = 0; gi < groups.size(); ++gi) {
                if (group_pages[gi] == 0) {
                    if (h == 0) st.items_skipped += 1;
                    continue;
                }
                fa::Item it;
                std::memset(&it, 0, sizeof it);
                it.chunk = int32_t(c);
                it.head = h;
                it.row_off = groups[gi].first;
                it.n_rows = groups[gi].second;
                it.n_pages = group_pages[gi];
                const int64_t kv = int64_t(it.n_pages) * kPageSize * fa::kHeadDim * 2 * 2;
                if (tc) {
                    em.items_tc.push_back(it);
                    st.kv_bytes_tensor += kv;
                } else {
                    (it.n_rows <= 8 ? em.items_r8 : em.items_rows).push_back(it);
                    st.kv_bytes_rows += kv;
                }
            }
        }
        if (em.rows.size() > size_t(INT32_MAX)) return FA_ERR_UNSUPPORTED;
    }

    // longest items first (stable, so a chunk's row groups and heads stay adjacent and share
    // its pages in L2): the last wave of CTAs is made of short items
    auto by_len = [&](const fa::Item &a, const fa::Item &b) {
        return a.n_pages > b.n_pages;
    };
    std::stable_sort(em.items_tc.begin(), em.items_tc.end(), by_len);
    std::stable_sort(em.items_rows.begin(), em.items_rows.end(), by_len);
    std::stable_sort(em.items_r8.begin(), em.items_r8.end(), by_len);
    if (in.reps) {  // the scoring pass takes every item, in units of <= 16 128-key tiles
        for (const auto *list : {&em.items_tc, &em.items_rows, &em.items_r8})
            em.score_items.insert(em.score_items.end(), list->begin(), list->end());
        for (size_t i = 0; i < em.score_items.size(); ++i) {
            const int32_t tiles = int32_t(ceil_div(em.score_items[i].n_pages, 8));
            for (int32_t t0 = 0; t0 < tiles; t0 += fa::kScoreUnitTiles) {
                em.score_units.push_back(int32_t(i));
                em.score_units.push_back(t0);
                em.score_units.push_back(std::min(fa::kScoreUnitTiles, tiles - t0));
                em.score_units.push_back(0);
            }
            if (em.score_units.size() > size_t(INT32_MAX)) return FA_ERR_UNSUPPORTED;
        }
    }

    // Persistent CTAs of the tcgen05 kernel: the SMs it holds while the row kernels stream
    // the private runs on the others (and on each SM a tcgen05 CTA leaves once the work
    // counter runs dry).  For every candidate count n the planner replays the device's work
    // counter -- items in queue order, each to the CTA that frees first -- and lets the row
    // work stream on the SMs left and freed, then keeps the n whose last kernel ends first.
    // Rates measured on B300: a tcgen05 item costs about kTcTileUs per 128-token tile plus
    // 2 us; row work streams about 85 GB/s per SM beside it and at most 6.2 TB/s in all.  fa_plan_opts.tensor_ctas > 0
    // overrides the choice.
    {
        const int sms = opts.num_sms > 0 ? opts.num_sms : 148;
        int n_best = std::max<int>(1, std::min<int64_t>(sms, int64_t(em.items_tc.size())));
        if (!em.items_tc.empty() && st.kv_bytes_rows > 0) {
            std::vector<double> cost(em.items_tc.size());
            for (size_t i = 0; i < em.items_tc.size(); ++i)
                cost[i] = kTcTileUs * 1e-6 * double((em.items_tc[i].n_pages + 7) / 8) + 2e-6;
            const double row_bytes = double(st.kv_bytes_rows), rate_sm = 85e9, rate_all = 6.2e12;
            double t_best = 1e30;
            std::vector<double> fin;
            for (int n = 1; n <= std::min<int64_t>(sms, int64_t(em.items_tc.size())); ++n) {
                // list scheduling in queue order: a min-heap of CTA finish times
                std::priority_queue<double, std::vector<double>, std::greater<double>> heap;
                for (int c = 0; c < n; ++c) heap.push(0.0);
                for (double c : cost) {
                    const double t = heap.top();
                    heap.pop();
                    heap.push(t + c);
                }
                fin.clear();
                while (!heap.empty()) {
                    fin.push_back(heap.top());
                    heap.pop();
                }
                // row work on the free SMs: sms - n, plus one more at each CTA's finish time
                double left = row_bytes, t = 0.0;
                int free_sms = sms - n;
                for (size_t e = 0; e <= fin.size() && left > 0.0; ++e) {
                    const double t_next = e < fin.size() ? fin[e] : 1e30;
                    const double rate = std::min(rate_all, rate_sm * free_sms);
                    if (rate > 0.0 && left <= rate * (t_next - t)) {
                        t += left / rate;
                        left = 0.0;
                        break;
                    }
                    left -= rate * (t_next - t);
                    t = t_next;
                    ++free_sms;
                }
                const double t_end = std::max(fin.back(), t);
                if (t_end < t_best * 0.999) {  // the smallest n within 0.1% of the best
                    t_best = t_end;
                    n_best = n;
                }
            }
        }
        int n = opts.tensor_ctas > 0 ? opts.tensor_ctas : n_best;
        n = std::max(1, std::min(n, sms));
        plan->tc_ctas = int32_t(std::min<int64_t>(n, std::max<size_t>(em.items_tc.size(), 1)));
        st.tensor_ctas = em.items_tc.empty() ? 0 : plan->tc_ctas;
    }

    st.num_chunks = int64_t(em.chunks.size());
    st.num_items_rows = int64_t(em.items_rows.size()) + int64_t(em.items_r8.size());
    st.num_items_row8 = int64_t(em.items_r8.size());
    st.num_items_tensor = int64_t(em.items_tc.size());
    st.partial_rows = prow;
    st.total_q = in.q_off[B];
    if (em.items_rows.size() > size_t(INT32_MAX) || em.items_tc.size() > size_t(INT32_MAX) ||
        em.items_r8.size() > size_t(INT32_MAX) ||
        em.chunk_pages.size() > size_t(INT32_MAX))
        return FA_ERR_UNSUPPORTED;

    // blob layout
    fa::Layout &L = plan->lay;
    std::memset(&L, 0, sizeof L);
    int64_t off = fa::kAlign;  // error word
    auto place = [&](int64_t bytes) { const int64_t at = off; off = align_up(off + std::max<int64_t>(bytes, 1)); return at; };
    L.chunk_pages = place(int64_t(em.chunk_pages.size()) * 4);
    L.chunks = place(int64_t(em.chunks.size()) * sizeof(fa::Chunk));
    L.items_rows = place(int64_t(em.items_rows.size()) * sizeof(fa::Item));
    L.items_tc = place(int64_t(em.items_tc.size()) * sizeof(fa::Item));
    L.items_r8 = place(int64_t(em.items_r8.size()) * sizeof(fa::Item));
    L.rows = place(int64_t(em.rows.size()) * sizeof(fa::RowRec));
    L.branches = place(int64_t(em.branches.size()) * sizeof(fa::Branch));
    L.q_merge = place(int64_t(em.q_merge.size()) * sizeof(fa::QMerge));
    L.merge_bases = place(int64_t(em.merge_bases.size()) * 4);
    L.merge_lpos = place(int64_t(em.merge_lpos.size()) * 4);
    L.mask_words = place(int64_t(em.mask_words.size()) * 4);
    L.score_items = place(int64_t(em.score_items.size()) * sizeof(fa::Item));
    L.score_units = place(int64_t(em.score_units.size()) * 4);
    L.occ_pos = place(int64_t(em.occ_pos.size()) * 4);
    L.row_pos = place(int64_t(em.row_pos.size()) * 4);
    L.entry_off = place(int64_t(em.entry_off.size()) * 4);
    L.word_off = place(int64_t(em.word_off.size()) * 4);
    L.total = off;
    L.n_score_items = int32_t(em.score_items.size());
    L.n_score_units = int32_t(em.score_units.size() / 4);
    L.total_entries = em.entry_off.empty() ? 0 : em.entry_off.back();
    L.total_words = em.word_off.empty() ? 0 : em.word_off.back();
    L.n_chunk_pages = int32_t(em.chunk_pages.size());
    L.n_chunks = int32_t(em.chunks.size());
    L.n_items_rows = int32_t(em.items_rows.size());
    L.n_items_tc = int32_t(em.items_tc.size());
    L.n_items_r8 = int32_t(em.items_r8.size());
    L.n_rows = int32_t(em.rows.size());
    L.n_branches = B;
    L.total_q = in.q_off[B];
    L.n_merge_bases = int32_t(em.merge_bases.size());
    L.n_mask_words = int32_t(em.mask_words.size());
    plan->blob.assign(size_t(L.total), 0);
    auto put = [&](int64_t at, const void *src, size_t bytes) { if (bytes) std::memcpy(plan->blob.data() + at, src, bytes); };
    put(L.chunk_pages, em.chunk_pages.data(), em.chunk_pages.size() * 4);
    put(L.chunks, em.chunks.data(), em.chunks.size() * sizeof(fa::Chunk));
    put(L.items_rows, em.items_rows.data(), em.items_rows.size() * sizeof(fa::Item));
    put(L.items_tc, em.items_tc.data(), em.items_tc.size() * sizeof(fa::Item));
    put(L.items_r8, em.items_r8.data(), em.items_r8.size() * sizeof(fa::Item));
    put(L.rows, em.rows.data(), em.rows.size() * sizeof(fa::RowRec));
    put(L.branches, em.branches.data(), em.branches.size() * sizeof(fa::Branch));
    put(L.q_merge, em.q_merge.data(), em.q_merge.size() * sizeof(fa::QMerge));
    put(L.merge_bases, em.merge_bases.data(), em.merge_bases.size() * 4);
    put(L.merge_lpos, em.merge_lpos.data(), em.merge_lpos.size() * 4);
    put(L.mask_words, em.mask_words.data(), em.mask_words.size() * 4);
    put(L.score_items, em.score_items.data(), em.score_items.size() * sizeof(fa::Item));
    put(L.score_units, em.score_units.data(), em.score_units.size() * 4);
    put(L.occ_pos, em.occ_pos.data(), em.occ_pos.size() * 4);
    put(L.row_pos, em.row_pos.data(), em.row_pos.size() * 4);
    put(L.entry_off, em.entry_off.data(), em.entry_off.size() * 4);
    put(L.word_off, em.word_off.data(), em.word_off.size() * 4);
    plan->partial_rows = prow;
    plan->representatives = in.reps;
    plan->merge_wide = 2 * merged_long > merged_all && st.merge_rows <= 2048;
    return FA_OK;
}

}  // namespace

extern "C" int fork_attn_plan_create(const fa_dims *dims, const fa_desc *desc,
                                     const fa_plan_opts *opts, fa_plan **out_plan) {
    if (!dims || !desc || !out_plan) return FA_ERR_NULL;
    try {
        Input in{dims, desc, 0, {}, {}};
        fa_plan_opts o;
        std::memset(&o, 0, sizeof o);
        if (opts) o = *opts;
        in.reps = o.representatives == 1;
        int rc = validate(in);
        if (rc != FA_OK) return rc;
        if (o.chunk_pages < 0 || o.num_sms < 0 || o.tensor_ctas < 0 || o.tensor_chunk_pages < 0 ||
            (o.representatives != 0 && o.representatives != 1) || o.reserved[0] || o.reserved[1])
            return FA_ERR_INVALID;
        fa_plan *p = new fa_plan();
        p->dims = *dims;
        p->G = in.G;
        p->num_pages_pool = desc->num_pages_pool;
        p->dev_plan = nullptr;
        p->dev_scratch = nullptr;
        p->uploaded = false;
        p->err_word = nullptr;
        rc = build_plan(in, o, p);
        if (rc != FA_OK) {
            delete p;
            return rc;
        }
        *out_plan = p;
        return FA_OK;
    } catch (const std::bad_alloc &) {
        return FA_ERR_NOMEM;
    }
}

extern "C" int fork_attn_plan_sizes(const fa_plan *plan, size_t *plan_bytes, size_t *scratch_bytes) {
    if (!plan || !plan_bytes || !scratch_bytes) return FA_ERR_NULL;
    *plan_bytes = size_t(plan->lay.total);
    *scratch_bytes = size_t(fa::plan_scratch_bytes(plan));
    return FA_OK;
}

extern "C" int fork_attn_plan_stats(const fa_plan *plan, fa_plan_stats *stats) {
    if (!plan || !stats) return FA_ERR_NULL;
    *stats = plan->stats;
    return FA_OK;
}

extern "C" int fork_attn_plan_destroy(fa_plan *plan) {
    delete plan;
    return FA_OK;
}

extern "C" const char *fork_attn_strerror(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_NULL: return "a required pointer is NULL";
        case FA_ERR_INVALID: return "malformed descriptor or dimensions";
        case FA_ERR_UNSUPPORTED: return "shape not supported (head_dim 128, page_size 16, Hq % Hkv == 0, G <= 32)";
        case FA_ERR_RANGE: return "an index is out of range";
        case FA_ERR_ALIGN: return "a device pointer is not suitably aligned";
        case FA_ERR_NOT_UPLOADED: return "plan not uploaded";
        case FA_ERR_CUDA: return "a CUDA call failed";
        case FA_ERR_NOMEM: return "host allocation failed";
        case FA_ERR_BUFFER_SMALL: return "a caller buffer is too small";
        case FA_ERR_DEVICE: return "a kernel reported a device-side fault";
        case FA_ERR_SCRATCH_LIMIT: return "plan needs more device memory than the built-in static scratch array holds";
        default: return "unknown status";
    }
}
