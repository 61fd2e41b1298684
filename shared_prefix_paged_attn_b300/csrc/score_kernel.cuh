// Key scoring by representative queries: the second pass, on the 5th-generation tensor cores.
//
// AgentKV blog (rit.work), "Как AgentKV выбирает и освобождает записи кэша": before a
// compression the recent queries of every phase are merged into one set of representatives
// (32 in the main experiments); each key is scored by the mean attention the representatives
// give it, and the keys with the largest scores are kept.  For branch b with representatives
// r < R and query heads h < Hq:
//     score(j) = 1 / (R Hq) * sum_{r,h} exp(s_{r,h,j} - lse_{r,h}),   s = scale <q_{r,h}, k_j>,
// lse_{r,h} the log-sum-exp of s_{r,h,.} over the branch's visible entries.  The first pass
// (the decode kernels on a plan of representative queries) gives lse; this kernel recomputes
// S transposed, S^T = K Q^T, one 128-key tile at a time against every row (representative,
// head of the KV head's group, reading branch) of a work item, M = 128 keys, N <= 256 rows,
// and sums exp2(s scale log2 e - lse log2 e) over each reading branch's columns: a score per
// (KV head, key, reading branch), written to a per-head array that the reduce kernel sums.
//
// Persistent CTAs, one per SM, take units (up to 16 tiles of one work item) from a counter in
// the plan's header, in the plan's order: the row groups of one chunk and head sit next to
// each other there, so they run at about the same time on different SMs and read the same K
// tiles through L2.  A CTA's k-th unit is its "segment" k.  Roles:
//   warp 0        TMA producer: each tile's 8 pages of K (two 64-dim boxes per page) into a
//                 2-stage ring, pages past the chunk's end at an out-of-range page index
//                 (zero fill), and an L2 prefetch of the tile two ahead;
//   warp 1        allocates 512 TMEM columns (two accumulators of 256), issues the 8 MMAs of
//                 each tile (one elected lane) into the accumulator the epilogue has freed;
//   warps 2, 3    segment loader: claims the next unit, then loads its item's Q rows
//                 (swizzled as the MMA's B operand), each row's -lse * log2 e and the column
//                 ranges of the reading branches into one of two buffers while the other is
//                 in use;
//   warps 4-7     epilogue: thread t owns key t of the tile (TMEM lane t), reads its 256-column
//                 row 32 columns at a time, sums the exponentials per reading branch and
//                 writes each sum where that branch sees the key.
// Every wait is bounded; on expiry the CTA sets the error word and winds down.
#pragma once
#include "plan_layout.h"
#include "ptx.cuh"
#include "tc_ptx.cuh"

namespace fa {
namespace sck {

constexpr int kTilePages = 8;
constexpr int kTileTok = kTilePages * kPageSize;  // 128 keys per tile
constexpr int kHalfBytes = kTileTok * 128;         // 64 dims of 128 keys: 16 KiB
constexpr int kTileBytes = 2 * kHalfBytes;         // 32 KiB of K per tile
constexpr int kStages = 2;
constexpr int kRows = 256;                         // rows of one work item at most
constexpr int kQHalf = kRows * 128;                // 64 dims of 256 rows: 32 KiB
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;

struct Params {
    CUtensorMap kmap;  // K pages as [pool][Hkv][16][128], boxes of 64 dims x 16 tokens
    const __nv_bfloat16 *q;
    const float *lse;           // [total_q * Hq] natural-log lse of each representative row
    const int32_t *chunk_pages;
    const Chunk *chunks;
    const Item *items;          // the plan's score_items
    const int4 *units;          // [n_units] (item, first tile, tiles, 0)
    const RowRec *rows;
    const int32_t *occ_pos;     // per reader and chunk page: score index of the page's slot 0
    const int32_t *row_pos;     // [rows] the row's reader's run in occ_pos
    const uint32_t *mask_words;
    float *part;                // [Hkv][total_entries] per-head scores
    int32_t *err;
    int32_t *queue;             // work counter (zero at launch)
    int64_t total_entries;
    int32_t n_units, G, pool_pages;
    float scale_log2;
};

struct Smem {
    alignas(1024) uint8_t q[2][2 * kQHalf];
    alignas(1024) uint8_t k[kStages][kTileBytes];
    float nlse2[2][kRows];          // -lse * log2 e per column (-inf: the row sees nothing)
    int32_t seg_base[2][kRows];     // per reading branch (group of columns): its run in occ_pos
    int32_t seg_mask[2][kRows];     // ... and its visibility words (-1: all visible)
    uint32_t seg_last[2][kRows / 32];  // bit c: column c is its group's last
    float span[2][4][32];           // a group's sum over columns < 128, handed to the other half
    alignas(8) uint64_t kfull[kStages], kfree[kStages], accfull[2], accfree[2], unitready[2], qready[2], segfree[2], fin;
    uint64_t spanbar[2][4];
    int32_t unit[2];                // the unit of segment k in unit[k & 1] (-1: no more work)
    uint32_t tmem_base;
    int32_t abort;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "fits the 227 KiB opt-in shared memory of one CTA");

// Bounded wait that also gives up once another role of the CTA has aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const volatile int32_t *abort) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t i = 0; i < ptx::kWaitSpinCap; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && (*abort || ptx::globaltimer() - t0 > ptx::kWaitNs)) return false;
    }
    return false;
}

__device__ __forceinline__ void fail(Smem &sm, int32_t *err) {
    *reinterpret_cast<volatile int32_t *>(&sm.abort) = 1;
    atomicOr(err, kErrTimeout | kErrScore);
}

// Explicit shared-memory loads (the CTA's shared block is reached through an aligned
// pointer, which the compiler would otherwise read with generic loads).
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ int32_t lds_s32(uint32_t a) { return int32_t(lds_u32(a)); }
// Barrier of the two loader warps (named barrier 1, 64 threads) that also ANDs a predicate
// over them.
__device__ __forceinline__ bool bar_and_64(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
        "barrier.cta.red.and.pred po, 1, 64, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(v))
        : "memory");
    return r != 0;
}
__device__ __forceinline__ float sum2(uint64_t v) {
    float lo, hi;
    ptx::f2_split(v, lo, hi);
    return lo + hi;
}

// The unit of segment k, once the loader has claimed it (-1: the queue is empty); false when
// the wait gave up.
__device__ __forceinline__ bool next_unit(Smem &sm, int k, int &u) {
    const bool ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.unitready[k & 1]), (k >> 1) & 1, &sm.abort));
    u = ok ? *reinterpret_cast<volatile int32_t *>(&sm.unit[k & 1]) : -1;
    return ok;
}

// Warp 0: the K tiles of each unit into the 2-stage ring, and an L2 prefetch of the tile two
// ahead in the same unit; returns how many tiles it issued.
__device__ __forceinline__ int producer(const Params &p, Smem &sm, int lane) {
    const volatile int32_t *abort = &sm.abort;
    int c = 0;
    for (int k = 0;; ++k) {
        int u;
        if (!next_unit(sm, k, u)) {
            if (lane == 0) fail(sm, p.err);
            return c;
        }
        if (u < 0) return c;
        const int4 un = p.units[u];
        const Item it = p.items[un.x];
        const int32_t *pages = p.chunk_pages + p.chunks[it.chunk].page_off;
        auto page_of = [&](int kp) { return kp < it.n_pages ? __ldg(pages + kp) : p.pool_pages; };
        for (int j = un.y; j < un.y + un.z; ++j, ++c) {
            const int s = c % kStages;
            if (c >= kStages) {
                const bool ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.kfree[s]), ((c / kStages) - 1) & 1, abort));
                if (!ok) {
                    if (lane == 0) fail(sm, p.err);
                    return c;
                }
            }
            const uint32_t dst = ptx::smem_u32(sm.k[s]), bar = ptx::smem_u32(&sm.kfull[s]);
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar, kTileBytes);
            __syncwarp();
            if (lane < kTilePages) {
                const int32_t page = page_of(j * kTilePages + lane);
                ptx::tma_load_4d(dst + lane * 2048, &p.kmap, bar, 0, 0, it.head, page);
                ptx::tma_load_4d(dst + kHalfBytes + lane * 2048, &p.kmap, bar, 64, 0, it.head, page);
            } else if (lane < 2 * kTilePages && j + 2 < un.y + un.z) {
                const int32_t page = page_of((j + 2) * kTilePages + lane - kTilePages);
                ptx::tma_prefetch_4d(&p.kmap, 0, 0, it.head, page);
                ptx::tma_prefetch_4d(&p.kmap, 64, 0, it.head, page);
            }
            __syncwarp();
        }
    }
}

// Warp 1: per tile, S^T = K Q^T into the free accumulator (N = the item's rows, rounded up
// to 16), then the ring stage is released and the epilogue told.
__device__ __forceinline__ void mma_warp(const Params &p, Smem &sm, uint32_t tmem, int lane) {
    const volatile int32_t *abort = &sm.abort;
    bool ok = true;
    auto wait = [&](uint64_t &bar, uint32_t parity) {
        ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&bar), parity, abort));
        return ok;
    };
    int c = 0;
    for (int k = 0; ok; ++k) {
        int u;
        ok = next_unit(sm, k, u);
        if (!ok || u < 0) break;
        if (!wait(sm.qready[k & 1], (k >> 1) & 1)) break;  // the unit's Q rows are in place
        const int4 un = p.units[u];
        const int n = p.items[un.x].n_rows;
        const uint32_t idesc = tc::idesc_bf16(128, ((n + 15) / 16) * 16, false, false);
        const uint64_t qdesc = tc::sdesc_sw128(ptx::smem_u32(sm.q[k & 1]), 16, 1024);
        for (int j = 0; j < un.z; ++j, ++c) {
            const int s = c % kStages, b = c & 1;
            if (!wait(sm.kfull[s], (c / kStages) & 1)) break;
            if (c >= 2 && !wait(sm.accfree[b], ((c >> 1) - 1) & 1)) break;
            tc::fence_after();
            const uint64_t kdesc = tc::sdesc_sw128(ptx::smem_u32(sm.k[s]), 16, 1024);
            const uint32_t d = tmem + 256 * b;
            if (tc::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    // K step kk: dims 16 kk .. 16 kk + 15 = half kk / 4, 32-byte column kk % 4
                    const uint64_t koff = uint64_t(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
                    const uint64_t qoff = uint64_t(((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4);
                    tc::mma_ss(d, kdesc + koff, qdesc + qoff, idesc, kk > 0 ? 1u : 0u);
                }
                tc::commit(ptx::smem_u32(&sm.accfull[b]));
                tc::commit(ptx::smem_u32(&sm.kfree[s]));
            }
            __syncwarp();
        }
    }
    if (!ok && lane == 0) fail(sm, p.err);
    // every MMA issued is complete before TMEM is freed or the CTA leaves
    if (lane == 0) tc::commit(ptx::smem_u32(&sm.fin));
    __syncwarp();
    const volatile int32_t never = 0;
    wait_bar(ptx::smem_u32(&sm.fin), 0, &never);
}

// Warps 2-3 (64 threads, i = 0..63): segment k claims the next unit of the queue once the
// epilogue is done with segment k - 2 (whose buffers it reuses), announces it, then loads the
// unit's rows into buffer k & 1.
__device__ __forceinline__ void loader(const Params &p, Smem &sm, int i) {
    const volatile int32_t *abort = &sm.abort;
    for (int k = 0;; ++k) {
        const int x = k & 1;
        // both loader warps have passed the wait (and agree on its outcome) before the claim
        const bool ok = bar_and_64(k < 2 || wait_bar(ptx::smem_u32(&sm.segfree[x]), ((k >> 1) - 1) & 1, abort));
        if (!ok) {
            if (i == 0) fail(sm, p.err);
            return;
        }
        if (i == 0) {
            const int u = atomicAdd(p.queue, 1);
            *reinterpret_cast<volatile int32_t *>(&sm.unit[x]) = u < p.n_units ? u : -1;
            ptx::mbar_arrive(ptx::smem_u32(&sm.unitready[x]));
        }
        asm volatile("bar.sync 1, 64;" ::: "memory");
        const int u = *reinterpret_cast<volatile int32_t *>(&sm.unit[x]);
        if (u < 0) return;
        const Item it = p.items[p.units[u].x];
        const int n = it.n_rows;
        const int hq0 = it.head * p.G;
        // per row: -lse log2 e, its reader's run of page positions, its visibility words
        for (int r = i; r < n; r += 64) {
            const RowRec rr = p.rows[it.row_off + r];
            const float l = __ldg(p.lse + rr.qrow0 + hq0);
            sm.nlse2[x][r] = l == -INFINITY ? -INFINITY : -(l * 1.4426950408889634f);
            sm.seg_base[x][r] = __ldg(p.row_pos + it.row_off + r);
            sm.seg_mask[x][r] = rr.mask_off;
        }
        // column c closes its group when the next column reads elsewhere: one ballot per 32
        for (int c = i; c < kRows; c += 64) {
            bool last = false;
            if (c < n) {
                last = c == n - 1 ||
                       __ldg(p.row_pos + it.row_off + c) != __ldg(p.row_pos + it.row_off + c + 1) ||
                       __ldg(&p.rows[it.row_off + c].mask_off) != __ldg(&p.rows[it.row_off + c + 1].mask_off);
            }
            const uint32_t w = __ballot_sync(0xffffffffu, last);
            if ((i & 31) == 0) sm.seg_last[x][c >> 5] = w;
        }
        // Q rows as [half][row][64 dims], 128-byte swizzle: 16-byte chunk ch of row r at half
        // ch / 8, position (ch % 8) ^ (r % 8); eight loads in flight per thread
        uint8_t *qb = sm.q[x];
        for (int base = 0; base < n * 16; base += 64 * 8) {
            uint4 v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int idx = base + e * 64 + i;
                v[e] = make_uint4(0, 0, 0, 0);
                if (idx < n * 16) {
                    const int qrow = __ldg(&p.rows[it.row_off + (idx >> 4)].qrow0) + hq0;
                    v[e] = __ldg(reinterpret_cast<const uint4 *>(p.q + size_t(qrow) * kHeadDim) + (idx & 15));
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int idx = base + e * 64 + i;
                if (idx < n * 16) {
                    const int r = idx >> 4, ch = idx & 15;
                    *reinterpret_cast<uint4 *>(qb + (ch >> 3) * kQHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) = v[e];
                }
            }
        }
        tc::fence_proxy_async_smem();  // the generic writes of Q, seen by the tensor core
        ptx::mbar_arrive(ptx::smem_u32(&sm.qready[x]));
    }
}

// Warps 4-11 (t = 0..255): key k = t % 128 of each tile (TMEM lane k, in the lane quarter
// of warp 4 + t / 32), columns [128 h, 128 h + 128) with h = t / 128.  A group that runs
// across column 128 is summed in two parts: the first half hands its part over through
// span (double-buffered like the accumulators) and the second adds it first.
__device__ __forceinline__ void epilogue(const Params &p, Smem &sm, uint32_t tmem, int t) {
    const volatile int32_t *abort = &sm.abort;
    const int k = t & 127, half = t >> 7, quarter = k >> 5, lane = k & 31;
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    bool ok = true;
    int c = 0;
    uint32_t n_span = 0;  // tiles with a group across column 128: bit b = their count's parity per accumulator b
    for (int seg = 0; ok; ++seg) {
        int u;
        ok = next_unit(sm, seg, u);
        if (!ok || u < 0) break;
        ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.qready[seg & 1]), (seg >> 1) & 1, abort));
        if (!ok) break;
        const int4 un = p.units[u];
        const int item = un.x;
        for (int j = un.y; j < un.y + un.z && ok; ++j, ++c) {
        const int b = c & 1, x = seg & 1;
        // the tile's item, and the key's page position and visibility word for the first
        // column group, loaded before the wait for the accumulator
        const Item it = p.items[item];
        const int kp = j * kTilePages + (k >> 4), slot = k & 15;
        const bool key_ok = kp < it.n_pages;
        const int32_t cp = key_ok ? kp : 0;
        float *part = p.part + size_t(it.head) * size_t(p.total_entries);
        const int n = it.n_rows, col0 = half ? min(128, n - 1) : 0;
        const int mo0 = lds_s32(ptx::smem_u32(&sm.seg_mask[x][col0]));
        const int32_t pos0 = key_ok ? __ldg(p.occ_pos + lds_s32(ptx::smem_u32(&sm.seg_base[x][col0])) + cp) : 0;
        const uint32_t mw0 = (key_ok && mo0 >= 0) ? __ldg(p.mask_words + mo0 + (cp >> 1)) : 0xFFFFFFFFu;
        ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.accfull[b]), (c >> 1) & 1, abort));
        if (!ok) break;
        tc::fence_after();
        const uint32_t nl_addr = ptx::smem_u32(&sm.nlse2[x][0]);
        const uint32_t last_addr = ptx::smem_u32(&sm.seg_last[x][0]);
        float acc = 0.f;
        uint64_t acc2 = 0ull;  // two more running sums (even / odd columns), packed
        bool first = true;     // the key's values for the first column group were loaded early
        // a group across column 128 (the same test in both halves)
        const bool spanning = n > 128 && !((lds_u32(ptx::smem_u32(&sm.seg_last[x][3])) >> 31) & 1u);
        auto flush = [&](int col) {
            float total = acc + sum2(acc2);
            if (first && half && spanning) {  // the first half's part of this group
                ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.spanbar[b][quarter]), (n_span >> b) & 1u, abort));
                total = sm.span[b][quarter][lane] + total;
            }
            acc = 0.f;
            acc2 = 0ull;
            int32_t pos;
            uint32_t mw;
            if (first) {
                pos = pos0;
                mw = mw0;
                first = false;
            } else {
                const int mo = lds_s32(ptx::smem_u32(&sm.seg_mask[x][col]));
                pos = key_ok ? __ldg(p.occ_pos + lds_s32(ptx::smem_u32(&sm.seg_base[x][col])) + cp) : 0;
                mw = (key_ok && mo >= 0) ? __ldg(p.mask_words + mo + (cp >> 1)) : 0xFFFFFFFFu;
            }
            if (key_ok && ((mw >> ((cp & 1) * 16 + slot)) & 1u)) part[pos + slot] = total;
        };
        const uint64_t sl2 = ptx::f2(p.scale_log2, p.scale_log2);
        // columns 32 cc .. 32 cc + 31 of the key's accumulator row, in r
        auto columns = [&](int cc, const uint32_t (&r)[32]) {
            float4 nl[8];  // -lse log2 e of the 32 columns
#pragma unroll
            for (int q = 0; q < 8; ++q) nl[q] = lds_f4(nl_addr + (32 * cc + 4 * q) * 4);
            const uint32_t lastw = lds_u32(last_addr + 4 * cc);
            if (32 * cc + 32 <= n && (lastw & 0x7FFFFFFFu) == 0) {
                // 32 columns of one group (it may end at the last one): packed pairs
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float4 l4 = nl[q >> 1];
                    const uint64_t nl2 = (q & 1) ? ptx::f2(l4.z, l4.w) : ptx::f2(l4.x, l4.y);
                    float e0, e1;
                    ptx::f2_split(ptx::ffma2(ptx::f2(__uint_as_float(r[2 * q]), __uint_as_float(r[2 * q + 1])), sl2, nl2), e0, e1);
                    acc2 = ptx::fadd2(acc2, ptx::f2(ptx::ex2(e0), ptx::ex2(e1)));
                }
                if (lastw >> 31) flush(32 * cc + 31);
            } else {
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int col = 32 * cc + u;
                    if (col < n) {
                        const float4 l4 = nl[u >> 2];
                        const float l = (u & 3) == 0 ? l4.x : (u & 3) == 1 ? l4.y : (u & 3) == 2 ? l4.z : l4.w;
                        acc += ptx::ex2(fmaf(__uint_as_float(r[u]), p.scale_log2, l));
                        if ((lastw >> u) & 1u) flush(col);
                    }
                }
            }
        };
        // two register sets: the next 32 columns load from TMEM while these are summed
        // this half's 32-column chunks [cc0, cc1)
        const int cc0 = 4 * half, cc1 = min(cc0 + 4, (n + 31) / 32);
        const uint32_t acc_addr = tmem + 256 * b + lane_addr;
        uint32_t ra[32], rb[32];
        if (cc0 < cc1) tc::ld32(acc_addr + 32 * cc0, ra);
        for (int cc = cc0; cc < cc1; cc += 2) {
            tc::ld_wait();
            tc::tie32(ra);
            if (cc + 1 < cc1) tc::ld32(acc_addr + 32 * (cc + 1), rb);
            columns(cc, ra);
            if (cc + 1 >= cc1) break;
            tc::ld_wait();
            tc::tie32(rb);
            if (cc + 2 < cc1) tc::ld32(acc_addr + 32 * (cc + 2), ra);
            columns(cc + 1, rb);
        }
        if (spanning) {
            if (half == 0) {  // the open group's part, for the second half
                sm.span[b][quarter][lane] = acc + sum2(acc2);
                ptx::mbar_arrive(ptx::smem_u32(&sm.spanbar[b][quarter]));
            }
            n_span ^= 1u << b;
        }
        if (!ok) break;
        tc::fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&sm.accfree[b]));
        }
        if (ok) ptx::mbar_arrive(ptx::smem_u32(&sm.segfree[seg & 1]));
    }
    if (!ok && (k & 31) == 0) fail(sm, p.err);
}

__global__ void __launch_bounds__(kThreads, 1) score_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    // 1 KiB aligned (128-byte swizzled operands), offset from the shared array itself
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&sm.kfull[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&sm.kfree[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&sm.accfull[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&sm.accfree[b]), 256);
            for (int q = 0; q < 4; ++q) ptx::mbar_init(ptx::smem_u32(&sm.spanbar[b][q]), 32);
            ptx::mbar_init(ptx::smem_u32(&sm.unitready[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&sm.qready[b]), 64);
            ptx::mbar_init(ptx::smem_u32(&sm.segfree[b]), 256);
        }
        ptx::mbar_init(ptx::smem_u32(&sm.fin), 1);
        sm.abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) ptx::prefetch_tmap(&p.kmap);
    if (warp == 1) {
        tc::tmem_alloc(ptx::smem_u32(&sm.tmem_base), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        const int n = producer(p, sm, lane);
        // copies still in flight (an abort) land before the CTA leaves
        const volatile int32_t never = 0;
        for (int c = n - kStages < 0 ? 0 : n - kStages; c < n; ++c)
            wait_bar(ptx::smem_u32(&sm.kfull[c % kStages]), (c / kStages) & 1, &never);
    } else if (warp == 1) {
        mma_warp(p, sm, tmem, lane);
    } else if (warp < 4) {
        loader(p, sm, tid - 64);
    } else {
        epilogue(p, sm, tmem, tid - 128);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// score(j) = (sum over KV heads of the per-head scores) / (R_b Hq); an entry the branch does
// not see keeps the NaN its per-head scores were filled with.
__global__ void __launch_bounds__(256) score_reduce_kernel(const float *part, const int32_t *entry_off,
                                                           const Branch *branches, float *scores,
                                                           int64_t total_entries, int32_t n_branches,
                                                           int32_t hkv, int32_t hq) {
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total_entries;
         e += int64_t(gridDim.x) * blockDim.x) {
        int lo = 0, hi = n_branches - 1;  // the branch whose entries hold e
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(entry_off + mid) <= e) lo = mid; else hi = mid - 1;
        }
        float sum = 0.f;
        for (int g = 0; g < hkv; ++g) sum += part[size_t(g) * size_t(total_entries) + size_t(e)];
        scores[e] = sum / float(int64_t(__ldg(&branches[lo].n_q)) * hq);
    }
}

}  // namespace sck
}  // namespace fa
