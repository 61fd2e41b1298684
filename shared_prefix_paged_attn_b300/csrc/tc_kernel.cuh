// Shared-run kernel: attention of up to 256 stacked query rows (two M = 128 tiles) over one
// chunk of physical KV pages, on the 5th-generation tensor cores.
//
// Agentrix (gitlink.org.cn), section "初赛基础与决赛演进", CUDA ForkAttention: the KV pages
// that several branches share are read once for all of their queries.  The Ascend variant
// described in the same page's section "不同显卡与 AI 加速卡" packs the queries of several
// branches into one fused-attention call per segment.  Here the packing is a tile: every
// (branch, query token, query head of the KV head's GQA group) reading the chunk is one row
// of Q, so S = Q K^T and O += P V are dense M = 128 contractions on tcgen05.
//
// Persistent: the planner's number of CTAs (one per SM, the others left to the row kernels)
// take work items (chunk x KV head x row group of <= 256 rows) from a counter in the plan
// buffer; each CTA of 20 warps runs its items one after another, keeping its TMEM and
// re-initialising its mbarriers in between.  Per item:
//   warps 0 and 2        TMA producers: per 128-token tile, warp 0 loads the 8 pages of K into
//                        a 2-stage K ring, warp 2 the 8 pages of V into a 3-stage V ring, one
//                        4 KiB box per page (128-byte swizzle; a producer warp issues about
//                        one box per 100-160 cycles, so fewer, larger boxes keep it ahead);
//                        pages past the chunk's end are read at an out-of-range page index,
//                        which the copy fills with zeros;
//   warp 1               MMA issuer (one lane issues, the warp waits converged): each M
//                        tile's [P V, next QK^T] as one unit, the two tiles alternating;
//                        it allocates the 512 TMEM columns:
//                        O0 [0,128) O1 [128,256) S0/P0 [256,384) S1/P1 [384,512);
//   warp 3               idle;
//   warps 4-7, 8-11      softmax of M tile 0, columns 0-63 and 64-127 of each tile;
//   warps 12-15, 16-19   the same for M tile 1.  One row per thread (TMEM lane = row): S
//                        from TMEM, mask (visibility words, chunk end, causal limit), the
//                        row maximum of the two halves exchanged through shared memory,
//                        base-2 online softmax with a lazy rescale (the running max is only
//                        raised when a row's maximum grows by more than 2^8, which keeps
//                        P <= 256), P as bf16 written back over S in TMEM for the P V MMA.
// Two warpgroups per M tile halve each thread's share of a tile's exponentials, so a tile's
// softmax fits in the time the tensor core spends on the other M tile's MMAs.  The
// epilogue normalises O and writes the final output (single-chunk rows) or an fp32 partial
// (O, natural-log LSE) for the merge kernel.  Every wait is bounded (the exchange of row
// maxima too: it is an mbarrier, not a named barrier); on expiry the CTA sets the error word,
// drains its copies and MMAs (bounded) and frees its TMEM.
#pragma once
#include <cstddef>

#include "decode_params.cuh"
#include "ptx.cuh"
#include "tc_ptx.cuh"

namespace fa {
namespace tck {

constexpr int kTilePages = 8;
constexpr int kTileTok = kTilePages * kPageSize;   // 128 tokens per KV tile
constexpr int kHalfBytes = kTileTok * 128;          // 64 dims of 128 tokens: 16 KiB
constexpr int kTileBytes = 2 * kHalfBytes;          // 32 KiB per tile of K (or V)
constexpr int kKStages = 2;
constexpr int kVStages = 3;
constexpr int kRows = 2 * kTcRows;                  // 256 rows per work item
constexpr int kQHalf = kRows * 128;                 // 64 dims of 256 rows: 32 KiB
constexpr int kSoftmaxWGs = 4;                      // two per M tile (column halves)
constexpr int kThreads = 128 * (1 + kSoftmaxWGs);   // 640
// Register split (setmaxnreg): the block launches with kLaunchRegs per thread; warpgroup 0
// (producers, MMA warps) gives registers back, the four softmax warpgroups take more.
// 128 * kLowRegs + 512 * kHighRegs must not exceed 640 * (launch registers), which the host
// checks against the compiled kernel before the first launch.
constexpr int kLaunchRegs = 96;
constexpr int kLowRegs = 64;
constexpr int kHighRegs = 104;
static_assert(128 * kLowRegs + 128 * kSoftmaxWGs * kHighRegs <= kThreads * kLaunchRegs, "register split fits the launch");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256;

struct Smem {
    alignas(1024) uint8_t q[2 * kQHalf];
    alignas(1024) uint8_t k[kKStages][kTileBytes];
    alignas(1024) uint8_t v[kVStages][kTileBytes];
    alignas(8) uint64_t kfull[kKStages], kfree[kKStages], vfull[kVStages], vfree[kVStages];
    uint64_t sfull[2], pfull[2], odone[2], xfull[2], fin;
    float xmax[2][2][kTcRows];  // per M tile and column half: a tile's row maxima (then row sums)
    uint32_t tmem_base;
    int32_t abort;
    int32_t item;  // the work item the CTA is on (persistent CTAs take items from a queue)
};
// The struct's size is a multiple of its 1024-byte alignment; the bytes in use end at its
// last member, and what is left before the end is the slack for aligning the dynamic shared
// memory base (the kernel checks that it suffices).
constexpr size_t kSmemBytes = sizeof(Smem);
constexpr size_t kSmemUsed = offsetof(Smem, item) + sizeof(int32_t);
static_assert(kSmemBytes <= 232448, "fits the 227 KiB opt-in shared memory of one CTA");

constexpr uint32_t kIdescQK = tc::idesc_bf16(128, 128, false, false);  // Q, K both K-major
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, 128, false, true);   // P (TMEM), V MN-major

// Bounded wait that also gives up once another role of the CTA has aborted.  A waiting
// thread sleeps in the barrier (at most 20 us per try), so the warps that wait take no issue
// slots from those that work.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const volatile int32_t *abort) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t i = 0; i < ptx::kWaitSpinCap; ++i) {
        if (ptx::mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if ((i & 7u) == 7u && (*abort || ptx::globaltimer() - t0 > ptx::kWaitNs)) return false;
    }
    return false;
}

__device__ __forceinline__ void fail(Smem &sm, int32_t *err) {
    *reinterpret_cast<volatile int32_t *>(&sm.abort) = 1;
    atomicOr(err, kErrTimeout);
}

struct Row {
    int32_t qrow, climit, mask_off, prow;
};

// Row r of a work item -> (query row, causal limit in chunk tokens, visibility words, partial row).
__device__ __forceinline__ Row item_row(const DecodeParams &p, const Item &it, int r) {
    const int4 rec = __ldg(reinterpret_cast<const int4 *>(p.rows + it.row_off + r));
    return Row{rec.x + it.head * p.G, rec.y, rec.z, rec.w < 0 ? -1 : rec.w + it.head};
}

// Producer warp: lanes 0-7 each read one page id of the tile and issue that page's box; lane
// 0 arms the mbarrier first.  Pages past the chunk end are read at an out-of-range page
// index, which the copy fills with zeros.
// K tile: [page][group of 8 tokens][half][8 tokens][64 dims] (one box per page), so that a
// QK^T MMA with N = 128 tokens sees the 8-token groups of a dim-half at a uniform 2 KiB stride.
__device__ __forceinline__ void load_k_tile(const CUtensorMap *map, uint32_t dst, uint32_t bar, int32_t page,
                                            int head, int hkv, int lane) {
    if (lane == 0) ptx::mbar_arrive_expect_tx(bar, kTileBytes);
    __syncwarp();
    if (lane < kTilePages) ptx::tma_load_5d(dst + lane * 4096, map, bar, 0, 0, 0, 0, page * hkv + head);
    __syncwarp();
}

// V tile: [page][half][16 tokens][64 dims] (one box per page); a P V MMA step covers one page.
__device__ __forceinline__ void load_v_tile(const CUtensorMap *map, uint32_t dst, uint32_t bar, int32_t page,
                                            int head, int lane) {
    if (lane == 0) ptx::mbar_arrive_expect_tx(bar, kTileBytes);
    __syncwarp();
    if (lane < kTilePages) ptx::tma_load_5d(dst + lane * 4096, map, bar, 0, 0, 0, head, page);
    __syncwarp();
}

// Producer warps: warp 0 streams K tiles into a 2-stage ring, warp 2 streams V tiles into a
// 3-stage ring (V stays alive one pipeline step longer than K), each running ahead as far as
// its ring allows.
template <bool kIsV>
__device__ __forceinline__ void producer(const DecodeParams &p, Smem &sm, const Item &it, const Chunk &ch, int T,
                                         int lane) {
    constexpr int NS = kIsV ? kVStages : kKStages;
    const int32_t *pages = p.chunk_pages + ch.page_off;
    const volatile int32_t *abort = &sm.abort;
    const CUtensorMap *map = kIsV ? &p.vmap_page : &p.kmap_grp;
    if (lane == 0) ptx::prefetch_tmap(map);
    // every page id of the chunk (<= 256 = 8 x 32) up front: lane l holds pages l + 32 i
    int32_t pid[kMaxChunkPages / 32];
#pragma unroll
    for (int i = 0; i < kMaxChunkPages / 32; ++i) {
        const int idx = 32 * i + lane;
        pid[i] = idx < ch.n_pages ? __ldg(pages + idx) : p.pool_pages;
    }
    // page of tile j seen by lane l < 8: index 8 j + l, held by lane 8 (j % 4) + l in pid[j / 4]
    auto page_of = [&](int j) -> int32_t {
        const int q = j >> 2;
        int32_t v = pid[0];
#pragma unroll
        for (int i = 1; i < kMaxChunkPages / 32; ++i)
            if (q == i) v = pid[i];
        v = __shfl_sync(0xffffffffu, v, 8 * (j & 3) + (lane & 7));
        return (j * kTilePages + lane < ch.n_pages) ? v : p.pool_pages;
    };
    int issued = 0;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
        const int32_t page = page_of(j);
        const int s = j % NS;
        uint64_t &free_bar = kIsV ? sm.vfree[s] : sm.kfree[s];
        uint64_t &full_bar = kIsV ? sm.vfull[s] : sm.kfull[s];
        if (j >= NS) ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&free_bar), (j / NS - 1) & 1, abort));
        if (!ok) break;
        if (kIsV)
            load_v_tile(map, ptx::smem_u32(sm.v[s]), ptx::smem_u32(&full_bar), page, it.head, lane);
        else
            load_k_tile(map, ptx::smem_u32(sm.k[s]), ptx::smem_u32(&full_bar), page, it.head, p.Hkv, lane);
        ++issued;
    }
    if (issued < T && lane == 0) fail(sm, p.err);
    // every copy this warp started must land before the CTA's shared memory goes away
    const volatile int32_t never = 0;
    for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
        wait_bar(ptx::smem_u32(kIsV ? &sm.vfull[j % NS] : &sm.kfull[j % NS]), (j / NS) & 1, &never);
}

// MMA warp (warp 1): every lane waits on the barriers (the warp stays converged); one
// elected lane issues the MMAs and commits.  Per M tile m the chain is softmax(j) ->
// O_m += P_m(j) V_j -> S_m = Q_m K_(j+1)^T -> softmax(j+1) (S_m aliases P_m, so the next
// QK^T follows the P V that reads P_m).  The warp issues each M tile's pair [P V, QK^T] as one
// unit and alternates between the tiles, so the tensor core runs one tile's pair while the
// other tile's softmax runs; the MMAs of two tiles are never interleaved, which would make
// both tiles wait for both pairs and lock their softmaxes in step.
__device__ __forceinline__ void mma_issuer(Smem &sm, uint32_t tmem, int T, int MT, int lane) {
    const volatile int32_t *abort = &sm.abort;
    const uint32_t qa = ptx::smem_u32(sm.q);
    bool ok = true;
    auto wait = [&](uint64_t &bar, uint32_t parity) {
        ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&bar), parity, abort));
        return ok;
    };
    auto commit = [&](uint64_t &bar) {
        if (lane == 0) tc::commit(ptx::smem_u32(&bar));
        __syncwarp();
    };
    // descriptors are warp-uniform values computed by every lane; one elected lane issues
    auto pv_issue = [&](int j, int m) {  // O_m (+)= P_m V_j
        const uint64_t vdesc = tc::sdesc_sw128(ptx::smem_u32(sm.v[j % kVStages]), 2048, 1024);
        const uint32_t d = tmem + kColO + 128 * m, a = tmem + kColS + 128 * m;
        if (tc::elect_one()) {
#pragma unroll
            // page kk of the tile: V +4 KiB per page ((4096 >> 4) in the address field); P of
            // its 16 tokens in 8 columns, those of column half x (pages 4 x .. 4 x + 3) from
            // column 64 x on
            for (int kk = 0; kk < kTilePages; ++kk)
                tc::mma_ts(d, a + 8 * kk + 32 * (kk >> 2), vdesc + uint64_t(kk * (4096 >> 4)), kIdescPV,
                           (j > 0 || kk > 0) ? 1u : 0u);
            tc::commit(ptx::smem_u32(&sm.odone[m]));
        }
        __syncwarp();
    };
    auto qk_issue = [&](int j, int m) {  // S_m = Q_m K_j^T
        const uint64_t qdesc0 = tc::sdesc_sw128(qa + m * (kQHalf / 2), 16, 1024);
        const uint64_t kdesc = tc::sdesc_sw128(ptx::smem_u32(sm.k[j % kKStages]), 16, 2048);
        const uint32_t d = tmem + kColS + 128 * m;
        if (tc::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                // K step kk: dims 16 kk .. 16 kk + 15 = half kk / 4, 32-byte column kk % 4 (Q's
                // halves are 32 KiB apart, K's 1 KiB apart within each 2 KiB token group)
                const uint64_t qoff = uint64_t(((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4);
                const uint64_t koff = uint64_t(((kk >> 2) * 1024 + (kk & 3) * 32) >> 4);
                tc::mma_ss(d, qdesc0 + qoff, kdesc + koff, kIdescQK, kk > 0 ? 1u : 0u);
            }
            tc::commit(ptx::smem_u32(&sm.sfull[m]));
        }
        __syncwarp();
    };
    // S_m(0) of every tile, then per tile j and M tile m: [P_m(j) V_j, Q_m K_(j+1)^T]
    if (wait(sm.kfull[0], 0)) {
        tc::fence_after();
        for (int m = 0; m < MT; ++m) qk_issue(0, m);
        commit(sm.kfree[0]);
        for (int j = 0; j < T && ok; ++j) {
            const bool more = j + 1 < T;
            if (!wait(sm.vfull[j % kVStages], (j / kVStages) & 1)) break;
            for (int m = 0; m < MT; ++m) {
                if (!wait(sm.pfull[m], j & 1)) break;
                tc::fence_after();
                pv_issue(j, m);
                if (more && m == 0 && !wait(sm.kfull[(j + 1) % kKStages], ((j + 1) / kKStages) & 1)) break;
                tc::fence_after();
                if (more) qk_issue(j + 1, m);
            }
            if (!ok) break;
            commit(sm.vfree[j % kVStages]);
            if (more) commit(sm.kfree[(j + 1) % kKStages]);
        }
    }
    if (!ok && lane == 0) *reinterpret_cast<volatile int32_t *>(&sm.abort) = 1;
    // all MMAs are complete before TMEM is reused or freed, and the last arrivals on the
    // stage-free barriers have landed before the barriers are re-initialised for the next item
    commit(sm.fin);
    const volatile int32_t never = 0;
    wait_bar(ptx::smem_u32(&sm.fin), 0, &never);
    if (ok) {
        for (int st = 0; st < kKStages && st < T; ++st) {
            const int jl = st + ((T - 1 - st) / kKStages) * kKStages;  // last tile on stage st
            wait_bar(ptx::smem_u32(&sm.kfree[st]), (jl / kKStages) & 1, &never);
        }
        for (int st = 0; st < kVStages && st < T; ++st) {
            const int jl = st + ((T - 1 - st) / kVStages) * kVStages;
            wait_bar(ptx::smem_u32(&sm.vfree[st]), (jl / kVStages) & 1, &never);
        }
    }
}

// Softmax of M tile m, column half x (tokens 64 x .. 64 x + 63 of each 128-token tile), one
// row per thread.  The two halves of a row share one running maximum: each tile, both write
// their half's maximum to shared memory and arrive on the xfull[m] mbarrier (256 arrivals).
// Once a row has a running maximum, a half does not wait for the other before its
// exponentials: it computes P against the running maximum, then checks both halves' maxima;
// only if a row's maximum grew by more than 2^8 (rare after the first tiles) does it take the
// new maximum, read S from TMEM again and recompute.  Both halves take the same decisions
// from the same numbers.  P of a half goes to the first 32 of its own S columns (so neither
// half writes over S that the other may still read); each half keeps its own running sum and
// the epilogue adds them.
__device__ __forceinline__ void softmax(const DecodeParams &p, Smem &sm, const Chunk &ch, const Row &ri, bool valid,
                                        uint32_t tmem, int T, int m, int x, int wq, int lane) {
    const volatile int32_t *abort = &sm.abort;
    const uint32_t lane_base = uint32_t(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS + 128 * m + 64 * x;  // S columns of this half; P
                                                                      // in the first 32 of them
    const uint32_t tO = tmem + lane_base + kColO + 128 * m + 64 * x;  // its O columns (dims)
    const int row = wq * 32 + lane;
    const uint32_t xbar = ptx::smem_u32(&sm.xfull[m]);
    const int n_tok = ch.n_pages * kPageSize;
    const int n_words = (ch.n_pages + 1) >> 1;
    const float sl2 = p.scale_log2;
    float mrun = -INFINITY, lrun = 0.f;
    bool ok = true;
    // padding rows (zero Q) in a warp with real rows compute finite junk that is never
    // written; a warp of padding rows only keeps the barrier protocol
    const bool any_valid = __any_sync(0xffffffffu, valid);
    uint32_t s[64];
    uint32_t bits[2] = {0xffffffffu, 0xffffffffu};

    auto load_s = [&]() {  // S of this half from TMEM, masked
        tc::ld32(tS + 0, s + 0);
        tc::ld32(tS + 32, s + 32);
        tc::ld_wait();
        tc::tie32(s + 0);
        tc::tie32(s + 32);
        if (__any_sync(0xffffffffu, (bits[0] & bits[1]) != 0xffffffffu)) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
                if (!((bits[c >> 5] >> (c & 31)) & 1u)) s[c] = __float_as_uint(-INFINITY);
        }
    };
    // P = 2^(s * scale * log2 e - muse) as bf16 pairs into pk; returns the row sum of P.  The
    // scale-and-subtract and the sum run on packed fp32 pairs.
    auto exp_pack = [&](float muse, uint32_t (&pk)[32]) {
        const uint64_t sc2 = ptx::f2(sl2, sl2), nm2 = ptx::f2(-muse, -muse);
        uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};  // four pair-chains of the row sum
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            float a0, a1;
            ptx::f2_split(ptx::ffma2(ptx::f2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), sc2, nm2), a0, a1);
            a0 = ptx::ex2(a0);
            a1 = ptx::ex2(a1);
            rs2[c & 3] = ptx::fadd2(rs2[c & 3], ptx::f2(a0, a1));
            pk[c] = ptx::pack_bf16(a0, a1);
        }
        float a0, a1, b0, b1, c0, c1, d0, d1;
        ptx::f2_split(rs2[0], a0, a1);
        ptx::f2_split(rs2[1], b0, b1);
        ptx::f2_split(rs2[2], c0, c1);
        ptx::f2_split(rs2[3], d0, d1);
        return ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
    };
    auto store_p = [&](const uint32_t (&pk)[32]) {
        tc::st16(tS + 0, pk);
        tc::st16(tS + 16, pk + 16);
    };

    // visibility of this half's 64 tokens of tile j for the row: words of the reader, chunk
    // end, causal limit; loaded one tile ahead, so that their latency hides behind a tile
    uint32_t bits_next[2];
    auto tile_bits = [&](int j) {
        const int t0 = j * kTileTok + 64 * x;
        bits_next[0] = bits_next[1] = 0xffffffffu;
        if (valid && j < T && (ri.mask_off >= 0 || t0 + 64 > n_tok || ri.climit < t0 + 63)) {
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const int tq = t0 + 32 * w;
                uint32_t bw = 0xffffffffu;
                if (ri.mask_off >= 0) {
                    const int wi = tq >> 5;
                    bw = wi < n_words ? __ldg(p.mask_words + ri.mask_off + wi) : 0u;
                }
                const int lt = n_tok - tq;
                if (lt < 32) bw &= lt <= 0 ? 0u : ((1u << lt) - 1u);
                const int lc = ri.climit - tq + 1;
                if (lc < 32) bw &= lc <= 0 ? 0u : ((1u << lc) - 1u);
                bits_next[w] = bw;
            }
        }
    };
    tile_bits(0);

    for (int j = 0; j < T; ++j) {
        bits[0] = bits_next[0];
        bits[1] = bits_next[1];
        tile_bits(j + 1);
        ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.sfull[m]), j & 1, abort));
        if (!ok) break;
        if (!any_valid) {
            ptx::mbar_arrive(xbar);
            ok = __all_sync(0xffffffffu, wait_bar(xbar, j & 1, abort));
            if (!ok) break;
            ptx::mbar_arrive(ptx::smem_u32(&sm.pfull[m]));
            continue;
        }
        tc::fence_after();
        load_s();
        // this half's row max with eight independent chains of three-input maxima
        float mxk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mxk[k] = fmaxf(__uint_as_float(s[k]), __uint_as_float(s[k + 8]));
#pragma unroll
        for (int c = 16; c < 64; c += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mxk[k] = ptx::fmax3(mxk[k], __uint_as_float(s[c + k]), __uint_as_float(s[c + k + 8]));
        float mx = fmaxf(fmaxf(fmaxf(mxk[0], mxk[1]), fmaxf(mxk[2], mxk[3])),
                         fmaxf(fmaxf(mxk[4], mxk[5]), fmaxf(mxk[6], mxk[7])));
        if (!valid) mx = 0.f;
        sm.xmax[m][x][row] = mx;
        ptx::mbar_arrive(xbar);

        uint32_t pk[32];
        float lsum;
        bool rescale;
        float alpha = 1.f;
        // after the exchange: both halves' maxima (in the same order in both), and the lazy
        // rescale -- the running max is only raised when it grows by more than 2^8; the two
        // halves of a row see the same numbers, so their warps vote alike
        auto decide = [&]() {
            const float mnew = fmaxf(mrun, fmaxf(sm.xmax[m][0][row], sm.xmax[m][1][row]) * sl2);
            const bool rs = __any_sync(0xffffffffu, mrun != -INFINITY && mnew > mrun + 8.0f);
            if (rs) {
                if (mrun != -INFINITY && mnew > mrun) alpha = ptx::ex2(mrun - mnew);
                if (mnew > mrun) mrun = mnew;
                lrun *= alpha;
            } else if (mrun == -INFINITY) {
                mrun = mnew;
            }
            return rs;
        };
        if (__all_sync(0xffffffffu, mrun != -INFINITY)) {
            // every row of the warp has a running maximum: P against it while the other half's
            // maximum comes in
            lsum = exp_pack(mrun, pk);
            ok = __all_sync(0xffffffffu, wait_bar(xbar, j & 1, abort));
            if (!ok) break;
            rescale = decide();
            if (rescale) {
                // it moved: S again (still in TMEM: only this half writes these columns, and it
                // has not yet) with the new maximum
                load_s();
                lsum = exp_pack(mrun, pk);
            }
        } else {
            ok = __all_sync(0xffffffffu, wait_bar(xbar, j & 1, abort));
            if (!ok) break;
            rescale = decide();
            lsum = exp_pack(mrun == -INFINITY ? 0.f : mrun, pk);
        }
        store_p(pk);
        lrun += lsum;

        if (rescale) {
            // this half of O (the P V MMA of tile j-1 must be done) times alpha
            ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.odone[m]), (j - 1) & 1, abort));
            if (!ok) break;
            tc::fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t o[32];
                tc::ld32(tO + 32 * h, o);
                tc::ld_wait();
                tc::tie32(o);
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                tc::st32(tO + 32 * h, o);
            }
        }
        tc::st_wait();
        tc::fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&sm.pfull[m]));
    }
    if (!ok) {
        if (lane == 0) fail(sm, p.err);
        return;
    }

    // ---- epilogue: O / l, natural-log LSE; l = the two halves' sums (one more exchange) ----
    ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.odone[m]), (T - 1) & 1, abort));
    if (ok) {
        // every thread of the pair is past its last read of xmax (odone follows all pfull)
        sm.xmax[m][x][row] = lrun;
        ptx::mbar_arrive(xbar);
        ok = __all_sync(0xffffffffu, wait_bar(xbar, T & 1, abort));
    }
    if (!ok) {
        if (lane == 0) fail(sm, p.err);
        return;
    }
    if (!any_valid) return;
    const float ltot = sm.xmax[m][0][row] + sm.xmax[m][1][row];
    tc::fence_after();
    const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
    const float lse = ltot > 0.f ? (mrun + log2f(ltot)) * 0.69314718055994531f : -INFINITY;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t o[32];
        tc::ld32(tO + 32 * h, o);
        tc::ld_wait();
        tc::tie32(o);
        if (!valid) continue;
        const int d0 = 64 * x + 32 * h;  // first output dim of these 32 columns
        if (ri.prow >= 0) {
            float *dst = p.part_o + size_t(ri.prow) * kHeadDim + d0;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4 *>(dst + c) =
                    make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                                __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
        } else if (p.out_dtype == FA_F32) {
            float *dst = reinterpret_cast<float *>(p.out) + size_t(ri.qrow) * kHeadDim + d0;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4 *>(dst + c) =
                    make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                                __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
        } else {
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + size_t(ri.qrow) * kHeadDim + d0;
#pragma unroll
            for (int c = 0; c < 32; c += 8)
                *reinterpret_cast<uint4 *>(dst + c) =
                    make_uint4(ptx::pack_bf16(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv),
                               ptx::pack_bf16(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv),
                               ptx::pack_bf16(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv),
                               ptx::pack_bf16(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv));
        }
    }
    if (valid && x == 0) {
        if (ri.prow >= 0) p.part_lse[ri.prow] = lse;
        else p.lse[ri.qrow] = lse;
    }
}

__device__ __forceinline__ void init_barriers(Smem &sm, int MT) {
    for (int s = 0; s < kKStages; ++s) {
        ptx::mbar_init(ptx::smem_u32(&sm.kfull[s]), 1);
        ptx::mbar_init(ptx::smem_u32(&sm.kfree[s]), 1);  // the MMA warp's commit
    }
    for (int s = 0; s < kVStages; ++s) {
        ptx::mbar_init(ptx::smem_u32(&sm.vfull[s]), 1);
        ptx::mbar_init(ptx::smem_u32(&sm.vfree[s]), 1);
    }
    for (int m = 0; m < 2; ++m) {
        ptx::mbar_init(ptx::smem_u32(&sm.sfull[m]), 1);
        ptx::mbar_init(ptx::smem_u32(&sm.pfull[m]), 256);  // both column halves of the M tile
        ptx::mbar_init(ptx::smem_u32(&sm.odone[m]), 1);
        ptx::mbar_init(ptx::smem_u32(&sm.xfull[m]), 256);
    }
    ptx::mbar_init(ptx::smem_u32(&sm.fin), 1);
    ptx::fence_mbar_init();
}

__device__ __forceinline__ void inval_barriers(Smem &sm) {
    uint64_t *first = &sm.kfull[0], *last = &sm.fin;
    for (uint64_t *b = first; b <= last; ++b) ptx::mbar_inval(ptx::smem_u32(b));
}

// Persistent: p.tc_ctas CTAs (one per SM) take work items from a counter in the plan buffer
// (header word 1) until none is left, so that the SMs they leave to the row kernels are
// known and a CTA that runs out of work frees its SM at once.  The last CTA to leave resets
// the counters (header words 1 and 2) for the next decode.
__global__ void __launch_bounds__(kThreads, 1) tc_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
    const uintptr_t base = (raw + 1023) & ~uintptr_t(1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *queue = p.err + 1, *done = p.err + 2;
    ptx::launch_dependents();  // the next kernel of the decode may take the SMs this grid leaves
    if (base - raw + kSmemUsed > kSmemBytes) {  // (uniform) no room to align the buffers
        if (tid == 0) atomicOr(p.err, kErrBounds);
        return;
    }
    Smem &sm = *reinterpret_cast<Smem *>(base);

    auto item_ok = [&](int i) {  // items the planner never makes are refused, uniformly
        const Item it = p.items_tc[i];
        return p.chunks[it.chunk].n_pages <= kMaxChunkPages && it.n_rows <= kRows;
    };
    // the next item this CTA runs (a refused item sets the error word and is skipped)
    auto next_item = [&]() {
        int i = atomicAdd(queue, 1);
        while (i < p.n_items_tc && !item_ok(i)) {
            atomicOr(p.err, kErrBounds);
            i = atomicAdd(queue, 1);
        }
        return i;
    };
    auto item_mt = [&](int i) { return p.items_tc[i].n_rows > kTcRows ? 2 : 1; };

    if (tid == 0) {
        sm.abort = 0;
        sm.item = next_item();
        if (sm.item < p.n_items_tc) init_barriers(sm, item_mt(sm.item));
    }
    if (warp == 1) {
        tc::tmem_alloc(ptx::smem_u32(&sm.tmem_base), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem_base;

    // Each role ends the kernel in its own branch: code after a register re-split must not
    // be shared by warps with different register counts.  Both branches run the same
    // sequence of CTA barriers: per item B (barriers, Q ready), C (item done), D (next item
    // known); then E before TMEM is freed.
    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLowRegs));
        for (;;) {
            const int i = sm.item;
            if (i >= p.n_items_tc) break;
            const Item it = p.items_tc[i];
            const Chunk ch = p.chunks[it.chunk];
            const int T = (ch.n_pages + kTilePages - 1) / kTilePages;
            const int MT = it.n_rows > kTcRows ? 2 : 1;
            tc::fence_before();
            __syncthreads();  // B
            tc::fence_after();
            if (warp == 0) {
                producer<false>(p, sm, it, ch, T, lane);
            } else if (warp == 1) {
                mma_issuer(sm, tmem, T, MT, lane);
            } else if (warp == 2) {
                producer<true>(p, sm, it, ch, T, lane);
            }
            tc::fence_before();
            __syncthreads();  // C
            tc::fence_after();
            if (tid == 0) {
                inval_barriers(sm);
                sm.item = sm.abort ? p.n_items_tc : next_item();
                if (sm.item < p.n_items_tc) init_barriers(sm, item_mt(sm.item));
            }
            __syncthreads();  // D
        }
        if (tid == 0) {
            if (sm.abort) atomicOr(p.err, kErrTimeout);
            __threadfence();
            if (atomicAdd(done, 1) == int(gridDim.x) - 1) {  // no CTA reads the queue any more
                atomicExch(queue, 0);
                atomicExch(done, 0);
            }
        }
        tc::fence_before();
        __syncthreads();  // E
        if (warp == 1) {
            tc::fence_after();
            tc::tmem_dealloc(tmem, kTmemCols);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kHighRegs));
        // softmax warpgroups 1-4 (warps 4-19): M tile sm_m, column half sm_x
        const int wg = (warp >> 2) - 1;
        const int sm_m = wg >> 1, sm_x = wg & 1;
        // TMEM lane quarter of a warp is warp % 4, so row = 128 m + 32 (warp % 4) + lane
        const int r = sm_m * kTcRows + (warp & 3) * 32 + lane;
        for (;;) {
            const int i = sm.item;
            if (i >= p.n_items_tc) break;
            const Item it = p.items_tc[i];
            const Chunk ch = p.chunks[it.chunk];
            const int T = (ch.n_pages + kTilePages - 1) / kTilePages;
            const int MT = it.n_rows > kTcRows ? 2 : 1;
            // the row's table entry, and its half of the Q row -> shared memory, 128-byte
            // swizzled K-major (zeros for padding rows); the previous item's MMAs are all done
            // (barrier C)
            Row ri{0, 0x3fffffff, -1, -1};
            const bool valid = r < it.n_rows;
            if (valid) ri = item_row(p, it, r);
#pragma unroll 4
            for (int c = 8 * sm_x; c < 8 * sm_x + 8; ++c) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (valid) v = __ldg(reinterpret_cast<const uint4 *>(p.q + size_t(ri.qrow) * kHeadDim + c * 8));
                *reinterpret_cast<uint4 *>(sm.q + (c >> 3) * kQHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
            }
            tc::fence_proxy_async_smem();
            tc::fence_before();
            __syncthreads();  // B
            tc::fence_after();
            if (sm_m < MT) softmax(p, sm, ch, ri, valid, tmem, T, sm_m, sm_x, warp & 3, lane);
            tc::fence_before();
            __syncthreads();  // C
            tc::fence_after();
            __syncthreads();  // D
        }
        tc::fence_before();
        __syncthreads();  // E
    }
}

}  // namespace tck
}  // namespace fa
