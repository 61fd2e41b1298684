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
// buffer; each CTA of 12 warps runs its items one after another, keeping its TMEM and
// re-initialising its mbarriers in between.  Per item:
//   warps 0 and 2        TMA producers: per 128-token tile, warp 0 loads the 8 pages of K as
//                        2 KiB boxes (64 dims x 16 tokens, 128-byte swizzle) into a 2-stage
//                        K ring, warp 2 the 8 pages of V as whole 4 KiB page boxes into a
//                        2-stage V ring; pages past the chunk's end are read at an
//                        out-of-range page index, which the copy fills with zeros;
//   warps 1 and 3        MMA issuers for M tile 0 and 1 (one lane issues, the warp waits
//                        converged); warp 1 allocates the 512 TMEM columns:
//                        O0 [0,128) O1 [128,256) S0 [256,384) S1 [384,512);
//   warps 4-7, 8-11      softmax of M tile 0 and 1 (one row per thread, TMEM lane = row):
//                        S from TMEM, mask (visibility words, chunk end, causal limit), base-2
//                        online softmax with a lazy rescale (the running max is only raised
//                        when a row's maximum grows by more than 2^8, which keeps P <= 256),
//                        P as bf16 into a shared-memory buffer, the A operand of the P V MMA.
// S and P live apart, so the next tile's S = Q K^T is issued as soon as the softmax has
// loaded S into registers and runs during that softmax: each M tile's chain is one softmax
// after another, the MMAs beside it.  The one P buffer serves both M tiles in turn (tile j:
// M tile 0, then 1), in two 64-token halves: a softmax writes a half once the P V that read
// that half last is done, and hands each half to the P V as soon as it is stored.
// The epilogue normalises O and writes the final output (single-chunk rows) or an fp32
// partial (O, natural-log LSE) for the merge kernel.  Every wait is bounded; on expiry the
// CTA sets the error word, drains its copies and MMAs (bounded) and frees its TMEM.
#pragma once
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
constexpr int kVStages = 2;
constexpr int kRows = 2 * kTcRows;                  // 256 rows per work item
constexpr int kQHalf = kRows * 128;                 // 64 dims of 256 rows: 32 KiB
constexpr int kPHalf = kTcRows * 128;               // 64 tokens of P for 128 rows: 16 KiB
constexpr int kThreads = 384;
// Register split (setmaxnreg): the block launches with kLaunchRegs per thread; warpgroup 0
// (producer, MMA, two idle warps) gives registers back, the two softmax warpgroups take
// more.  128 * kLowRegs + 256 * kHighRegs must not exceed 384 * (launch registers), which
// the host checks against the compiled kernel before the first launch.
constexpr int kLaunchRegs = 168;
constexpr int kLowRegs = 80;
constexpr int kHighRegs = 208;
static_assert(128 * kLowRegs + 256 * kHighRegs <= kThreads * kLaunchRegs, "register split fits the launch");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256;

struct Smem {
    alignas(1024) uint8_t q[2 * kQHalf];
    alignas(1024) uint8_t k[kKStages][kTileBytes];
    alignas(1024) uint8_t v[kVStages][kTileBytes];
    alignas(1024) uint8_t pb[2 * kPHalf];  // P of one M tile: [token half][128 rows][64 tokens], swizzled
    alignas(8) uint64_t kfull[kKStages], kfree[kKStages], vfull[kVStages], vfree[kVStages];
    uint64_t sfull[2], sfree[2], pfull[2][2], odone[2][2], fin;  // P full / O done per token half
    uint32_t tmem_base;
    int32_t abort;
    int32_t item;  // the work item the CTA is on (persistent CTAs take items from a queue)
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "fits the 227 KiB opt-in shared memory of one CTA");

constexpr uint32_t kIdescQK = tc::idesc_bf16(128, 128, false, false);  // Q, K both K-major
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, 128, false, true);   // P K-major, V MN-major

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
    atomicOr(err, kErrTimeout | kErrTc);
}

struct Row {
    int32_t qrow, climit, mask_off, prow;
};

// Row r of a work item -> (query row, causal limit in chunk tokens, visibility words, partial row).
__device__ __forceinline__ Row item_row(const DecodeParams &p, const Item &it, int r) {
    const int4 rec = __ldg(reinterpret_cast<const int4 *>(p.rows + it.row_off + r));
    Row row{rec.x + it.head * p.G, rec.y, rec.z, rec.w < 0 ? -1 : rec.w + it.head};
    checked_row(p, row.qrow, row.prow, row.mask_off, it.n_pages, kErrTc);
    return row;
}

// Producer warp: lanes 0-7 each read one page id of the tile and issue that page's two
// boxes (64 dims each); lane 0 arms the mbarrier first.  Pages past the chunk end are read
// at an out-of-range page index, which the copy fills with zeros.
// K tile: [half][128 tokens][64 dims] (two boxes per page), so that a QK^T MMA with N = 128
// tokens sees 8-token groups at a uniform 1 KiB stride.
__device__ __forceinline__ void load_k_tile(const CUtensorMap *map, uint32_t dst, uint32_t bar, int32_t page,
                                            int head, int lane) {
    if (lane == 0) ptx::mbar_arrive_expect_tx(bar, kTileBytes);
    __syncwarp();
    if (lane < kTilePages) {
        ptx::tma_load_4d(dst + lane * 2048, map, bar, 0, 0, head, page);
        ptx::tma_load_4d(dst + kHalfBytes + lane * 2048, map, bar, 64, 0, head, page);
    }
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

// Producer warps: warp 0 streams K tiles, warp 2 V tiles, each into a 2-stage ring, running
// ahead as far as its ring allows.
template <bool kIsV>
__device__ __forceinline__ void producer(const DecodeParams &p, Smem &sm, const Item &it, const Chunk &ch, int T,
                                         int lane) {
    constexpr int NS = kIsV ? kVStages : kKStages;
    const int32_t *pages = p.chunk_pages + ch.page_off;
    const volatile int32_t *abort = &sm.abort;
    const CUtensorMap *map = kIsV ? &p.vmap_page : &p.kmap;
    if (lane == 0) ptx::prefetch_tmap(map);
    // every page id of the chunk (<= 256 = 8 x 32) up front: lane l holds pages l + 32 i
    int32_t pid[kMaxChunkPages / 32];
#pragma unroll
    for (int i = 0; i < kMaxChunkPages / 32; ++i) {
        const int idx = 32 * i + lane;
        pid[i] = idx < ch.n_pages ? __ldg(pages + idx) : p.pool_pages;
        if (kChecked && idx < ch.n_pages && (pid[i] < 0 || pid[i] >= p.pool_pages)) {
            atomicOr(p.err, kErrBounds | kErrTc);  // read as the zero-filled page past the pool
            pid[i] = p.pool_pages;
        }
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
            load_k_tile(map, ptx::smem_u32(sm.k[s]), ptx::smem_u32(&full_bar), page, it.head, lane);
        ++issued;
    }
    if (issued < T && lane == 0) fail(sm, p.err);
    // every copy this warp started must land before the CTA's shared memory goes away
    const volatile int32_t never = 0;
    for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
        wait_bar(ptx::smem_u32(kIsV ? &sm.vfull[j % NS] : &sm.kfull[j % NS]), (j / NS) & 1, &never);
}

// MMA warps: warp 1 issues every S = Q K^T, warp 3 every O (+)= P V, each for the M tiles in
// turn, so that a Q K^T waits only for its S to be free and its K tile -- never behind a P V
// that waits for a softmax.  Every lane waits on the barriers (the warp stays converged);
// one elected lane issues the MMAs and commits.  Per tile j and M tile m:
//   warp 1: once K_j has landed and the softmax has loaded S_m(j-1) (S free),
//           S_m = Q_m K_j^T; after the M tiles, one commit releases K_j;
//   warp 3: once V_j has landed and each token half of P_m(j) is in the shared buffer
//           (P full of that half), O_m (+)= P_m(j) V_j over that half, committing O done
//           of (M tile m, half); after the M tiles, one commit releases V_j (lse only: no
//           P V).
__device__ __forceinline__ void mma_issuer(Smem &sm, uint32_t tmem, int T, int MT, bool is_pv, int lane, bool lse_only) {
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
    const uint64_t pdesc0 = tc::sdesc_sw128(ptx::smem_u32(sm.pb), 16, 1024);
    auto pv = [&](int j, int m, int h) {  // O_m (+)= P_m V_j over tokens 64 h .. 64 h + 63
        const uint64_t vdesc = tc::sdesc_sw128(ptx::smem_u32(sm.v[j % kVStages]), 2048, 1024);
        const uint32_t d = tmem + kColO + 128 * m;
        if (tc::elect_one()) {
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
                // K step kk = page kk: tokens 16 kk .. 16 kk + 15 of P (token half h, 32-byte
                // column kq); +4 KiB per page of V: (4096 >> 4) in the address field
                const int kk = 4 * h + kq;
                const uint64_t poff = uint64_t((h * kPHalf + kq * 32) >> 4);
                tc::mma_ss(d, pdesc0 + poff, vdesc + uint64_t(kk * (4096 >> 4)), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
            }
            tc::commit(ptx::smem_u32(&sm.odone[m][h]));
        }
        __syncwarp();
    };
    auto qk = [&](int j, int m) {  // S_m = Q_m K_j^T
        const uint64_t qdesc0 = tc::sdesc_sw128(qa + m * (kQHalf / 2), 16, 1024);
        const uint64_t kdesc = tc::sdesc_sw128(ptx::smem_u32(sm.k[j % kKStages]), 16, 1024);
        const uint32_t d = tmem + kColS + 128 * m;
        if (tc::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                // K step kk: dims 16 kk .. 16 kk + 15 = half kk / 4, 32-byte column kk % 4
                const uint64_t qoff = uint64_t(((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4);
                const uint64_t koff = uint64_t(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
                tc::mma_ss(d, qdesc0 + qoff, kdesc + koff, kIdescQK, kk > 0 ? 1u : 0u);
            }
            tc::commit(ptx::smem_u32(&sm.sfull[m]));
        }
        __syncwarp();
    };
    for (int j = 0; j < T && ok; ++j) {
        if (!is_pv) {
            if (!wait(sm.kfull[j % kKStages], (j / kKStages) & 1)) break;
            for (int m = 0; m < MT && ok; ++m) {
                if (j > 0 && !wait(sm.sfree[m], (j - 1) & 1)) break;
                tc::fence_after();
                qk(j, m);
            }
            if (ok) commit(sm.kfree[j % kKStages]);
        } else if (!lse_only) {
            if (!wait(sm.vfull[j % kVStages], (j / kVStages) & 1)) break;
            for (int m = 0; m < MT && ok; ++m) {
                for (int h = 0; h < 2 && ok; ++h) {
                    if (!wait(sm.pfull[m][h], j & 1)) break;
                    tc::fence_after();
                    pv(j, m, h);
                }
            }
            if (ok) commit(sm.vfree[j % kVStages]);
        }
    }
    if (!ok && lane == 0) *reinterpret_cast<volatile int32_t *>(&sm.abort) = 1;
    // all MMAs issued by either MMA warp are complete before TMEM is reused or freed (fin
    // takes one arrival per MMA warp), and the last arrivals on the stage-free barriers have
    // landed before the barriers are re-initialised for the next item
    if (is_pv && lse_only) {
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sm.fin));  // issued no MMA
        __syncwarp();
    } else {
        commit(sm.fin);
    }
    const volatile int32_t never = 0;
    wait_bar(ptx::smem_u32(&sm.fin), 0, &never);
    if (ok && !is_pv) {
        for (int st = 0; st < kKStages && st < T; ++st) {
            const int jl = st + ((T - 1 - st) / kKStages) * kKStages;  // last tile on stage st
            wait_bar(ptx::smem_u32(&sm.kfree[st]), (jl / kKStages) & 1, &never);
        }
    }
    if (ok && is_pv && !lse_only) {
        for (int st = 0; st < kVStages && st < T; ++st) {
            const int jl = st + ((T - 1 - st) / kVStages) * kVStages;
            wait_bar(ptx::smem_u32(&sm.vfree[st]), (jl / kVStages) & 1, &never);
        }
    }
}

// Softmax warpgroup of M tile m (MT M tiles in use).  Per tile: S from TMEM, then S free for
// the next Q K^T; P into registers, then each token half into the shared buffer once the P V
// that read that half last is done, and P full of that half.
template <bool kLse>
__device__ __forceinline__ void softmax(const DecodeParams &p, Smem &sm, const Chunk &ch, const Row &ri, bool valid, uint32_t tmem,
                        int T, int m, int MT, int wq, int lane) {
    const volatile int32_t *abort = &sm.abort;
    const uint32_t lane_base = uint32_t(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS + 128 * m;
    const uint32_t tO = tmem + lane_base + kColO + 128 * m;
    const int n_tok = ch.n_pages * kPageSize;
    const int n_words = (ch.n_pages + 1) >> 1;
    const float sl2 = p.scale_log2;
    float mrun = -INFINITY, lrun = 0.f;
    bool ok = true;
    auto wait = [&](uint64_t &bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&bar), parity, abort)) != 0;
    };
    // The P buffer's uses go M tile 0, M tile 1 per tile (two M tiles) or tile after tile
    // (one), each in two token halves: the P V of an M tile commits O done of half h once it
    // has read that half.  The use before (tile j, M tile m) is M tile 0's of tile j (m = 1),
    // M tile 1's of tile j - 1 (m = 0), or the M tile's own of tile j - 1 -- and that use's
    // second half being done implies that this M tile's own P V of tile j - 1 is, which the O
    // rescale needs.
    auto pbuf_free = [&](int j, int h) {
        if (MT == 2 && m == 1) return wait(sm.odone[0][h], j & 1);
        return j == 0 || wait(sm.odone[MT == 2 ? 1 : 0][h], (j - 1) & 1);
    };

    if (!__any_sync(0xffffffffu, valid)) {
        // a warp of padding rows only keeps the barrier protocol (its rows of P are stale,
        // and its rows of O are never written); waiting for the P buffer keeps its arrival
        // on P full from running ahead into the next tile's phase
        for (int j = 0; j < T && ok; ++j) {
            ok = wait(sm.sfull[m], j & 1);
            if (!ok) break;
            ptx::mbar_arrive(ptx::smem_u32(&sm.sfree[m]));
            for (int h = 0; h < 2 && ok && !kLse; ++h) {
                ok = pbuf_free(j, h);
                if (ok) ptx::mbar_arrive(ptx::smem_u32(&sm.pfull[m][h]));
            }
        }
        if (!ok && lane == 0) fail(sm, p.err);
        return;
    }
    const uint32_t prow = ptx::smem_u32(sm.pb) + uint32_t(wq * 32 + lane) * 128;  // this row of P
    const uint32_t pswz = uint32_t(lane & 7);  // row % 8: the row's 16-byte chunk swizzle
    // the reader's visibility words of tile jj (all ones without a mask or past the chunk,
    // which the chunk-end mask then clears), fetched one tile ahead so that their latency
    // overlaps the tile before
    const bool has_mask = valid && ri.mask_off >= 0;
    auto fetch = [&](int jj, uint32_t(&w4)[4]) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int wi = 4 * jj + w;
            w4[w] = has_mask && wi < n_words ? __ldg(p.mask_words + ri.mask_off + wi) : 0xffffffffu;
        }
    };
    uint32_t nxt[4];
    fetch(0, nxt);
    for (int j = 0; j < T; ++j) {
        // visibility of the tile's 128 tokens for this row: words of the reader, chunk end,
        // causal limit; computed while the MMA runs
        const int t0 = j * kTileTok;
        uint32_t bits[4] = {nxt[0], nxt[1], nxt[2], nxt[3]};
        if (j + 1 < T) fetch(j + 1, nxt);
        if (valid && (t0 + kTileTok > n_tok || ri.climit < t0 + kTileTok - 1)) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int tq = t0 + 32 * w;
                const int lt = n_tok - tq;
                if (lt < 32) bits[w] &= lt <= 0 ? 0u : ((1u << lt) - 1u);
                const int lc = ri.climit - tq + 1;
                if (lc < 32) bits[w] &= lc <= 0 ? 0u : ((1u << lc) - 1u);
            }
        }
        ok = wait(sm.sfull[m], j & 1);
        if (!ok) break;
        tc::fence_after();
        uint32_t s[128];
        tc::ld32(tS + 0, s + 0);
        tc::ld32(tS + 32, s + 32);
        tc::ld32(tS + 64, s + 64);
        tc::ld32(tS + 96, s + 96);
        tc::ld_wait();
        tc::tie32(s + 0);
        tc::tie32(s + 32);
        tc::tie32(s + 64);
        tc::tie32(s + 96);
        // S is in registers: the next tile's Q K^T may overwrite it
        tc::fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&sm.sfree[m]));

        if (__any_sync(0xffffffffu, (bits[0] & bits[1] & bits[2] & bits[3]) != 0xffffffffu)) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
                if (!((bits[c >> 5] >> (c & 31)) & 1u)) s[c] = __float_as_uint(-INFINITY);
        }
        // row max with eight independent chains of three-input maxima
        float mxk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mxk[k] = fmaxf(__uint_as_float(s[k]), __uint_as_float(s[k + 8]));
#pragma unroll
        for (int c = 16; c < 128; c += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mxk[k] = ptx::fmax3(mxk[k], __uint_as_float(s[c + k]), __uint_as_float(s[c + k + 8]));
        float mx = fmaxf(fmaxf(fmaxf(mxk[0], mxk[1]), fmaxf(mxk[2], mxk[3])),
                         fmaxf(fmaxf(mxk[4], mxk[5]), fmaxf(mxk[6], mxk[7])));
        if (!valid) mx = 0.f;  // a padding row (zero Q) in a warp with real rows: finite junk
        const float mnew = fmaxf(mrun, mx * sl2);
        // lazy rescale: the running max is only raised when it grows by more than 2^8
        const bool rescale = __any_sync(0xffffffffu, mrun != -INFINITY && mnew > mrun + 8.0f);
        float alpha = 1.f;
        if (rescale) {
            if (mrun != -INFINITY && mnew > mrun) alpha = ptx::ex2(mrun - mnew);
            if (mnew > mrun) mrun = mnew;
            lrun *= alpha;
        } else if (mrun == -INFINITY) {
            mrun = mnew;
        }
        const float muse = mrun == -INFINITY ? 0.f : mrun;

        // P = 2^(s * scale * log2 e - m) as bf16 pairs, first into registers (while the other
        // M tile's P V reads the buffer); the scale-and-subtract and the row sum run on packed
        // fp32 pairs
        const uint64_t sc2 = ptx::f2(sl2, sl2), nm2 = ptx::f2(-muse, -muse);
        uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};  // four pair-chains of the row sum
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            float x, y;
            ptx::f2_split(ptx::ffma2(ptx::f2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), sc2, nm2), x, y);
            x = ptx::ex2(x);
            y = ptx::ex2(y);
            rs2[c & 3] = ptx::fadd2(rs2[c & 3], ptx::f2(x, y));
            pk[c] = ptx::pack_bf16(x, y);
        }
        {
            float a0, a1, b0, b1, c0, c1, d0, d1;
            ptx::f2_split(rs2[0], a0, a1);
            ptx::f2_split(rs2[1], b0, b1);
            ptx::f2_split(rs2[2], c0, c1);
            ptx::f2_split(rs2[3], d0, d1);
            lrun += ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
        }
        if (!kLse) {
            // then into the buffer, half by half, once the P V that read that half last is
            // done: tokens 8 c8 .. 8 c8 + 7 are 16-byte chunk c8 % 8 of the row in token half
            // c8 / 8; a half is handed to the P V as soon as it is stored
            ok = pbuf_free(j, 0);
            if (!ok) break;
            tc::fence_after();
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                ptx::st_shared_v4(prow + ((uint32_t(c8) ^ pswz) << 4), pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2],
                                  pk[4 * c8 + 3]);
            if (rescale) {
                // O of the previous tiles times alpha, before the P V of this tile starts; this M
                // tile's P V of tile j - 1 is done once the second half's last use is
                ok = pbuf_free(j, 1);
                if (!ok) break;
                tc::fence_after();
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t o[32];
                    tc::ld32(tO + 32 * h, o);
                    tc::ld_wait();
                    tc::tie32(o);
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    tc::st32(tO + 32 * h, o);
                }
                tc::st_wait();
            }
            tc::fence_proxy_async_smem();  // P, written through the generic proxy, to the MMA
            tc::fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&sm.pfull[m][0]));
            ok = pbuf_free(j, 1);
            if (!ok) break;
            tc::fence_after();
#pragma unroll
            for (int c8 = 8; c8 < 16; ++c8)
                ptx::st_shared_v4(prow + kPHalf + ((uint32_t(c8 & 7) ^ pswz) << 4), pk[4 * c8], pk[4 * c8 + 1],
                                  pk[4 * c8 + 2], pk[4 * c8 + 3]);
            tc::fence_proxy_async_smem();
            tc::fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&sm.pfull[m][1]));
        }
    }
    if (!ok) {
        if (lane == 0) fail(sm, p.err);
        return;
    }

    // ---- epilogue: O / l, natural-log LSE (lse only: zero partial O rows, no out) ----
    if (!kLse) {
        ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.odone[m][1]), (T - 1) & 1, abort));
        if (!ok) {
            if (lane == 0) fail(sm, p.err);
            return;
        }
        tc::fence_after();
    }
    const float inv = lrun > 0.f ? 1.f / lrun : 0.f;
    const float lse = lrun > 0.f ? (mrun + log2f(lrun)) * 0.69314718055994531f : -INFINITY;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        uint32_t o[32];
        if (!kLse) {
            tc::ld32(tO + 32 * h, o);
            tc::ld_wait();
            tc::tie32(o);
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = 0u;
        }
        if (!valid) continue;
        if (ri.prow >= 0) {
            float *dst = p.part_o + size_t(ri.prow) * kHeadDim + 32 * h;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4 *>(dst + c) =
                    make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                                __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
        } else if (p.out == nullptr) {
            // lse only: no output rows
        } else if (p.out_dtype == FA_F32) {
            float *dst = reinterpret_cast<float *>(p.out) + size_t(ri.qrow) * kHeadDim + 32 * h;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4 *>(dst + c) =
                    make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                                __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
        } else {
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + size_t(ri.qrow) * kHeadDim + 32 * h;
#pragma unroll
            for (int c = 0; c < 32; c += 8)
                *reinterpret_cast<uint4 *>(dst + c) =
                    make_uint4(ptx::pack_bf16(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv),
                               ptx::pack_bf16(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv),
                               ptx::pack_bf16(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv),
                               ptx::pack_bf16(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv));
        }
    }
    if (valid) {
        if (ri.prow >= 0) p.part_lse[ri.prow] = lse;
        else p.lse[ri.qrow] = lse;
    }
}

__device__ __forceinline__ void init_barriers(Smem &sm) {
    for (int s = 0; s < kKStages; ++s) {
        ptx::mbar_init(ptx::smem_u32(&sm.kfull[s]), 1);
        ptx::mbar_init(ptx::smem_u32(&sm.kfree[s]), 1);  // one commit after the M tiles' Q K^T
    }
    for (int s = 0; s < kVStages; ++s) {
        ptx::mbar_init(ptx::smem_u32(&sm.vfull[s]), 1);
        ptx::mbar_init(ptx::smem_u32(&sm.vfree[s]), 1);
    }
    for (int m = 0; m < 2; ++m) {
        ptx::mbar_init(ptx::smem_u32(&sm.sfull[m]), 1);
        ptx::mbar_init(ptx::smem_u32(&sm.sfree[m]), 128);
        for (int h = 0; h < 2; ++h) {
            ptx::mbar_init(ptx::smem_u32(&sm.pfull[m][h]), 128);
            ptx::mbar_init(ptx::smem_u32(&sm.odone[m][h]), 1);
        }
    }
    ptx::mbar_init(ptx::smem_u32(&sm.fin), 2);  // one arrival per MMA warp
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
// kLse: only each row's lse (no V, no P V; partial O rows are zeros and out is not written).
template <bool kLse>
__global__ void __launch_bounds__(kThreads, 1) tc_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *queue = p.err + 1, *done = p.err + 2;
    ptx::launch_dependents();  // the next kernel of the decode may take the SMs this grid leaves

    auto item_ok = [&](int i) {  // items the planner never makes are refused, uniformly
        const Item it = p.items_tc[i];
        return it.n_pages <= kMaxChunkPages && it.n_rows <= kRows;
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

    if (tid == 0) {
        sm.abort = 0;
        sm.item = next_item();
        if (sm.item < p.n_items_tc) init_barriers(sm);
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
            Chunk ch = p.chunks[it.chunk];
            ch.n_pages = it.n_pages;  // the pages this item reads (a prefix of the chunk)
            const int T = (ch.n_pages + kTilePages - 1) / kTilePages;
            const int MT = it.n_rows > kTcRows ? 2 : 1;
            tc::fence_before();
            __syncthreads();  // B
            tc::fence_after();
            if (warp == 0) {
                producer<false>(p, sm, it, ch, T, lane);
            } else if (warp == 1) {
                mma_issuer(sm, tmem, T, MT, false, lane, kLse);
            } else if (warp == 3) {
                mma_issuer(sm, tmem, T, MT, true, lane, kLse);
            } else if (warp == 2) {
                if (!kLse) producer<true>(p, sm, it, ch, T, lane);
            }
            tc::fence_before();
            __syncthreads();  // C
            tc::fence_after();
            if (tid == 0) {
                inval_barriers(sm);
                sm.item = sm.abort ? p.n_items_tc : next_item();
                if (sm.item < p.n_items_tc) init_barriers(sm);
            }
            __syncthreads();  // D
        }
        if (tid == 0) {
            if (sm.abort) atomicOr(p.err, kErrTimeout | kErrTc);
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
        const int sm_m = (warp >> 2) - 1;  // softmax warpgroup = M tile (warps 4-7, 8-11)
        // TMEM lane quarter of a warp is warp % 4, so row = 128 m + 32 (warp % 4) + lane
        const int r = sm_m * kTcRows + (warp & 3) * 32 + lane;
        for (;;) {
            const int i = sm.item;
            if (i >= p.n_items_tc) break;
            const Item it = p.items_tc[i];
            Chunk ch = p.chunks[it.chunk];
            ch.n_pages = it.n_pages;  // the pages this item reads (a prefix of the chunk)
            const int T = (ch.n_pages + kTilePages - 1) / kTilePages;
            const int MT = it.n_rows > kTcRows ? 2 : 1;
            // the row's table entry, and its Q row -> shared memory, 128-byte swizzled K-major
            // (zeros for padding rows); the previous item's MMAs are all done (barrier C)
            Row ri{0, 0x3fffffff, -1, -1};
            const bool valid = r < it.n_rows;
            if (valid) ri = item_row(p, it, r);
#pragma unroll 4
            for (int c = 0; c < 16; ++c) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (valid) v = __ldg(reinterpret_cast<const uint4 *>(p.q + size_t(ri.qrow) * kHeadDim + c * 8));
                *reinterpret_cast<uint4 *>(sm.q + (c >> 3) * kQHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
            }
            tc::fence_proxy_async_smem();
            tc::fence_before();
            __syncthreads();  // B
            tc::fence_after();
            if (sm_m < MT) softmax<kLse>(p, sm, ch, ri, valid, tmem, T, sm_m, MT, warp & 3, lane);
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
