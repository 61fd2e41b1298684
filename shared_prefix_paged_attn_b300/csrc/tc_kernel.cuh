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
// One CTA = 12 warps per work item (chunk x KV head x row group of <= 256 rows):
//   warp 0 (one thread)  TMA producer: per 128-token tile, the 8 pages of K (and of V) as
//                        2 KiB boxes (64 dims x 16 tokens, 128-byte swizzle) into a 3-stage
//                        K ring and a 2-stage V ring; pages past the chunk's end are read at
//                        an out-of-range page index, which the copy fills with zeros;
//   warp 1 (one thread)  MMA issuer; the whole warp allocates the 512 TMEM columns:
//                        O0 [0,128) O1 [128,256) S0/P0 [256,384) S1/P1 [384,512);
//   warps 4-7, 8-11      softmax of M tile 0 and 1 (one row per thread, TMEM lane = row):
//                        S from TMEM, mask (visibility words, chunk end, causal limit), base-2
//                        online softmax with a lazy rescale (the running max is only raised
//                        when a row's maximum grows by more than 2^8, which keeps P <= 256),
//                        P as bf16 written back over S in TMEM for the P V MMA.
// While one softmax warpgroup works on its tile, the tensor core runs the other one's MMAs.
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
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kRows = 2 * kTcRows;                  // 256 rows per work item
constexpr int kQHalf = kRows * 128;                 // 64 dims of 256 rows: 32 KiB
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256;

struct Smem {
    alignas(1024) uint8_t q[2 * kQHalf];
    alignas(1024) uint8_t k[kKStages][kTileBytes];
    alignas(1024) uint8_t v[kVStages][kTileBytes];
    alignas(8) uint64_t kfull[kKStages], kfree[kKStages], vfull[kVStages], vfree[kVStages];
    uint64_t sfull[2], pfull[2], odone[2], fin;
    uint32_t tmem_base;
    int32_t abort;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "fits the 227 KiB opt-in shared memory of one CTA");

constexpr uint32_t kIdescQK = tc::idesc_bf16(128, 128, false, false);  // Q, K both K-major
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, 128, false, true);   // P (TMEM), V MN-major

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
    atomicOr(err, kErrTimeout);
}

struct Row {
    int32_t qrow, climit, mask_off, prow;
};

// Row r of a work item -> (query row, causal limit in chunk tokens, visibility words, partial row).
__device__ __forceinline__ Row item_row(const DecodeParams &p, const Item &it, int r) {
    int e = it.ent_off, acc = 0;
    Ent en = p.ents[e];
    while (r >= acc + en.ni * p.G) {
        acc += en.ni * p.G;
        en = p.ents[++e];
    }
    const int i = en.i0 + (r - acc) / p.G;
    const int jh = (r - acc) % p.G;
    const Occ oc = p.occs[en.occ];
    const Branch br = p.branches[oc.branch];
    Row x;
    x.qrow = (br.q_begin + i) * p.Hq + it.head * p.G + jh;
    x.climit = br.qpos0 + i - oc.lpos0;
    x.mask_off = oc.mask_off;
    x.prow = oc.prow_base < 0 ? -1 : oc.prow_base + it.head * (br.n_q * p.G) + i * p.G + jh;
    return x;
}

__device__ __forceinline__ void load_tile(const DecodeParams &p, const CUtensorMap *map, uint32_t dst,
                                          uint32_t bar, const int32_t *pages, int n_pages, int j, int head) {
    ptx::mbar_arrive_expect_tx(bar, kTileBytes);
#pragma unroll 1
    for (int pg = 0; pg < kTilePages; ++pg) {
        const int idx = j * kTilePages + pg;
        const int page = idx < n_pages ? pages[idx] : p.pool_pages;  // out of range: zero fill
        ptx::tma_load_4d(dst + pg * 2048, map, bar, 0, 0, head, page);
        ptx::tma_load_4d(dst + kHalfBytes + pg * 2048, map, bar, 64, 0, head, page);
    }
}

__device__ void producer(const DecodeParams &p, Smem &sm, const Item &it, const Chunk &ch, int T) {
    const int32_t *pages = p.chunk_pages + ch.page_off;
    const volatile int32_t *abort = &sm.abort;
    int k_issued = 0, v_issued = 0;
    // K runs one tile ahead of V: K0, K1, V0, K2, V1, ...
    load_tile(p, &p.kmap, ptx::smem_u32(sm.k[0]), ptx::smem_u32(&sm.kfull[0]), pages, ch.n_pages, 0, it.head);
    k_issued = 1;
    for (int j = 0; j < T; ++j) {
        const int jk = j + 1;
        if (jk < T) {
            const int s = jk % kKStages;
            if (jk >= kKStages && !wait_bar(ptx::smem_u32(&sm.kfree[s]), (jk / kKStages - 1) & 1, abort)) break;
            load_tile(p, &p.kmap, ptx::smem_u32(sm.k[s]), ptx::smem_u32(&sm.kfull[s]), pages, ch.n_pages, jk,
                      it.head);
            ++k_issued;
        }
        const int s = j % kVStages;
        if (j >= kVStages && !wait_bar(ptx::smem_u32(&sm.vfree[s]), (j / kVStages - 1) & 1, abort)) break;
        load_tile(p, &p.vmap, ptx::smem_u32(sm.v[s]), ptx::smem_u32(&sm.vfull[s]), pages, ch.n_pages, j, it.head);
        ++v_issued;
    }
    if (k_issued < T || v_issued < T) fail(sm, p.err);
    // every copy this CTA started must land before its shared memory goes away
    const volatile int32_t never = 0;
    for (int j = (k_issued > kKStages ? k_issued - kKStages : 0); j < k_issued; ++j)
        wait_bar(ptx::smem_u32(&sm.kfull[j % kKStages]), (j / kKStages) & 1, &never);
    for (int j = (v_issued > kVStages ? v_issued - kVStages : 0); j < v_issued; ++j)
        wait_bar(ptx::smem_u32(&sm.vfull[j % kVStages]), (j / kVStages) & 1, &never);
}

__device__ void mma_issuer(Smem &sm, uint32_t tmem, int T, int MT) {
    const volatile int32_t *abort = &sm.abort;
    const uint32_t qa = ptx::smem_u32(sm.q);
    bool ok = true;
    auto pv = [&](int m, int j) {  // O_m (+)= P_m V_j
        const uint32_t vb = ptx::smem_u32(sm.v[j % kVStages]);
#pragma unroll
        for (int kk = 0; kk < kTilePages; ++kk)
            tc::mma_ts(tmem + kColO + 128 * m, tmem + kColS + 128 * m + 8 * kk,
                       tc::sdesc_sw128(vb + kk * 2048, kHalfBytes, 1024), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        tc::commit(ptx::smem_u32(&sm.odone[m]));
    };
    for (int j = 0; j < T && ok; ++j) {
        for (int m = 0; m < MT && ok; ++m) {
            if (j > 0) {
                if (m == 0 && !wait_bar(ptx::smem_u32(&sm.vfull[(j - 1) % kVStages]), ((j - 1) / kVStages) & 1, abort)) {
                    ok = false;
                    break;
                }
                if (!wait_bar(ptx::smem_u32(&sm.pfull[m]), (j - 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                pv(m, j - 1);
            }
            if (m == 0) {
                if (!wait_bar(ptx::smem_u32(&sm.kfull[j % kKStages]), (j / kKStages) & 1, abort)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
            }
            const uint32_t kb = ptx::smem_u32(sm.k[j % kKStages]);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                tc::mma_ss(tmem + kColS + 128 * m, tc::sdesc_sw128(qa + (kk >> 2) * kQHalf + m * (kQHalf / 2) + (kk & 3) * 32, 16, 1024),
                           tc::sdesc_sw128(kb + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
            }
            tc::commit(ptx::smem_u32(&sm.sfull[m]));
        }
        if (!ok) break;
        tc::commit(ptx::smem_u32(&sm.kfree[j % kKStages]));
        if (j > 0) tc::commit(ptx::smem_u32(&sm.vfree[(j - 1) % kVStages]));
    }
    if (ok) {
        if (wait_bar(ptx::smem_u32(&sm.vfull[(T - 1) % kVStages]), ((T - 1) / kVStages) & 1, abort)) {
            for (int m = 0; m < MT && ok; ++m) {
                if (!wait_bar(ptx::smem_u32(&sm.pfull[m]), (T - 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                pv(m, T - 1);
            }
        } else {
            ok = false;
        }
    }
    if (!ok) *reinterpret_cast<volatile int32_t *>(&sm.abort) = 1;
    // all MMAs issued by this thread are complete before TMEM is freed
    tc::commit(ptx::smem_u32(&sm.fin));
    const volatile int32_t never = 0;
    wait_bar(ptx::smem_u32(&sm.fin), 0, &never);
}

__device__ void softmax(const DecodeParams &p, Smem &sm, const Chunk &ch, const Row &ri, bool valid, uint32_t tmem,
                        int T, int m, int wq, int lane) {
    const volatile int32_t *abort = &sm.abort;
    const uint32_t lane_base = uint32_t(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS + 128 * m;
    const uint32_t tO = tmem + lane_base + kColO + 128 * m;
    const int n_tok = ch.n_pages * kPageSize;
    const int n_words = (ch.n_pages + 1) >> 1;
    const float sl2 = p.scale_log2;
    float mrun = -INFINITY, lrun = 0.f;
    bool ok = true;

    for (int j = 0; j < T; ++j) {
        ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.sfull[m]), j & 1, abort));
        if (!ok) break;
        tc::fence_after();

        // visibility of the tile's 128 tokens for this row: words of the reader, chunk end,
        // causal limit (all ones when nothing is masked)
        const int t0 = j * kTileTok;
        uint32_t bits[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
        const bool masked = valid && (ri.mask_off >= 0 || t0 + kTileTok > n_tok || ri.climit < t0 + kTileTok - 1);
        if (masked) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int tq = t0 + 32 * w;
                uint32_t b = 0xffffffffu;
                if (ri.mask_off >= 0) {
                    const int wi = tq >> 5;
                    b = wi < n_words ? __ldg(p.mask_words + ri.mask_off + wi) : 0u;
                }
                const int lt = n_tok - tq;
                if (lt < 32) b &= lt <= 0 ? 0u : ((1u << lt) - 1u);
                const int lc = ri.climit - tq + 1;
                if (lc < 32) b &= lc <= 0 ? 0u : ((1u << lc) - 1u);
                bits[w] = b;
            }
        }
        const bool any_masked = __any_sync(0xffffffffu, masked);

        // pass 1: row max over the visible scores (32 columns at a time, next load in flight)
        float mx = -INFINITY;
        {
            uint32_t a[32], b[32];
            tc::ld32(tS, a);
            tc::ld_wait();
            tc::tie32(a);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                if (h < 3) tc::ld32(tS + 32 * (h + 1), b);
                if (any_masked) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (!((bits[h] >> c) & 1u)) a[c] = __float_as_uint(-INFINITY);
                }
#pragma unroll
                for (int c = 0; c < 32; ++c) mx = fmaxf(mx, __uint_as_float(a[c]));
                if (h < 3) {
                    tc::ld_wait();
                    tc::tie32(b);
#pragma unroll
                    for (int c = 0; c < 32; ++c) a[c] = b[c];
                }
            }
        }
        if (!valid) mx = -INFINITY;
        const float mnew = fmaxf(mrun, mx * sl2);
        const bool want = mrun != -INFINITY && mnew > mrun + 8.0f;
        if (__any_sync(0xffffffffu, want)) {
            // raise the running max of this warp's rows; O of the previous tiles is rescaled
            float alpha = 1.f;
            if (mrun != -INFINITY && mnew > mrun) alpha = ptx::ex2(mrun - mnew);
            if (mnew > mrun) mrun = mnew;
            lrun *= alpha;
            ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.odone[m]), (j - 1) & 1, abort));
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
        } else if (mrun == -INFINITY) {
            mrun = mnew;
        }
        const float muse = mrun == -INFINITY ? 0.f : mrun;

        // pass 2: P = 2^(s * scale * log2 e - m) as bf16 pairs over S's first 64 columns
        float rs = 0.f;
        {
            uint32_t a[32], b[32];
            tc::ld32(tS, a);
            tc::ld_wait();
            tc::tie32(a);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                if (h < 3) tc::ld32(tS + 32 * (h + 1), b);
                if (any_masked) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (!((bits[h] >> c) & 1u)) a[c] = __float_as_uint(-INFINITY);
                }
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    float x = 0.f, y = 0.f;
                    if (valid) {
                        x = ptx::ex2(fmaf(__uint_as_float(a[2 * c]), sl2, -muse));
                        y = ptx::ex2(fmaf(__uint_as_float(a[2 * c + 1]), sl2, -muse));
                    }
                    rs += x + y;
                    pk[c] = ptx::pack_bf16(x, y);
                }
                // columns 16h .. 16h+15 held scores 16h .. 16h+15, already read
                tc::st16(tS + 16 * h, pk);
                if (h < 3) {
                    tc::ld_wait();
                    tc::tie32(b);
#pragma unroll
                    for (int c = 0; c < 32; ++c) a[c] = b[c];
                }
            }
        }
        lrun += rs;
        tc::st_wait();
        tc::fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&sm.pfull[m]));
    }
    if (!ok) {
        if (lane == 0) fail(sm, p.err);
        return;
    }

    // ---- epilogue: O / l, natural-log LSE ----
    ok = __all_sync(0xffffffffu, wait_bar(ptx::smem_u32(&sm.odone[m]), (T - 1) & 1, abort));
    if (!ok) {
        if (lane == 0) fail(sm, p.err);
        return;
    }
    tc::fence_after();
    const float inv = lrun > 0.f ? 1.f / lrun : 0.f;
    const float lse = lrun > 0.f ? (mrun + log2f(lrun)) * 0.69314718055994531f : -INFINITY;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        uint32_t o[32];
        tc::ld32(tO + 32 * h, o);
        tc::ld_wait();
        tc::tie32(o);
        if (!valid) continue;
        if (ri.prow >= 0) {
            float *dst = p.part_o + size_t(ri.prow) * kHeadDim + 32 * h;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4 *>(dst + c) =
                    make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                                __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
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

__global__ void __launch_bounds__(kThreads, 1) tc_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Item it = p.items_tc[blockIdx.x];
    const Chunk ch = p.chunks[it.chunk];
    const int T = (ch.n_pages + kTilePages - 1) / kTilePages;
    const int MT = it.n_rows > kTcRows ? 2 : 1;

    if (tid == 0) {
        for (int s = 0; s < kKStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&sm.kfull[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&sm.kfree[s]), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&sm.vfull[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&sm.vfree[s]), 1);
        }
        for (int m = 0; m < 2; ++m) {
            ptx::mbar_init(ptx::smem_u32(&sm.sfull[m]), 1);
            ptx::mbar_init(ptx::smem_u32(&sm.pfull[m]), 128);
            ptx::mbar_init(ptx::smem_u32(&sm.odone[m]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&sm.fin), 1);
        sm.abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(ptx::smem_u32(&sm.tmem_base), kTmemCols);
        tc::tmem_relinquish();
    }
    // softmax threads: their row's table entry, and the stacked Q row -> shared memory,
    // 128-byte swizzled K-major (zeros for padding rows)
    Row ri{0, 0x3fffffff, -1, -1};
    bool valid = false;
    if (warp >= 4) {
        const int r = tid - 128;
        valid = r < it.n_rows;
        if (valid) ri = item_row(p, it, r);
#pragma unroll 4
        for (int c = 0; c < 16; ++c) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (valid) v = __ldg(reinterpret_cast<const uint4 *>(p.q + size_t(ri.qrow) * kHeadDim + c * 8));
            *reinterpret_cast<uint4 *>(sm.q + (c >> 3) * kQHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
        }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        if (lane == 0) producer(p, sm, it, ch, T);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer(sm, tmem, T, MT);
        __syncwarp();
    } else if (warp >= 4) {
        const int m = (warp - 4) >> 2;
        if (m < MT) softmax(p, sm, ch, ri, valid, tmem, T, m, warp & 3, lane);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && sm.abort) atomicOr(p.err, kErrTimeout);
}

}  // namespace tck
}  // namespace fa
