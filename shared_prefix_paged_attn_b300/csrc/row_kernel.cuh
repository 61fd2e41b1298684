// Row kernel: attention of up to 32 stacked query rows over one chunk of physical KV pages.
//
// Used for page runs with few readers (a branch's private pages, mounted sibling blocks,
// small forks).  Octopus (zicq.com), "Attention-Only KV Mounting": a mounted block is read in
// place like the owner's own KV.  AKV (news.farwalk.ai), "AKV 如何工作？": dropped entries
// are skipped through the visibility words and keep their positions.
//
// Design (sm_103a):
//   - one CTA = 4 warps per work item (chunk x KV head x row group); warp w owns pages
//     w, w+4, w+8, ... of the chunk and runs its own 3-stage ring: lane 0 issues two TMA
//     tensor loads per page (K and V, each a whole page-head of two 64-dim halves, 128-byte
//     swizzle) that complete on the slot's mbarrier; the rows' visibility words are loaded a
//     page ahead;
//   - the dot products run on the warp MMA (m16n8k16 bf16 -> fp32): S = Q K^T with the
//     stacked rows as M (one or two 16-row tiles), then O += P V with P taken from the S
//     accumulators without leaving registers;
//   - online softmax in base 2 with row max / sum reduced by quad shuffles; masked slots
//     (drop bits, segment edges, the causal cut of multi-token queries) are set to -inf;
//   - the four warps' (max, sum, O) are combined in shared memory in a fixed order (bitwise
//     run-to-run deterministic) and written as the final output (a branch with one chunk) or
//     as an fp32 partial (O normalised, natural-log LSE) for the merge kernel.
#pragma once
#include "decode_params.cuh"
#include "ptx.cuh"

namespace fa {
namespace rowk {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr int kPageBytes = kPageSize * kHeadDim * 2;  // 4 KiB: one page of one KV head
constexpr int kSlotBytes = 2 * kPageBytes;             // K then V
constexpr int kRingBytes = kWarps * kStages * kSlotBytes;
constexpr int kQHalfBytes = kRowsMax * 128;            // 64 dims x 32 rows
constexpr int kObufStride = 132;                       // floats per row of the combine buffer

struct RowInfo {
    int32_t qrow;      // row of q / out / lse = (query token) * Hq + head
    int32_t climit;    // chunk tokens t <= climit are causally visible
    int32_t mask_off;  // visibility words of the row's reader, -1 = all visible
    int32_t prow;      // partial row, or -1 for a direct write
};

struct Smem {
    alignas(1024) uint8_t ring[kRingBytes];
    alignas(1024) uint8_t qs[2 * kQHalfBytes];
    alignas(8) uint64_t bars[kWarps][kStages];
    RowInfo rows[kRowsMax];
    float wm[kWarps][kRowsMax];
    float wl[kWarps][kRowsMax];
    float rowM[kRowsMax];
    float rowL[kRowsMax];
};
static_assert(kWarps * kRowsMax * kObufStride * 4 <= kRingBytes, "combine buffer reuses the ring");
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack

__device__ __forceinline__ uint32_t swz(uint32_t box, int row, int chunk16) {
    // 128-byte swizzle of a box of 128-byte rows whose base is 1024-byte aligned
    return box + row * 128 + (((chunk16 & 7) ^ (row & 7)) << 4);
}

__device__ __forceinline__ void issue_page(const DecodeParams &p, uint32_t slot, uint32_t bar,
                                           int head, int page) {
    // one whole-page box each for K and V: [2 halves of 64 dims][16 tokens][128 bytes], the
    // same image as two 64-dim boxes 2 KiB apart
    ptx::mbar_arrive_expect_tx(bar, kSlotBytes);
    ptx::tma_load_5d(slot, &p.kmap_page, bar, 0, 0, 0, head, page);
    ptx::tma_load_5d(slot + kPageBytes, &p.vmap_page, bar, 0, 0, 0, head, page);
}

template <int MT>
__device__ __forceinline__ void run_pages(const DecodeParams &p, Smem &sm, const Item &it,
                                          const Chunk &ch, bool need_mask, float (&o)[2][16][4],
                                          float (&m)[2][2], float (&l)[2][2], bool &ok) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int n_pages = ch.n_pages;
    const int32_t *pages = p.chunk_pages + ch.page_off;
    const uint32_t ring = ptx::smem_u32(sm.ring) + warp * kStages * kSlotBytes;
    const uint32_t qs = ptx::smem_u32(sm.qs);

    // page ids of this warp's pages (k = warp + 4 i): lane l holds index i = 32 b + l of the
    // current batch b, and the next batch is already loaded, so issuing never waits on them
    auto pid_at = [&](int i) -> int32_t {
        const int k = warp + kWarps * i;
        return k < n_pages ? checked_page(p, __ldg(pages + k), kErrRow) : 0;
    };
    int32_t pid_cur = pid_at(lane), pid_nxt = pid_at(32 + lane);
    int issued = 0;
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
        const int k = warp + kWarps * s;
        const int32_t page = __shfl_sync(0xffffffffu, pid_cur, s);
        if (k < n_pages) {
            if (lane == 0) issue_page(p, ring + s * kSlotBytes, ptx::smem_u32(&sm.bars[warp][s]), it.head, page);
            ++issued;
        }
    }

    int32_t moff[2][2], clim[2][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const RowInfo &ri = sm.rows[mt * 16 + gid + 8 * hr];
            moff[mt][hr] = ri.mask_off;
            clim[mt][hr] = ri.climit;
        }

    // visibility words of this warp's next page for its rows (all ones: no word), loaded a page
    // ahead so that their latency hides behind the page before
    uint32_t wnx[2][2] = {{0xFFFFFFFFu, 0xFFFFFFFFu}, {0xFFFFFFFFu, 0xFFFFFFFFu}};
    auto fetch_words = [&](int kq) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
                if (moff[mt][hr] >= 0) wnx[mt][hr] = __ldg(p.mask_words + moff[mt][hr] + (kq >> 1));
    };
    if (need_mask && warp < n_pages) fetch_words(warp);

    int j = 0;
    for (;; ++j) {
        const int k = warp + kWarps * j;
        if (k >= n_pages) break;
        uint32_t wcur[2][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) wcur[mt][hr] = wnx[mt][hr];
        if (need_mask && k + kWarps < n_pages) fetch_words(k + kWarps);
        const int s = j % kStages;
        const uint32_t bar = ptx::smem_u32(&sm.bars[warp][s]);
        const bool landed = __all_sync(0xffffffffu, ptx::mbar_wait(bar, (j / kStages) & 1));
        if (!landed) {
            ok = false;
            break;
        }
        const uint32_t kb = ring + s * kSlotBytes;
        const uint32_t vb = kb + kPageBytes;

        // ---- S = Q K^T  (rows x 16 tokens) ----
        float sc[2][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[mt][nt][e] = 0.f;
        {
            const int mi = lane >> 3;
            const int ktok = (lane & 7) + ((mi >> 1) << 3);
            const int qrow_l = (lane & 7) + ((mi & 1) << 3);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int kcd = 2 * kk + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ptx::ldsm_x4(swz(kb + (kcd >> 3) * 2048, ktok, kcd), b0, b1, b2, b3);
                const int qcd = 2 * kk + (mi >> 1);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    ptx::ldsm_x4(swz(qs + (qcd >> 3) * kQHalfBytes, mt * 16 + qrow_l, qcd), a0, a1, a2, a3);
                    ptx::mma_bf16(sc[mt][0], a0, a1, a2, a3, b0, b1);
                    ptx::mma_bf16(sc[mt][1], a0, a1, a2, a3, b2, b3);
                }
            }
        }

        // ---- scale, mask, online softmax ----
        uint32_t pa[2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                uint32_t m16 = 0xFFFFu;
                if (need_mask) {
                    m16 = (wcur[mt][hr] >> ((k & 1) * 16)) & 0xFFFFu;
                    const int lim = clim[mt][hr] - 16 * k;
                    if (lim < 15) m16 &= (lim < 0) ? 0u : ((2u << lim) - 1u);
                }
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float v = sc[mt][nt][2 * hr + e] * p.scale_log2;
                        if (!((m16 >> (nt * 8 + tig * 2 + e)) & 1u)) v = -INFINITY;
                        sc[mt][nt][2 * hr + e] = v;
                        mx = fmaxf(mx, v);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                // lazy rescale: the running max only moves when the page's maximum exceeds it
                // by more than 2^8 (P <= 256 in bf16 then); the four lanes of a row agree
                const float m_old = m[mt][hr];
                float m_use = m_old;
                const bool rescale = m_old == -INFINITY || mx > m_old + 8.f;
                if (rescale) {
                    const float m_new = fmaxf(m_old, mx);
                    m_use = (m_new == -INFINITY) ? 0.f : m_new;
                    const float alpha = ptx::ex2(m_old - m_use);
                    m[mt][hr] = m_new;
                    l[mt][hr] *= alpha;
#pragma unroll
                    for (int dt = 0; dt < 16; ++dt) {
                        o[mt][dt][2 * hr] *= alpha;
                        o[mt][dt][2 * hr + 1] *= alpha;
                    }
                }
                float rs = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pv = ptx::ex2(sc[mt][nt][2 * hr + e] - m_use);
                        sc[mt][nt][2 * hr + e] = pv;
                        rs += pv;
                    }
                l[mt][hr] += rs;
            }
            pa[mt][0] = ptx::pack_bf16(sc[mt][0][0], sc[mt][0][1]);
            pa[mt][1] = ptx::pack_bf16(sc[mt][0][2], sc[mt][0][3]);
            pa[mt][2] = ptx::pack_bf16(sc[mt][1][0], sc[mt][1][1]);
            pa[mt][3] = ptx::pack_bf16(sc[mt][1][2], sc[mt][1][3]);
        }

        // ---- O += P V ----
        {
            const int mi = lane >> 3;
            const int vtok = (lane & 7) + ((mi & 1) << 3);
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                const int cd = 2 * np + (mi >> 1);
                uint32_t v0, v1, v2, v3;
                ptx::ldsm_x4_t(swz(vb + (cd >> 3) * 2048, vtok, cd), v0, v1, v2, v3);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    ptx::mma_bf16(o[mt][2 * np], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], v0, v1);
                    ptx::mma_bf16(o[mt][2 * np + 1], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], v2, v3);
                }
            }
        }

        __syncwarp();
        const int in_ = j + kStages;  // index of the next page in this warp's list
        if ((in_ & 31) == 0) {
            pid_cur = pid_nxt;
            pid_nxt = pid_at(in_ + 32 + lane);
        }
        const int32_t page = __shfl_sync(0xffffffffu, pid_cur, in_ & 31);
        const int kn = k + kWarps * kStages;
        if (kn < n_pages) {
            if (lane == 0) issue_page(p, kb, bar, it.head, page);
            ++issued;
        }
    }
    if (!ok) {
        // give the copies still in flight a bounded chance to land before the smem is reused
        for (int jj = j + 1; jj < issued; ++jj)
            ptx::mbar_wait(ptx::smem_u32(&sm.bars[warp][jj % kStages]), (jj / kStages) & 1);
        if (lane == 0) atomicOr(p.err, kErrTimeout | kErrRow);
    }
}

__global__ void __launch_bounds__(kThreads, 2) row_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const Item it = p.items[blockIdx.x];
    ptx::launch_dependents();  // the next kernel of the decode may take the SMs this grid leaves
    Chunk ch = p.chunks[it.chunk];
    ch.n_pages = it.n_pages;  // the pages this item reads (a prefix of the chunk)

    if (tid == 0) {
        for (int w = 0; w < kWarps; ++w)
            for (int s = 0; s < kStages; ++s) ptx::mbar_init(ptx::smem_u32(&sm.bars[w][s]), 1);
        ptx::fence_mbar_init();
    }
    // the item's row records: one 16-byte load per row
    bool row_needs_mask = false;
    if (tid < kRowsMax) {
        RowInfo ri{0, 0x3fffffff, -1, -1};
        if (tid < it.n_rows) {
            const int4 rec = __ldg(reinterpret_cast<const int4 *>(p.rows + it.row_off + tid));
            ri.qrow = rec.x + it.head * p.G;
            ri.climit = rec.y;
            ri.mask_off = rec.z;
            ri.prow = rec.w < 0 ? -1 : rec.w + it.head;
            checked_row(p, ri.qrow, ri.prow, ri.mask_off, ch.n_pages, kErrRow);
            row_needs_mask = ri.mask_off >= 0 || ri.climit < kPageSize * ch.n_pages - 1;
        }
        sm.rows[tid] = ri;
    }
    const bool need_mask = __syncthreads_or(row_needs_mask);

    // stacked Q rows -> shared memory (same 128-byte swizzle as the K/V boxes), padding = 0
    for (int idx = tid; idx < kRowsMax * 16; idx += kThreads) {
        const int r = idx >> 4, c = idx & 15;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < it.n_rows) v = *reinterpret_cast<const uint4 *>(p.q + size_t(sm.rows[r].qrow) * kHeadDim + c * 8);
        *reinterpret_cast<uint4 *>(sm.qs + (c >> 3) * kQHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
    }
    __syncthreads();

    float o[2][16][4];
    float m[2][2], l[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int dt = 0; dt < 16; ++dt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][dt][e] = 0.f;
        m[mt][0] = m[mt][1] = -INFINITY;
        l[mt][0] = l[mt][1] = 0.f;
    }
    bool ok = true;
    if (it.n_rows <= 16)
        run_pages<1>(p, sm, it, ch, need_mask, o, m, l, ok);
    else
        run_pages<2>(p, sm, it, ch, need_mask, o, m, l, ok);
    const int MTr = it.n_rows <= 16 ? 1 : 2;

    // ---- combine the four warps ----
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            l[mt][hr] += __shfl_xor_sync(0xffffffffu, l[mt][hr], 1);
            l[mt][hr] += __shfl_xor_sync(0xffffffffu, l[mt][hr], 2);
        }
    const bool failed = __syncthreads_or(!ok);  // also: every warp is done with its ring
    if (tig == 0) {
        for (int mt = 0; mt < MTr; ++mt)
            for (int hr = 0; hr < 2; ++hr) {
                const int r = mt * 16 + gid + 8 * hr;
                sm.wm[warp][r] = m[mt][hr];
                sm.wl[warp][r] = l[mt][hr];
            }
    }
    __syncthreads();
    float *obuf = reinterpret_cast<float *>(sm.ring) + warp * kRowsMax * kObufStride;
    for (int mt = 0; mt < MTr; ++mt)
        for (int hr = 0; hr < 2; ++hr) {
            const int r = mt * 16 + gid + 8 * hr;
            float M = -INFINITY;
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.wm[w][r]);
            const float Mu = (M == -INFINITY) ? 0.f : M;
            float L = 0.f;
            for (int w = 0; w < kWarps; ++w) L += ptx::ex2(sm.wm[w][r] - Mu) * sm.wl[w][r];
            const float f = ptx::ex2(m[mt][hr] - Mu);
#pragma unroll
            for (int dt = 0; dt < 16; ++dt) {
                float2 v = make_float2(o[mt][dt][2 * hr] * f, o[mt][dt][2 * hr + 1] * f);
                *reinterpret_cast<float2 *>(obuf + r * kObufStride + dt * 8 + tig * 2) = v;
            }
            if (warp == 0 && tig == 0) {
                sm.rowM[r] = M;
                sm.rowL[r] = L;
            }
        }
    __syncthreads();
    if (failed) return;

    const float *ob = reinterpret_cast<const float *>(sm.ring);
    for (int idx = tid; idx < it.n_rows * 32; idx += kThreads) {
        const int r = idx >> 5, c4 = idx & 31;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float4 v = *reinterpret_cast<const float4 *>(ob + (w * kRowsMax + r) * kObufStride + c4 * 4);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        const float L = sm.rowL[r];
        const float inv = L > 0.f ? 1.f / L : 0.f;
        acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
        const RowInfo ri = sm.rows[r];
        if (ri.prow >= 0) {
            *reinterpret_cast<float4 *>(p.part_o + size_t(ri.prow) * kHeadDim + c4 * 4) = acc;
        } else if (p.out_dtype == FA_F32) {
            *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + size_t(ri.qrow) * kHeadDim + c4 * 4) = acc;
        } else {
            uint2 pk = make_uint2(ptx::pack_bf16(acc.x, acc.y), ptx::pack_bf16(acc.z, acc.w));
            *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + size_t(ri.qrow) * kHeadDim + c4 * 4) = pk;
        }
    }
    if (tid < it.n_rows) {
        const float L = sm.rowL[tid];
        const float lse = L > 0.f ? (sm.rowM[tid] + log2f(L)) * 0.69314718055994531f : -INFINITY;
        const RowInfo ri = sm.rows[tid];
        if (ri.prow >= 0) p.part_lse[ri.prow] = lse;
        else p.lse[ri.qrow] = lse;
    }
}

}  // namespace rowk
}  // namespace fa
