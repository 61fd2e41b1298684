// Row kernel for at most 8 stacked query rows (the private and mounted runs of one branch
// with a GQA group of 4 or 8 and one query token): attention over one chunk of pages.
//
// Octopus (zicq.com), "Attention-Only KV Mounting": a mounted block is read in place like
// the owner's own KV.  AKV (news.farwalk.ai), "AKV 如何工作？": dropped entries are skipped
// through the visibility words and keep their positions.
//
// With so few rows the usual orientation (rows as the MMA's M) wastes half of every m16n8k16,
// so the kernel works transposed:
//   S^T = K Q^T     M = the page's 16 tokens, N = the 8 rows, K = 128 dims in 8 steps; Q is a
//                   register-resident B fragment;
//   O^T += V^T P^T  M = 16 dims (8 tiles of the 128), N = the 8 rows, K = the page's 16
//                   tokens; P^T is the S^T accumulator turned into a B fragment with two
//                   movmatrix transposes.
// Each thread holds 4 scores per page (2 tokens x 2 rows).  Online softmax in base 2 with a
// lazy rescale: the running max only moves when a score exceeds it by more than 2^8, which
// each lane checks on its own scores; only then is the page max of each row reduced over the
// 8 lanes sharing its column.  Four warps per CTA, each over pages w, w+4, ...
// with its own 2-stage TMA ring, three CTAs per SM (a warp's page time is mostly its own
// instruction latency, so more warps per SM stream more than deeper rings); the warps'
// (max, sum, O) are combined in shared memory in a fixed order (bitwise run-to-run
// deterministic).
#pragma once
#include "decode_params.cuh"
#include "ptx.cuh"

namespace fa {
namespace r8k {

constexpr int kRows = 8;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;  // with 3 CTAs per SM: 12 warps streaming pages per SM
constexpr int kPageBytes = kPageSize * kHeadDim * 2;  // 4 KiB: one page of one KV head
constexpr int kSlotBytes = 2 * kPageBytes;             // K then V
constexpr int kRingBytes = kWarps * kStages * kSlotBytes;
constexpr int kObufStride = 132;                       // floats per row of the combine buffer

struct RowInfo {
    int32_t qrow, climit, mask_off, prow;
};

struct Smem {
    alignas(1024) uint8_t ring[kRingBytes];
    alignas(8) uint64_t bars[kWarps][kStages];
    RowInfo rows[kRows];
    float wm[kWarps][kRows];
    float wl[kWarps][kRows];
    float rowM[kRows];
    float rowL[kRows];
};
static_assert(kWarps * kRows * kObufStride * 4 <= kRingBytes, "combine buffer reuses the ring");
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack

__device__ __forceinline__ uint32_t swz(uint32_t box, int row, int chunk16) {
    // 128-byte swizzle of a box of 128-byte rows whose base is 1024-byte aligned
    return box + row * 128 + (((chunk16 & 7) ^ (row & 7)) << 4);
}

__device__ __forceinline__ void issue_page(const DecodeParams &p, uint32_t slot, uint32_t bar, int head, int page) {
    // one whole-page box each for K and V: [2 halves of 64 dims][16 tokens][128 bytes], the
    // same image as two 64-dim boxes 2 KiB apart
    ptx::mbar_arrive_expect_tx(bar, kSlotBytes);
    ptx::tma_load_5d(slot, &p.kmap_page, bar, 0, 0, 0, head, page);
    ptx::tma_load_5d(slot + kPageBytes, &p.vmap_page, bar, 0, 0, 0, head, page);
}

__global__ void __launch_bounds__(kThreads, 3) row8_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const Item it = p.items_r8[blockIdx.x];
    ptx::launch_dependents();  // the next kernel of the decode may take the SMs this grid leaves
    Chunk ch = p.chunks[it.chunk];
    ch.n_pages = it.n_pages;  // the pages this item reads (a prefix of the chunk)
    const int n_pages = ch.n_pages;
    const int32_t *pages = p.chunk_pages + ch.page_off;

    if (tid == 0) {
        for (int w = 0; w < kWarps; ++w)
            for (int s = 0; s < kStages; ++s) ptx::mbar_init(ptx::smem_u32(&sm.bars[w][s]), 1);
        ptx::fence_mbar_init();
    }
    bool row_needs_mask = false;
    if (tid < kRows) {
        RowInfo ri{0, 0x3fffffff, -1, -1};
        if (tid < it.n_rows) {
            const int4 rec = __ldg(reinterpret_cast<const int4 *>(p.rows + it.row_off + tid));
            ri = RowInfo{rec.x + it.head * p.G, rec.y, rec.z, rec.w < 0 ? -1 : rec.w + it.head};
            checked_row(p, ri.qrow, ri.prow, ri.mask_off, n_pages, kErrRow8);
            row_needs_mask = ri.mask_off >= 0 || ri.climit < kPageSize * n_pages - 1;
        }
        sm.rows[tid] = ri;
    }
    const bool need_mask = __syncthreads_or(row_needs_mask);

    // Q^T as B fragments: step kk holds row gid's dims 16 kk + 2 tig (+1) and + 8 (zero for
    // padding rows)
    uint32_t qb[8][2];
    {
        const bool qv = gid < it.n_rows;
        const __nv_bfloat16 *qr = p.q + size_t(sm.rows[gid].qrow) * kHeadDim;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            qb[kk][0] = qv ? __ldg(reinterpret_cast<const uint32_t *>(qr + 16 * kk + 2 * tig)) : 0u;
            qb[kk][1] = qv ? __ldg(reinterpret_cast<const uint32_t *>(qr + 16 * kk + 8 + 2 * tig)) : 0u;
        }
    }
    // this thread's two rows (the MMA's N columns 2 tig, 2 tig + 1)
    const RowInfo ra = sm.rows[2 * tig], rb = sm.rows[2 * tig + 1];

    const uint32_t ring = ptx::smem_u32(sm.ring) + warp * kStages * kSlotBytes;
    // page ids of this warp's pages (k = warp + 4 i): lane l holds index i = 32 b + l of the
    // current batch b, and the next batch is already loaded, so issuing never waits on them
    auto pid_at = [&](int i) -> int32_t {
        const int k = warp + kWarps * i;
        return k < n_pages ? checked_page(p, __ldg(pages + k), kErrRow8) : 0;
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

    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;  // la, lb: this lane's tokens only
    const float sl2 = p.scale_log2;
    bool ok = true;
    const int mi = lane >> 3, r8 = lane & 7;

    // visibility words of this warp's next page for rows ra, rb (all ones: no word), loaded a
    // page ahead so that their latency hides behind the page before
    uint32_t wa_nx = 0xFFFFFFFFu, wb_nx = 0xFFFFFFFFu;
    auto fetch_words = [&](int kq) {
        if (ra.mask_off >= 0) wa_nx = __ldg(p.mask_words + ra.mask_off + (kq >> 1));
        if (rb.mask_off >= 0) wb_nx = __ldg(p.mask_words + rb.mask_off + (kq >> 1));
    };
    if (need_mask && warp < n_pages) fetch_words(warp);

    int j = 0;
    for (;; ++j) {
        const int k = warp + kWarps * j;
        if (k >= n_pages) break;
        const uint32_t words_a = wa_nx, words_b = wb_nx;
        if (need_mask && k + kWarps < n_pages) fetch_words(k + kWarps);
        const int s = j % kStages;
        const uint32_t bar = ptx::smem_u32(&sm.bars[warp][s]);
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar, (j / kStages) & 1))) {
            ok = false;
            break;
        }
        const uint32_t kb = ring + s * kSlotBytes;
        const uint32_t vb = kb + kPageBytes;

        // ---- S^T = K Q^T: 16 tokens x 8 rows, even and odd K steps in two independent
        // accumulator chains (half the dependent MMA latency) ----
        float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; kk += 2) {
            // block mi: tokens r8 + 8 (mi & 1), dims 16 kk + 8 (mi >> 1) .. + 7
            uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
            ptx::ldsm_x4(swz(kb + (kk >> 2) * 2048, r8 + 8 * (mi & 1), 2 * kk + (mi >> 1)), a0, a1, a2, a3);
            ptx::ldsm_x4(swz(kb + (kk >> 2) * 2048, r8 + 8 * (mi & 1), 2 * kk + 2 + (mi >> 1)), c0, c1, c2, c3);
            ptx::mma_bf16(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
            ptx::mma_bf16(sd, c0, c1, c2, c3, qb[kk + 1][0], qb[kk + 1][1]);
        }
        // sc: (token gid, row 2 tig), (token gid, row 2 tig + 1), (token gid + 8, ...) x 2
        float x0 = (sc[0] + sd[0]) * sl2, x1 = (sc[1] + sd[1]) * sl2, x2 = (sc[2] + sd[2]) * sl2,
              x3 = (sc[3] + sd[3]) * sl2;
        if (need_mask) {
            uint32_t ka = (words_a >> ((k & 1) * 16)) & 0xFFFFu, kb16 = (words_b >> ((k & 1) * 16)) & 0xFFFFu;
            const int lima = ra.climit - 16 * k, limb = rb.climit - 16 * k;
            if (lima < 15) ka &= lima < 0 ? 0u : ((2u << lima) - 1u);
            if (limb < 15) kb16 &= limb < 0 ? 0u : ((2u << limb) - 1u);
            if (!((ka >> gid) & 1u)) x0 = -INFINITY;
            if (!((kb16 >> gid) & 1u)) x1 = -INFINITY;
            if (!((ka >> (gid + 8)) & 1u)) x2 = -INFINITY;
            if (!((kb16 >> (gid + 8)) & 1u)) x3 = -INFINITY;
        }
        // The running max only moves when some score of a row exceeds it by more than 2^8
        // (with ma = -inf any visible score does): each lane checks its own four scores, and
        // only then are the page maxima reduced over the 8 lanes of each row.
        const bool grow = x0 > ma + 8.0f || x2 > ma + 8.0f || x1 > mb + 8.0f || x3 > mb + 8.0f;
        if (__any_sync(0xffffffffu, grow)) {
            float pa = fmaxf(x0, x2), pb = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                pa = fmaxf(pa, __shfl_xor_sync(0xffffffffu, pa, off));
                pb = fmaxf(pb, __shfl_xor_sync(0xffffffffu, pb, off));
            }
            // raise the running max of the rows; O^T columns and sums follow
            const float na = fmaxf(ma, pa), nb = fmaxf(mb, pb);
            const float aa = (ma == -INFINITY || na == -INFINITY) ? 1.f : ptx::ex2(ma - na);
            const float ab = (mb == -INFINITY || nb == -INFINITY) ? 1.f : ptx::ex2(mb - nb);
            ma = na;
            mb = nb;
            la *= aa;
            lb *= ab;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                o[mt][0] *= aa;
                o[mt][1] *= ab;
                o[mt][2] *= aa;
                o[mt][3] *= ab;
            }
        }
        const float ua = ma == -INFINITY ? 0.f : ma, ub = mb == -INFINITY ? 0.f : mb;
        const float p0 = ptx::ex2(x0 - ua), p1 = ptx::ex2(x1 - ub), p2 = ptx::ex2(x2 - ua), p3 = ptx::ex2(x3 - ub);
        la += p0 + p2;
        lb += p1 + p3;
        // P^T as the B fragment: transpose the [token][row] 8x8 blocks to [row][token]
        const uint32_t b0 = ptx::movmatrix_t(ptx::pack_bf16(p0, p1));
        const uint32_t b1 = ptx::movmatrix_t(ptx::pack_bf16(p2, p3));

        // ---- O^T += V^T P^T: 8 tiles of 16 dims ----
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            // block mi: tokens r8 + 8 (mi >> 1), dims 16 mt + 8 (mi & 1) .. + 7, transposed
            uint32_t a0, a1, a2, a3;
            ptx::ldsm_x4_t(swz(vb + (mt >> 2) * 2048, r8 + 8 * (mi >> 1), 2 * mt + (mi & 1)), a0, a1, a2, a3);
            ptx::mma_bf16(o[mt], a0, a1, a2, a3, b0, b1);
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
        if (lane == 0) atomicOr(p.err, kErrTimeout | kErrRow8);
    }

    // ---- combine the four warps ----
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, off);
        lb += __shfl_xor_sync(0xffffffffu, lb, off);
    }
    const bool failed = __syncthreads_or(!ok);  // also: every warp is done with its ring
    if (gid == 0) {
        sm.wm[warp][2 * tig] = ma;
        sm.wm[warp][2 * tig + 1] = mb;
        sm.wl[warp][2 * tig] = la;
        sm.wl[warp][2 * tig + 1] = lb;
    }
    __syncthreads();
    float *obuf = reinterpret_cast<float *>(sm.ring) + warp * kRows * kObufStride;
    {
        float M[2], L[2], f[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = 2 * tig + h;
            M[h] = -INFINITY;
            for (int w = 0; w < kWarps; ++w) M[h] = fmaxf(M[h], sm.wm[w][r]);
            const float Mu = (M[h] == -INFINITY) ? 0.f : M[h];
            L[h] = 0.f;
            for (int w = 0; w < kWarps; ++w) L[h] += ptx::ex2(sm.wm[w][r] - Mu) * sm.wl[w][r];
            f[h] = ptx::ex2((h ? mb : ma) - Mu);
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            obuf[(2 * tig) * kObufStride + 16 * mt + gid] = o[mt][0] * f[0];
            obuf[(2 * tig + 1) * kObufStride + 16 * mt + gid] = o[mt][1] * f[1];
            obuf[(2 * tig) * kObufStride + 16 * mt + gid + 8] = o[mt][2] * f[0];
            obuf[(2 * tig + 1) * kObufStride + 16 * mt + gid + 8] = o[mt][3] * f[1];
        }
        if (warp == 0 && gid == 0) {
            sm.rowM[2 * tig] = M[0];
            sm.rowM[2 * tig + 1] = M[1];
            sm.rowL[2 * tig] = L[0];
            sm.rowL[2 * tig + 1] = L[1];
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
            const float4 v = *reinterpret_cast<const float4 *>(ob + (w * kRows + r) * kObufStride + c4 * 4);
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

}  // namespace r8k
}  // namespace fa
