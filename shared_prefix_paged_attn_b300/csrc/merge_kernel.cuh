// Log-sum-exp merge of partial results.
//
// Agentrix (gitlink.org.cn), section "初赛基础与决赛演进", CUDA ForkAttention: after the
// common part is computed once for all branches and the private parts per branch, each
// branch's results are merged.  For a (query token, query head) row with partials
// (O_k, lse_k) over disjoint sets of entries:
//     L = max_k lse_k + ln sum_k exp(lse_k - max_k lse_k),    O = sum_k exp(lse_k - L) O_k.
// One warp per row; each lane owns 4 of the 128 dims.  The token's merge record (64 bytes)
// holds the bases of up to five partials, so a row with that many loads the record, then
// every partial's lse and O slice at once: two dependent loads in all.  Longer lists take
// their bases from the branch's list, the lse values spread over the lanes (max and weights
// by shuffles), kF O loads in flight at a time: 4, or 8 for a plan of few merged rows whose
// partials sit mostly in such rows (fewer resident warps, which such a plan does not fill
// anyway, and a row's loads in half the rounds).  The O terms are summed in the plan's fixed order either way, so the result is
// bitwise run-to-run deterministic and the same for both kF.
#pragma once
#include "decode_params.cuh"
#include "ptx.cuh"

namespace fa {
namespace mergek {

constexpr int kThreads = 256;

__device__ __forceinline__ void store_row(const DecodeParams &p, int row, int lane, float4 acc, float lse) {
    if (p.out == nullptr) {
        // lse only
    } else if (p.out_dtype == FA_F32) {
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + size_t(row) * kHeadDim + lane * 4) = acc;
    } else {
        uint2 pk = make_uint2(ptx::pack_bf16(acc.x, acc.y), ptx::pack_bf16(acc.z, acc.w));
        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + size_t(row) * kHeadDim + lane * 4) = pk;
    }
    if (lane == 0) p.lse[row] = lse;
}

template <int kF>
__global__ void __launch_bounds__(kThreads, kF > 4 ? 4 : 6) merge_kernel(const __grid_constant__ DecodeParams p) {
    const int row = int((blockIdx.x * size_t(kThreads) + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.total_rows) return;
    const int qt = row / p.Hq, h = row % p.Hq;
    // the token's 64-byte record: every lane loads the same four 16-byte words (a broadcast)
    const int4 *rec = reinterpret_cast<const int4 *>(p.q_merge + qt);
    const int4 r0 = __ldg(rec), r1 = __ldg(rec + 1), r2 = __ldg(rec + 2), r3 = __ldg(rec + 3);
    if (r0.z) return;  // its only chunk wrote the output
    const int n = r0.y, i = r0.w, pos = r1.x;
    const int g = h / p.G, jh = h % p.G;
    const int off = (i * p.G + jh) * p.Hkv + g;
    // checked build: a partial row outside the scratch is flagged and left out
    auto row_ok = [&](int pr) {
        if (!kChecked || (pr >= 0 && pr < p.n_partial_rows)) return true;
        atomicOr(p.err, kErrBounds | kErrMerge);
        return false;
    };

    if (n <= kMergeInline) {
        // every partial's lse and its O slice loaded at once, then summed in the plan's order
        const int base[kMergeInline] = {r1.y, r1.z, r1.w, r2.x, r2.y};
        const int lpos[kMergeInline] = {r2.z, r2.w, r3.x, r3.y, r3.z};
        float ls[kMergeInline];
        float4 v[kMergeInline];
#pragma unroll
        for (int k = 0; k < kMergeInline; ++k) {
            const bool use = k < n && lpos[k] <= pos && row_ok(base[k] + off);
            ls[k] = use ? p.part_lse[base[k] + off] : -INFINITY;
            v[k] = use ? *reinterpret_cast<const float4 *>(p.part_o + size_t(base[k] + off) * kHeadDim + lane * 4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMergeInline; ++k) M = fmaxf(M, ls[k]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int k = 0; k < kMergeInline; ++k) {
                if (ls[k] != -INFINITY) {
                    const float w = expf(ls[k] - M);
                    L += w;
                    acc.x += w * v[k].x; acc.y += w * v[k].y;
                    acc.z += w * v[k].z; acc.w += w * v[k].w;
                }
            }
            const float inv = 1.f / L;
            acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
        }
        store_row(p, row, lane, acc, (M == -INFINITY) ? -INFINITY : M + logf(L));
        return;
    }

    // more partials than the record holds: their bases from the branch's list
    const int32_t *bases = p.merge_bases + r0.x;
    const int32_t *lp = p.merge_lpos + r0.x;
    // a partial whose chunk starts after the token holds nothing it sees (and may never have
    // been written): it gets weight zero
    auto seen = [&](int k) { return __ldg(lp + k) <= pos && row_ok(bases[k] + off); };

    // partial k's lse sits in lane k % 32 (rounds of 32); max and weights by shuffles
    float M = -INFINITY;
    for (int k0 = 0; k0 < n; k0 += 32)
        if (k0 + lane < n && seen(k0 + lane)) M = fmaxf(M, p.part_lse[bases[k0 + lane] + off]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
        for (int k0 = 0; k0 < n; k0 += 32) {
            const int kn = min(32, n - k0);
            float wl = 0.f;
            int pr = 0;
            if (lane < kn && seen(k0 + lane)) {
                pr = bases[k0 + lane] + off;
                wl = expf(p.part_lse[pr] - M);
            }
            // the O terms in the plan's order, kF loads in flight (the last group is
            // predicated rather than walked one partial at a time)
            for (int k = 0; k < kn; k += kF) {
                float w[kF];
                int r[kF];
                float4 v[kF];
#pragma unroll
                for (int u = 0; u < kF; ++u) {
                    w[u] = __shfl_sync(0xffffffffu, wl, (k + u) & 31);
                    r[u] = __shfl_sync(0xffffffffu, pr, (k + u) & 31);
                }
#pragma unroll
                for (int u = 0; u < kF; ++u)
                    v[u] = k + u < kn && w[u] != 0.f
                               ? *reinterpret_cast<const float4 *>(p.part_o + size_t(r[u]) * kHeadDim + lane * 4)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int u = 0; u < kF; ++u) {
                    if (k + u < kn && w[u] != 0.f) {
                        L += w[u];
                        acc.x += w[u] * v[u].x; acc.y += w[u] * v[u].y;
                        acc.z += w[u] * v[u].z; acc.w += w[u] * v[u].w;
                    }
                }
            }
        }
        const float inv = 1.f / L;
        acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    }
    store_row(p, row, lane, acc, (M == -INFINITY) ? -INFINITY : M + logf(L));
}

}  // namespace mergek
}  // namespace fa

namespace fa {
namespace mergek {

// Merge of whole per-part results of the same query rows (a problem split into parts that
// each saw a disjoint share of every branch's entries, for instance one range of logical
// positions per GPU): part k holds out_k [rows][128] fp32 and lse_k [rows]; the same log-sum-
// exp merge as above, parts in order, one warp per row.
__global__ void __launch_bounds__(kThreads) merge_parts_kernel(const float *part_out, const float *part_lse,
                                                               int32_t n_parts, int64_t rows, void *out,
                                                               int32_t out_dtype, float *lse) {
    const int64_t row = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float M = -INFINITY;
    for (int k0 = 0; k0 < n_parts; k0 += 32)
        if (k0 + lane < n_parts) M = fmaxf(M, part_lse[size_t(k0 + lane) * rows + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
        for (int k = 0; k < n_parts; ++k) {
            const float l = part_lse[size_t(k) * rows + row];
            if (l == -INFINITY) continue;  // the part saw nothing of this row
            const float w = expf(l - M);
            const float4 v = *reinterpret_cast<const float4 *>(part_out + (size_t(k) * rows + row) * kHeadDim + lane * 4);
            L += w;
            acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
        }
        const float inv = 1.f / L;
        acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    }
    if (out_dtype == FA_F32) {
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + size_t(row) * kHeadDim + lane * 4) = acc;
    } else {
        uint2 pk = make_uint2(ptx::pack_bf16(acc.x, acc.y), ptx::pack_bf16(acc.z, acc.w));
        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(out) + size_t(row) * kHeadDim + lane * 4) = pk;
    }
    if (lane == 0) lse[row] = (M == -INFINITY) ? -INFINITY : M + logf(L);
}

}  // namespace mergek
}  // namespace fa
