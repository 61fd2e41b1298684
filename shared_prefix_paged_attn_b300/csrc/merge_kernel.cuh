// Log-sum-exp merge of partial results.
//
// Agentrix (gitlink.org.cn), section "初赛基础与决赛演进", CUDA ForkAttention: after the
// common part is computed once for all branches and the private parts per branch, each
// branch's results are merged.  For a (query token, query head) row with partials
// (O_k, lse_k) over disjoint sets of entries:
//     L = max_k lse_k + ln sum_k exp(lse_k - max_k lse_k),    O = sum_k exp(lse_k - L) O_k.
// One warp per row; each lane owns 4 of the 128 dims.  The row's merge record is one load;
// the partials' lse values are spread over the lanes (max and weights by shuffles); the O
// terms are summed in the plan's fixed order, eight loads in flight at a time, so the result
// is bitwise run-to-run deterministic.
#pragma once
#include "decode_params.cuh"
#include "ptx.cuh"

namespace fa {
namespace mergek {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) merge_kernel(const __grid_constant__ DecodeParams p) {
    const int row = int((blockIdx.x * size_t(kThreads) + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.total_rows) return;
    const int qt = row / p.Hq, h = row % p.Hq;
    const int4 qm = __ldg(reinterpret_cast<const int4 *>(p.q_merge) + qt);  // merge_off, n, direct, i
    if (qm.z) return;  // its only chunk wrote the output
    const int g = h / p.G, jh = h % p.G;
    const int off = (qm.w * p.G + jh) * p.Hkv + g;
    const int32_t *bases = p.merge_bases + qm.x;
    const int n = qm.y;

    // partial k's lse sits in lane k % 32 (rounds of 32); max and weights by shuffles
    float M = -INFINITY;
    for (int k0 = 0; k0 < n; k0 += 32)
        if (k0 + lane < n) M = fmaxf(M, p.part_lse[bases[k0 + lane] + off]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
        for (int k0 = 0; k0 < n; k0 += 32) {
            const int kn = min(32, n - k0);
            float wl = 0.f;
            int pr = 0;
            if (lane < kn) {
                pr = bases[k0 + lane] + off;
                wl = expf(p.part_lse[pr] - M);
            }
            // the O terms in the plan's order, eight loads in flight (the last group is
            // predicated rather than walked one partial at a time)
            for (int k = 0; k < kn; k += 8) {
                float w[8];
                int r[8];
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    w[u] = __shfl_sync(0xffffffffu, wl, (k + u) & 31);
                    r[u] = __shfl_sync(0xffffffffu, pr, (k + u) & 31);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    v[u] = k + u < kn ? *reinterpret_cast<const float4 *>(p.part_o + size_t(r[u]) * kHeadDim + lane * 4)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (k + u < kn) {
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
    if (p.out_dtype == FA_F32) {
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + size_t(row) * kHeadDim + lane * 4) = acc;
    } else {
        uint2 pk = make_uint2(ptx::pack_bf16(acc.x, acc.y), ptx::pack_bf16(acc.z, acc.w));
        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + size_t(row) * kHeadDim + lane * 4) = pk;
    }
    if (lane == 0) p.lse[row] = (M == -INFINITY) ? -INFINITY : M + logf(L);
}

}  // namespace mergek
}  // namespace fa
