// Top-k keep of scored cache entries: one CTA per branch.
//
// AgentKV blog (rit.work), "Как AgentKV выбирает и освобождает записи кэша": the entries with
// the largest mean attention from the representatives are kept.  For branch b, of its visible
// entries (a finite score; the ones it does not see hold NaN) the k_b with the largest scores
// are kept; equal scores keep the smaller logical index; k_b >= the visible count keeps them
// all, k_b <= 0 none.  The result is the branch's new visibility bits (bit j % 32 of word
// word_off[b] + j / 32 for logical index j), the layout the planner and compaction take.
//
// Scores are >= 0, so their fp32 bit patterns order as the values do.  The k-th largest
// pattern T is found by radix selection over the top 12, middle 12 and low 8 bits (a
// histogram in shared memory per round, its bins scanned from the top), which also gives how
// many entries equal to T are kept; a last pass keeps every entry above T and, when not all
// entries equal to T fit, the first of them in index order (a block-wide prefix count), one
// 32-bit word per warp.
#pragma once
#include <stdint.h>

namespace fa {
namespace topk {

constexpr int kThreads = 1024;
constexpr int kBins = 4096;

// Exclusive prefix sum over the block (thread order) of v; *total gets the sum of all.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_sums, uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = warp_sums[lane], wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        warp_sums[lane] = wi - w;  // exclusive prefix of the warp sums
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    const uint32_t r = warp_sums[warp] + incl - v;
    *total = warp_sums[32];
    __syncthreads();  // warp_sums may be reused right after
    return r;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const float *scores, const int32_t *entry_off,
                                                        const int32_t *word_off, const int32_t *keep_k,
                                                        uint32_t *keep_bits) {
    __shared__ uint32_t hist[kBins];
    __shared__ uint32_t warp_sums[33];
    __shared__ uint32_t sel[3];  // selected bin, entries above it, entries in it
    const int b = blockIdx.x, tid = threadIdx.x;
    const int64_t e0 = entry_off[b];
    const int n = int(entry_off[b + 1] - e0);
    const float *sc = scores + e0;
    const int k = keep_k[b];

    // radix selection of the k-th largest bit pattern among the visible entries
    uint32_t prefix = 0, mask = 0;
    int64_t remaining = k;
    bool keep_all = false, keep_none = k <= 0;
    uint32_t n_equal = 0;
    const int shifts[3] = {20, 8, 0};
    const uint32_t widths[3] = {0xFFFu, 0xFFFu, 0xFFu};
    for (int round = 0; round < 3 && !keep_all && !keep_none; ++round) {
        for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
        __syncthreads();
        const int sh = shifts[round];
        const uint32_t wd = widths[round];
        auto count = [&](float s) {
            if (s != s) return;  // not visible
            const uint32_t bits = __float_as_uint(s);
            if ((bits & mask) == prefix) atomicAdd(&hist[(bits >> sh) & wd], 1u);
        };
        // the entries up to the first 16-byte boundary one by one, then four per load
        const int head = min(n, int((4 - ((reinterpret_cast<uintptr_t>(sc) >> 2) & 3)) & 3));
        if (tid < head) count(sc[tid]);
        const float4 *sc4 = reinterpret_cast<const float4 *>(sc + head);
        const int n4 = (n - head) >> 2;
        for (int e = tid; e < n4; e += kThreads) {
            const float4 v = sc4[e];
            count(v.x);
            count(v.y);
            count(v.z);
            count(v.w);
        }
        for (int e = head + 4 * n4 + tid; e < n; e += kThreads) count(sc[e]);
        __syncthreads();
        // bins from the top: thread i sums bins 4095 - 4i .. 4092 - 4i
        uint32_t local = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) local += hist[kBins - 1 - 4 * tid - u];
        uint32_t total;
        const uint32_t above = block_excl_scan(local, warp_sums, &total);
        if (round == 0) {
            if (int64_t(total) <= remaining) keep_all = true;  // k >= visible entries
        }
        if (!keep_all) {
            if (above < remaining && remaining <= int64_t(above) + local) {
                uint32_t acc = above;
                for (int u = 0; u < 4; ++u) {
                    const int bin = kBins - 1 - 4 * tid - u;
                    if (remaining <= int64_t(acc) + hist[bin]) {
                        sel[0] = uint32_t(bin);
                        sel[1] = acc;
                        sel[2] = hist[bin];
                        break;
                    }
                    acc += hist[bin];
                }
            }
            __syncthreads();
            prefix |= sel[0] << sh;
            mask |= widths[round] << sh;
            remaining -= sel[1];
            n_equal = sel[2];  // after the last round: the visible entries equal to T
        }
        __syncthreads();
    }
    // keep: above T, or equal to T among the first `remaining` in index order
    const uint32_t T = prefix;
    uint32_t carry = 0;
    const int lane = tid & 31, warp = tid >> 5;
    const int n_words = (n + 31) / 32;
    if (keep_all || keep_none || int64_t(n_equal) <= remaining) {
        // every entry equal to T is kept too: no order needed, one word per warp at a time
        for (int wi = warp; wi < n_words; wi += kThreads / 32) {
            const int e = 32 * wi + lane;
            bool keep = false;
            if (e < n && !keep_none) {
                const float s = sc[e];
                keep = s == s && (keep_all || __float_as_uint(s) >= T);
            }
            const uint32_t word = __ballot_sync(0xffffffffu, keep);
            if (lane == 0) keep_bits[word_off[b] + wi] = word;
        }
        return;
    }
    for (int base = 0; base < n; base += kThreads) {
        const int e = base + tid;
        bool vis = false, gt = false, eq = false;
        if (e < n) {
            const float s = sc[e];
            vis = s == s;
            if (vis) {
                const uint32_t bits = __float_as_uint(s);
                gt = bits > T;
                eq = bits == T;
            }
        }
        uint32_t n_eq;
        const uint32_t before = block_excl_scan(eq ? 1u : 0u, warp_sums, &n_eq);
        const bool keep = !keep_none && vis && (keep_all || gt || (eq && int64_t(carry) + before < remaining));
        const uint32_t word = __ballot_sync(0xffffffffu, keep);
        const int wi = (base >> 5) + warp;
        if (lane == 0 && wi < n_words) keep_bits[word_off[b] + wi] = word;
        carry += n_eq;
    }
}

}  // namespace topk
}  // namespace fa
