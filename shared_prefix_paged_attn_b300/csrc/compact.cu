// Physical compaction of branches' kept cache entries, with optional repositioning.
//
// AgentKV blog (rit.work), "Как AgentKV выбирает и освобождает записи кэша": the kept entries
// are physically packed into fresh pages so that the freed pages go back to the allocator and
// a smaller cache is also fewer bytes read.  AKV (news.farwalk.ai), "AKV 如何工作？": Repos
// rewrites the kept keys to positions 0..r-1 with a RoPE rotation; values stay as they are.
//
// Host: a plan lists, per kept entry of the listed branches (logical order, branch after
// branch; with share_prefix the listed branches' common prefix once, first), its source
// slot, its destination slot and the position change n - j.  Device: one warp per entry,
// looping over the KV heads with eight heads' loads in flight; each lane moves 8 bytes of K
// and of V per head.  With repositioning the warp computes the entry's rotation factors once
// and applies them to the keys of every head; a lane rotates its four K values against the
// partner dims (i <-> i + 64) of lane ^ 16.  The rotation angle
// delta * theta_i is reduced exactly: theta_i / (2 pi) is held as a 64-bit fixed-point
// fraction of a turn, so delta times it, modulo 2^64, is the angle's fraction of a turn
// whatever the size of delta; the nearest quarter turn is applied exactly (swaps, signs) and
// sincosf only sees the residual in [-pi/4, pi/4).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <new>
#include <vector>

#include "../../include/fork_attn.h"

namespace fa {
namespace compactk {

constexpr int kHeadDim = 128;
constexpr int kPageSize = 16;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct Params {
    unsigned long long frac[kHeadDim / 2];  // theta_i / (2 pi) in units of 2^-64 turns
    __nv_bfloat16 *k;
    __nv_bfloat16 *v;
    const int32_t *src;    // [n] source slot (page * 16 + offset)
    const int32_t *dst;    // [n] destination slot
    const int32_t *delta;  // [n] new position - old position
    int64_t n_units;       // n * Hkv
    int32_t hkv;
    int32_t reposition;
};

__device__ __forceinline__ size_t slot_offset(int32_t slot, int g, int hkv) {
    // element offset of (page, head g, token) in [pages][Hkv][16][128]
    return ((size_t(slot >> 4) * hkv + g) * kPageSize + (slot & 15)) * kHeadDim;
}

// The rotation factors of lane `lane`'s four dims i = 4 (lane % 16) + c for a position
// change d: the nearest quarter turn of d theta_i applied exactly, sincosf on the residual.
__device__ __forceinline__ void rotation(const Params &p, int lane, int32_t d, float (&co)[4], float (&sn)[4]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int i = (lane & 15) * 4 + c;
        const unsigned long long turn = (unsigned long long)(long long)d * p.frac[i];
        const unsigned q = unsigned((turn + (1ull << 61)) >> 62);
        const long long res = (long long)(turn - ((unsigned long long)q << 62));
        const float ang = float(res) * 3.4061215800865545e-19f;  // 2 pi / 2^64
        float s0, c0;
        sincosf(ang, &s0, &c0);
        co[c] = q == 0 ? c0 : q == 1 ? -s0 : q == 2 ? -c0 : s0;
        sn[c] = q == 0 ? s0 : q == 1 ? c0 : q == 2 ? -s0 : -c0;
    }
}

// One warp per entry: with repositioning its rotation factors are computed once and applied
// to the keys of every KV head; eight heads' K and V loads are in flight at a time.
constexpr int kHeadsInFlight = 8;

__global__ void __launch_bounds__(kThreads) compact_kernel(const __grid_constant__ Params p) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t n_warps = (int64_t(gridDim.x) * kThreads) >> 5;
    const int64_t n_entries = p.n_units / p.hkv;
    const bool first = lane < 16;
    for (int64_t e = warp0; e < n_entries; e += n_warps) {
        const int32_t src = __ldg(p.src + e), dst = __ldg(p.dst + e);
        const int32_t d = p.reposition ? __ldg(p.delta + e) : 0;
        float co[4], sn[4];
        if (d != 0) rotation(p, lane, d, co, sn);  // warp-uniform
        for (int g0 = 0; g0 < p.hkv; g0 += kHeadsInFlight) {
            uint2 kv[kHeadsInFlight], vv[kHeadsInFlight];
#pragma unroll
            for (int u = 0; u < kHeadsInFlight; ++u) {
                kv[u] = vv[u] = make_uint2(0, 0);
                if (g0 + u < p.hkv) {
                    const size_t so = slot_offset(src, g0 + u, p.hkv) + lane * 4;
                    kv[u] = *reinterpret_cast<const uint2 *>(p.k + so);
                    vv[u] = *reinterpret_cast<const uint2 *>(p.v + so);
                }
            }
#pragma unroll
            for (int u = 0; u < kHeadsInFlight; ++u) {
                if (g0 + u >= p.hkv) break;  // warp-uniform
                const size_t doff = slot_offset(dst, g0 + u, p.hkv) + lane * 4;
                *reinterpret_cast<uint2 *>(p.v + doff) = vv[u];
                uint2 out = kv[u];
                if (d != 0) {
                    // lane l < 16 holds dims 4l..4l+3 (first halves), lane l + 16 the partners + 64
                    const uint2 part = make_uint2(__shfl_xor_sync(0xffffffffu, kv[u].x, 16),
                                                  __shfl_xor_sync(0xffffffffu, kv[u].y, 16));
                    const __nv_bfloat162 *m2 = reinterpret_cast<const __nv_bfloat162 *>(&kv[u]);
                    const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&part);
                    const float mine[4] = {__low2float(m2[0]), __high2float(m2[0]), __low2float(m2[1]), __high2float(m2[1])};
                    const float other[4] = {__low2float(p2[0]), __high2float(p2[0]), __low2float(p2[1]), __high2float(p2[1])};
                    float r[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        // first half: x_i cos - x_{i+64} sin; second half: x_{i+64} cos + x_i sin
                        r[c] = first ? mine[c] * co[c] - other[c] * sn[c] : mine[c] * co[c] + other[c] * sn[c];
                    __nv_bfloat162 o0 = __floats2bfloat162_rn(r[0], r[1]), o1 = __floats2bfloat162_rn(r[2], r[3]);
                    out.x = *reinterpret_cast<uint32_t *>(&o0);
                    out.y = *reinterpret_cast<uint32_t *>(&o1);
                }
                *reinterpret_cast<uint2 *>(p.k + doff) = out;
            }
        }
    }
}

}  // namespace compactk
}  // namespace fa

struct fa_compact {
    int32_t hkv = 0;
    int32_t reposition = 0;
    double rope_base = 10000.0;
    std::vector<int64_t> kept;   // per listed branch
    int64_t shared_kept = 0;     // kept entries of the shared run (share_prefix)
    int64_t prefix_len = 0;      // the common prefix's logical entries (share_prefix)
    std::vector<int32_t> blob;   // [src n][dst n][delta n]
    int64_t n = 0;
    void *dev_work = nullptr;
};

namespace {

inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" int fork_attn_compact_create(const fa_compact_dims *dims, const fa_desc *d, const int32_t *branches,
                                        int32_t num_branches, const int32_t *dst_page_ids, int64_t num_dst_pages,
                                        fa_compact **out) {
    if (!dims || !d || !out || (num_branches > 0 && !branches) || (num_dst_pages > 0 && !dst_page_ids))
        return FA_ERR_NULL;
    if (dims->head_dim != 128 || dims->page_size != 16) return FA_ERR_UNSUPPORTED;
    if (dims->num_kv_heads < 1 || num_branches < 0 || num_dst_pages < 0) return FA_ERR_INVALID;
    if (dims->reposition && !(dims->rope_base > 1.0)) return FA_ERR_INVALID;
    if (!d->page_ids || !d->segs || !d->branch_seg_off || !d->branch_segs || d->num_branches < 1) return FA_ERR_NULL;
    if ((d->vis_bits == nullptr) != (d->vis_word_off == nullptr)) return FA_ERR_INVALID;
    const int64_t pool = d->num_pages_pool;
    if (pool < 1 || pool > (int64_t(1) << 27)) return FA_ERR_RANGE;  // slots fit in int32
    if ((dims->share_prefix != 0 && dims->share_prefix != 1) || dims->reserved != 0) return FA_ERR_INVALID;
    try {
        std::unique_ptr<fa_compact> c(new fa_compact());
        c->hkv = dims->num_kv_heads;
        c->reposition = dims->reposition != 0;
        c->rope_base = dims->rope_base;
        std::vector<char> used(size_t(pool), 0);  // source pages of the listed branches
        std::vector<char> taken(size_t(pool), 0);  // destination pages
        // pass 1: every listed branch's logical entries as (physical slot, visible)
        std::vector<std::vector<int32_t>> slots(static_cast<size_t>(num_branches));
        std::vector<std::vector<char>> vis(static_cast<size_t>(num_branches));
        for (int32_t k = 0; k < num_branches; ++k) {
            const int32_t b = branches[k];
            if (b < 0 || b >= d->num_branches) return FA_ERR_INVALID;
            const int32_t s0 = d->branch_seg_off[b], s1 = d->branch_seg_off[b + 1];
            if (s0 < 0 || s1 < s0) return FA_ERR_INVALID;
            int64_t j = 0;
            const int64_t w0 = d->vis_word_off ? d->vis_word_off[b] : 0;
            for (int32_t si = s0; si < s1; ++si) {
                const int32_t sid = d->branch_segs[si];
                if (sid < 0 || sid >= d->num_segs) return FA_ERR_RANGE;
                const fa_segment sg = d->segs[sid];
                if (sg.len < 1 || sg.tok_begin < 0 || sg.tok_begin >= 16 || sg.page_off < 0) return FA_ERR_INVALID;
                const int64_t last_page = sg.page_off + (sg.tok_begin + int64_t(sg.len) - 1) / 16;
                if (last_page >= d->num_page_ids) return FA_ERR_RANGE;
                for (int32_t t = 0; t < sg.len; ++t, ++j) {
                    const int64_t pos = sg.tok_begin + t;
                    const int32_t page = d->page_ids[sg.page_off + pos / 16];
                    if (page < 0 || page >= pool) return FA_ERR_RANGE;
                    used[size_t(page)] = 1;
                    bool v = true;
                    if (d->vis_bits) {
                        const int64_t wi = w0 + j / 32;
                        if (wi < 0 || wi >= d->num_vis_words) return FA_ERR_RANGE;
                        v = (d->vis_bits[wi] >> (j % 32)) & 1u;
                    }
                    slots[k].push_back(page * 16 + int32_t(pos % 16));
                    vis[k].push_back(v ? 1 : 0);
                }
            }
        }
        // the common prefix: entries at which every listed branch has the same slot and bit
        int64_t P = 0;
        if (dims->share_prefix && num_branches > 0) {
            size_t lim = slots[0].size();
            for (const auto &x : slots) lim = std::min(lim, x.size());
            while (size_t(P) < lim) {
                bool same = true;
                for (int32_t k = 1; k < num_branches && same; ++k)
                    same = slots[k][size_t(P)] == slots[0][size_t(P)] && vis[k][size_t(P)] == vis[0][size_t(P)];
                if (!same) break;
                ++P;
            }
        }
        // pass 2: the shared run once, then each branch's entries after it, each run from a
        // fresh destination page; entry n of a branch moves from position j to n
        std::vector<int32_t> src, dst, dl;
        int64_t next_dst = 0;
        auto place = [&](int64_t count) -> int {  // destination slots of `count` packed entries
            const int64_t np = ceil_div64(count, 16);
            if (next_dst + np > num_dst_pages) return FA_ERR_INVALID;
            for (int64_t q = 0; q < np; ++q) {
                const int32_t page = dst_page_ids[next_dst + q];
                if (page < 0 || page >= pool) return FA_ERR_RANGE;
                if (taken[size_t(page)]) return FA_ERR_INVALID;  // listed twice
                taken[size_t(page)] = 1;
            }
            for (int64_t e = 0; e < count; ++e) dst.push_back(dst_page_ids[next_dst + e / 16] * 16 + int32_t(e % 16));
            next_dst += np;
            return FA_OK;
        };
        int64_t kept_s = 0;
        if (num_branches > 0)
            for (int64_t j = 0; j < P; ++j)
                if (vis[0][size_t(j)]) {
                    src.push_back(slots[0][size_t(j)]);
                    dl.push_back(int32_t(kept_s - j));
                    ++kept_s;
                }
        if (const int rc = place(kept_s)) return rc;
        for (int32_t k = 0; k < num_branches; ++k) {
            int64_t kept = kept_s;
            for (size_t j = size_t(P); j < slots[k].size(); ++j)
                if (vis[k][j]) {
                    src.push_back(slots[k][j]);
                    dl.push_back(int32_t(kept - int64_t(j)));
                    ++kept;
                }
            if (const int rc = place(kept - kept_s)) return rc;
            c->kept.push_back(kept);
        }
        c->shared_kept = kept_s;
        c->prefix_len = P;
        for (int64_t q = 0; q < next_dst; ++q)
            if (used[size_t(dst_page_ids[q])]) return FA_ERR_INVALID;  // would overwrite a source
        c->n = int64_t(src.size());
        c->blob.reserve(size_t(3 * c->n));
        c->blob.insert(c->blob.end(), src.begin(), src.end());
        c->blob.insert(c->blob.end(), dst.begin(), dst.end());
        c->blob.insert(c->blob.end(), dl.begin(), dl.end());
        *out = c.release();
        return FA_OK;
    } catch (const std::bad_alloc &) {
        return FA_ERR_NOMEM;
    }
}

extern "C" int fork_attn_compact_sizes(const fa_compact *c, int64_t *kept_tokens, size_t *work_bytes) {
    if (!c) return FA_ERR_NULL;
    if (kept_tokens)
        for (size_t k = 0; k < c->kept.size(); ++k) kept_tokens[k] = c->kept[k];
    if (work_bytes) *work_bytes = size_t(std::max<int64_t>(c->n, 1)) * 3 * sizeof(int32_t);
    return FA_OK;
}

extern "C" int fork_attn_compact_shared(const fa_compact *c, int64_t *shared_kept, int64_t *prefix_len) {
    if (!c) return FA_ERR_NULL;
    if (shared_kept) *shared_kept = c->shared_kept;
    if (prefix_len) *prefix_len = c->prefix_len;
    return FA_OK;
}

extern "C" int fork_attn_compact_upload(fa_compact *c, void *dev_work, size_t work_bytes, void *stream) {
    if (!c || !dev_work) return FA_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(dev_work) & 255u) return FA_ERR_ALIGN;
    const size_t need = size_t(std::max<int64_t>(c->n, 1)) * 3 * sizeof(int32_t);
    if (work_bytes < need) return FA_ERR_BUFFER_SMALL;
    if (c->n > 0 && cudaMemcpyAsync(dev_work, c->blob.data(), size_t(c->n) * 3 * sizeof(int32_t),
                                    cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FA_ERR_CUDA;
    c->dev_work = dev_work;
    return FA_OK;
}

extern "C" int fork_attn_compact_run(const fa_compact *c, void *k_pages, void *v_pages, void *stream) {
    if (!c || !k_pages || !v_pages) return FA_ERR_NULL;
    if (!c->dev_work) return FA_ERR_NOT_UPLOADED;
    if ((reinterpret_cast<uintptr_t>(k_pages) | reinterpret_cast<uintptr_t>(v_pages)) & 15u) return FA_ERR_ALIGN;
    if (c->n == 0) return FA_OK;
    fa::compactk::Params p;
    std::memset(&p, 0, sizeof p);
    for (int i = 0; i < fa::compactk::kHeadDim / 2; ++i) {
        // theta_i / (2 pi) as a fraction of a turn in units of 2^-64 (theta_i <= 1 < 2 pi)
        const long double turn = std::pow((long double)c->rope_base, -2.0L * i / fa::compactk::kHeadDim) /
                                 (2.0L * 3.14159265358979323846264338327950288L);
        p.frac[i] = (unsigned long long)(turn * 18446744073709551616.0L);
    }
    const int32_t *w = static_cast<const int32_t *>(c->dev_work);
    p.k = static_cast<__nv_bfloat16 *>(k_pages);
    p.v = static_cast<__nv_bfloat16 *>(v_pages);
    p.src = w;
    p.dst = w + c->n;
    p.delta = w + 2 * c->n;
    p.n_units = c->n * c->hkv;
    p.hkv = c->hkv;
    p.reposition = c->reposition;
    const int64_t blocks = std::min<int64_t>(ceil_div64(c->n, fa::compactk::kWarps), 148 * 8);
    fa::compactk::compact_kernel<<<unsigned(blocks), fa::compactk::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" int fork_attn_compact_destroy(fa_compact *c) {
    if (!c) return FA_ERR_NULL;
    delete c;
    return FA_OK;
}
