// C ABI of key scoring and top-k keep (fork_attn_score, fork_attn_topk): argument checks and
// the launches of the scoring, head-reduce and top-k kernels on a plan of representative
// queries.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "plan_internal.h"
#include "score_kernel.cuh"
#include "tensor_map.h"
#include "topk_kernel.cuh"

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int score_setup(int *num_sms) {
    static std::mutex mu;
    static bool done[128] = {false};
    static int sms[128] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(mu);
    if (!done[dev]) {
        if (cudaFuncSetAttribute(fa::sck::score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(fa::sck::kSmemBytes)) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        done[dev] = true;
    }
    *num_sms = sms[dev];
    return FA_OK;
}

}  // namespace

extern "C" int fork_attn_score(const void *q, const void *k_pages, const fa_plan *plan, const float *lse,
                               float *scores, void *stream) {
    if (!q || !k_pages || !plan || !lse || !scores) return FA_ERR_NULL;
    if (!plan->representatives) return FA_ERR_INVALID;
    if (!plan->uploaded) return FA_ERR_NOT_UPLOADED;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(lse, 4) || !aligned(scores, 4)) return FA_ERR_ALIGN;
    const fa::Layout &L = plan->lay;
    const int64_t E = L.total_entries;
    if (E == 0) return FA_OK;
    int num_sms = 0;
    if (const int rc = score_setup(&num_sms)) return rc;
    fa::sck::Params p;
    std::memset(&p, 0, sizeof p);
    if (!fa::tmap::encode_pages(&p.kmap, k_pages, plan->num_pages_pool, plan->dims.num_kv_heads)) return FA_ERR_CUDA;
    uint8_t *base = static_cast<uint8_t *>(plan->dev_plan);
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.lse = lse;
    p.chunk_pages = reinterpret_cast<const int32_t *>(base + L.chunk_pages);
    p.chunks = reinterpret_cast<const fa::Chunk *>(base + L.chunks);
    p.items = reinterpret_cast<const fa::Item *>(base + L.score_items);
    p.units = reinterpret_cast<const int4 *>(base + L.score_units);
    p.rows = reinterpret_cast<const fa::RowRec *>(base + L.rows);
    p.occ_pos = reinterpret_cast<const int32_t *>(base + L.occ_pos);
    p.row_pos = reinterpret_cast<const int32_t *>(base + L.row_pos);
    p.mask_words = reinterpret_cast<const uint32_t *>(base + L.mask_words);
    p.part = reinterpret_cast<float *>(static_cast<uint8_t *>(plan->dev_scratch) + fa::score_part_offset(plan));
    p.err = reinterpret_cast<int32_t *>(base);
    p.queue = p.err + 3;
    p.total_entries = E;
    p.n_units = L.n_score_units;
    p.G = plan->G;
    p.pool_pages = int32_t(plan->num_pages_pool);
    p.scale_log2 = plan->dims.scale * 1.4426950408889634f;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int32_t hkv = plan->dims.num_kv_heads;
    // per-head scores start as NaN: an entry no item writes is one its branch does not see
    if (cudaMemsetAsync(p.part, 0xFF, size_t(hkv) * size_t(E) * sizeof(float), st) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaMemsetAsync(p.queue, 0, sizeof(int32_t), st) != cudaSuccess) return FA_ERR_CUDA;
    plan->err_word = p.err;
    if (p.n_units > 0) {
        const int grid = std::min(num_sms, p.n_units);
        fa::sck::score_kernel<<<grid, fa::sck::kThreads, fa::sck::kSmemBytes, st>>>(p);
        if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    }
    const int64_t blocks = std::min<int64_t>((E + 255) / 256, int64_t(num_sms) * 8);
    fa::sck::score_reduce_kernel<<<unsigned(blocks), 256, 0, st>>>(
        p.part, reinterpret_cast<const int32_t *>(base + L.entry_off), reinterpret_cast<const fa::Branch *>(base + L.branches),
        scores, E, L.n_branches, hkv, plan->dims.num_q_heads);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" int fork_attn_topk(const fa_plan *plan, const float *scores, const int32_t *keep_k, uint32_t *keep_bits,
                              void *stream) {
    if (!plan || !scores || !keep_k || !keep_bits) return FA_ERR_NULL;
    if (!plan->representatives) return FA_ERR_INVALID;
    if (!plan->uploaded) return FA_ERR_NOT_UPLOADED;
    if (!aligned(scores, 4) || !aligned(keep_k, 4) || !aligned(keep_bits, 4)) return FA_ERR_ALIGN;
    const fa::Layout &L = plan->lay;
    uint8_t *base = static_cast<uint8_t *>(plan->dev_plan);
    fa::topk::topk_kernel<<<unsigned(L.n_branches), fa::topk::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        scores, reinterpret_cast<const int32_t *>(base + L.entry_off), reinterpret_cast<const int32_t *>(base + L.word_off),
        keep_k, keep_bits);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" int fork_attn_score_sizes(const fa_plan *plan, int64_t *total_entries, int64_t *total_words) {
    if (!plan) return FA_ERR_NULL;
    if (!plan->representatives) return FA_ERR_INVALID;
    if (total_entries) *total_entries = plan->lay.total_entries;
    if (total_words) *total_words = plan->lay.total_words;
    return FA_OK;
}
