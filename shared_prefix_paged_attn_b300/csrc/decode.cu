// Launcher side of the C ABI: plan upload, tensor-map encoding, kernel launches, error word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "merge_kernel.cuh"
#include "plan_internal.h"
#include "tensor_map.h"
#include "row8_kernel.cuh"
#include "row_kernel.cuh"
#include "tc_kernel.cuh"

namespace {

using fa::tmap::encode_pages;
using fa::tmap::encode_pages_whole;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int set_smem_attr() {
    // once per device: the kernels need more than the default 48 KiB of dynamic smem
    static std::mutex mu;
    static bool done[128] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(mu);
    if (!done[dev]) {
        if (cudaFuncSetAttribute(fa::rowk::row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(fa::rowk::kSmemBytes)) != cudaSuccess ||
            cudaFuncSetAttribute(fa::tck::tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(fa::tck::kSmemBytes)) != cudaSuccess ||
            cudaFuncSetAttribute(fa::tck::tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(fa::tck::kSmemBytes)) != cudaSuccess ||
            cudaFuncSetAttribute(fa::r8k::row8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(fa::r8k::kSmemBytes)) != cudaSuccess)
            return FA_ERR_CUDA;
        // the tcgen05 kernel re-splits its registers with setmaxnreg; the split must fit in
        // what the block is launched with, or the increase would wait forever
        cudaFuncAttributes fattr;
        for (const void *k : {reinterpret_cast<const void *>(fa::tck::tc_kernel<false>),
                              reinterpret_cast<const void *>(fa::tck::tc_kernel<true>)}) {
            if (cudaFuncGetAttributes(&fattr, k) != cudaSuccess) return FA_ERR_CUDA;
            if (int64_t(fattr.numRegs) * fa::tck::kThreads <
                128 * int64_t(fa::tck::kLowRegs) + int64_t(fa::tck::kThreads - 128) * fa::tck::kHighRegs)
                return FA_ERR_UNSUPPORTED;
        }
        done[dev] = true;
    }
    return FA_OK;
}

int fill_params(const fa_plan *plan, const void *q, const void *k_pages, const void *v_pages, void *out,
                float *lse, void *scratch, fa::DecodeParams &p) {
    std::memset(&p, 0, sizeof p);
    if (!encode_pages(&p.kmap, k_pages, plan->num_pages_pool, plan->dims.num_kv_heads) ||
        !encode_pages(&p.vmap, v_pages, plan->num_pages_pool, plan->dims.num_kv_heads) ||
        !encode_pages_whole(&p.kmap_page, k_pages, plan->num_pages_pool, plan->dims.num_kv_heads) ||
        !encode_pages_whole(&p.vmap_page, v_pages, plan->num_pages_pool, plan->dims.num_kv_heads))
        return FA_ERR_CUDA;
    const fa::Layout &L = plan->lay;
    uint8_t *base = static_cast<uint8_t *>(plan->dev_plan);
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.out = out;
    p.lse = lse;
    p.part_o = static_cast<float *>(scratch);
    p.part_lse = scratch ? reinterpret_cast<float *>(static_cast<uint8_t *>(scratch) +
                                                     fa::scratch_lse_offset(plan->partial_rows))
                         : nullptr;
    p.chunk_pages = reinterpret_cast<const int32_t *>(base + L.chunk_pages);
    p.chunks = reinterpret_cast<const fa::Chunk *>(base + L.chunks);
    p.items = reinterpret_cast<const fa::Item *>(base + L.items_rows);
    p.items_tc = reinterpret_cast<const fa::Item *>(base + L.items_tc);
    p.items_r8 = reinterpret_cast<const fa::Item *>(base + L.items_r8);
    p.rows = reinterpret_cast<const fa::RowRec *>(base + L.rows);
    p.branches = reinterpret_cast<const fa::Branch *>(base + L.branches);
    p.q_merge = reinterpret_cast<const fa::QMerge *>(base + L.q_merge);
    p.merge_bases = reinterpret_cast<const int32_t *>(base + L.merge_bases);
    p.merge_lpos = reinterpret_cast<const int32_t *>(base + L.merge_lpos);
    p.mask_words = reinterpret_cast<const uint32_t *>(base + L.mask_words);
    p.err = reinterpret_cast<int32_t *>(base);
    p.Hq = plan->dims.num_q_heads;
    p.Hkv = plan->dims.num_kv_heads;
    p.G = plan->G;
    p.out_dtype = plan->dims.out_dtype;
    p.scale_log2 = plan->dims.scale * 1.4426950408889634f;
    p.n_items = L.n_items_rows;
    p.n_items_tc = L.n_items_tc;
    p.n_items_r8 = L.n_items_r8;
    p.pool_pages = int32_t(plan->num_pages_pool);
    p.tc_ctas = plan->tc_ctas;
    p.total_rows = L.total_q * plan->dims.num_q_heads;
    p.n_partial_rows = int32_t(plan->partial_rows);
    p.n_mask_words = L.n_mask_words;
    return FA_OK;
}

bool needs_merge(const fa_plan *plan) { return plan->stats.merge_rows > 0; }

// Launches the decode kernels on `st`.  chain = true (fork_attn_decode): the tcgen05 kernel
// first, then the row kernels as programmatic dependent launches -- each CTA of the kernel
// before releases its dependents as soon as it starts, so the row kernels' CTAs are placed
// only after every persistent tcgen05 CTA holds its SM, and fill the SMs left over and those
// the tcgen05 CTAs free -- then the merge as an ordinary launch, which waits for all of them.
// The row kernels do not read what the tcgen05 kernel writes.  chain = false: the kernels
// one after another, with `events` (optional, 8 handles) recorded around each of them in the
// order row8, row, tcgen05, merge.
int launch_all(const fa::DecodeParams &p, const fa_plan *plan, cudaStream_t st, void **events, bool chain) {
    bool ev_ok = true;
    auto rec = [&](int i) {
        if (events) ev_ok = ev_ok && cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) == cudaSuccess;
    };
    bool after_kernel = false;  // a kernel of this decode precedes the next launch on `st`
    auto launch = [&](auto kernel, int grid, int threads, size_t smem) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(grid));
        cfg.blockDim = dim3(unsigned(threads));
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = chain && after_kernel ? 1 : 0;
        after_kernel = true;
        return cudaLaunchKernelEx(&cfg, kernel, p) == cudaSuccess;
    };
    bool ok = true;
    if (chain) {
        if (p.n_items_tc > 0)
            ok = ok && (p.lse_only ? launch(fa::tck::tc_kernel<true>, p.tc_ctas, fa::tck::kThreads, fa::tck::kSmemBytes)
                                   : launch(fa::tck::tc_kernel<false>, p.tc_ctas, fa::tck::kThreads, fa::tck::kSmemBytes));
        if (p.n_items_r8 > 0) ok = ok && launch(fa::r8k::row8_kernel, p.n_items_r8, fa::r8k::kThreads, fa::r8k::kSmemBytes);
        if (p.n_items > 0) ok = ok && launch(fa::rowk::row_kernel, p.n_items, fa::rowk::kThreads, fa::rowk::kSmemBytes);
    } else {
        rec(0);
        if (p.n_items_r8 > 0) ok = ok && launch(fa::r8k::row8_kernel, p.n_items_r8, fa::r8k::kThreads, fa::r8k::kSmemBytes);
        rec(1);
        rec(2);
        if (p.n_items > 0) ok = ok && launch(fa::rowk::row_kernel, p.n_items, fa::rowk::kThreads, fa::rowk::kSmemBytes);
        rec(3);
        rec(4);
        if (p.n_items_tc > 0)
            ok = ok && (p.lse_only ? launch(fa::tck::tc_kernel<true>, p.tc_ctas, fa::tck::kThreads, fa::tck::kSmemBytes)
                                   : launch(fa::tck::tc_kernel<false>, p.tc_ctas, fa::tck::kThreads, fa::tck::kSmemBytes));
        rec(5);
    }
    rec(6);
    if (needs_merge(plan)) {
        const int64_t threads = int64_t(p.total_rows) * 32;
        const int blocks = int((threads + fa::mergek::kThreads - 1) / fa::mergek::kThreads);
        if (plan->merge_wide)
            fa::mergek::merge_kernel<8><<<blocks, fa::mergek::kThreads, 0, st>>>(p);
        else
            fa::mergek::merge_kernel<4><<<blocks, fa::mergek::kThreads, 0, st>>>(p);
    }
    rec(7);
    const bool launched = ok && cudaGetLastError() == cudaSuccess;
    if (!ev_ok) return FA_ERR_INVALID;
    return launched ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" int fork_attn_plan_upload(fa_plan *plan, void *dev_plan_buf, size_t plan_buf_bytes,
                                     void *dev_scratch_buf, size_t scratch_buf_bytes, void *stream) {
    if (!plan || !dev_plan_buf) return FA_ERR_NULL;
    const size_t need_plan = size_t(plan->lay.total);
    const size_t need_scratch = size_t(fa::plan_scratch_bytes(plan));
    if (!aligned(dev_plan_buf, fa::kAlign)) return FA_ERR_ALIGN;
    if (plan_buf_bytes < need_plan) return FA_ERR_BUFFER_SMALL;
    if (need_scratch > 0) {
        if (!dev_scratch_buf) return FA_ERR_NULL;
        if (!aligned(dev_scratch_buf, fa::kAlign)) return FA_ERR_ALIGN;
        if (scratch_buf_bytes < need_scratch) return FA_ERR_BUFFER_SMALL;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(dev_plan_buf, plan->blob.data(), need_plan, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return FA_ERR_CUDA;
    plan->dev_plan = dev_plan_buf;
    plan->dev_scratch = dev_scratch_buf;
    plan->uploaded = true;
    plan->err_word = static_cast<int32_t *>(dev_plan_buf);
    return FA_OK;
}

extern "C" int fork_attn_decode_timed(const void *q, const void *k_pages, const void *v_pages,
                                      const fa_plan *plan, void *out, float *lse, void *stream,
                                      void **events, int32_t n_events) {
    if (!plan || !q || !k_pages || !v_pages || !out || !lse) return FA_ERR_NULL;
    if (!plan->uploaded) return FA_ERR_NOT_UPLOADED;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(lse, 16))
        return FA_ERR_ALIGN;
    if (events && n_events != 4) return FA_ERR_INVALID;
    int rc = set_smem_attr();
    if (rc != FA_OK) return rc;
    fa::DecodeParams p;
    rc = fill_params(plan, q, k_pages, v_pages, out, lse, plan->dev_scratch, p);
    if (rc != FA_OK) return rc;
    return launch_all(p, plan, static_cast<cudaStream_t>(stream), events, false);
}

extern "C" int fork_attn_decode(const void *q, const void *k_pages, const void *v_pages,
                                const fa_plan *plan, void *out, float *lse, void *stream) {
    if (!plan || !q || !k_pages || !v_pages || !out || !lse) return FA_ERR_NULL;
    if (!plan->uploaded) return FA_ERR_NOT_UPLOADED;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(lse, 16))
        return FA_ERR_ALIGN;
    int rc = set_smem_attr();
    if (rc != FA_OK) return rc;
    fa::DecodeParams p;
    rc = fill_params(plan, q, k_pages, v_pages, out, lse, plan->dev_scratch, p);
    if (rc != FA_OK) return rc;
    plan->err_word = static_cast<int32_t *>(plan->dev_plan);
    return launch_all(p, plan, static_cast<cudaStream_t>(stream), nullptr, true);
}

extern "C" int fork_attn_check(fa_plan *plan, int32_t *device_error, void *stream) {
    if (!plan || !device_error) return FA_ERR_NULL;
    if (!plan->err_word) return FA_ERR_NOT_UPLOADED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t word = 0;
    if (cudaMemcpyAsync(&word, plan->err_word, sizeof word, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return FA_ERR_CUDA;
    *device_error = word;
    if (word != 0) {
        if (cudaMemsetAsync(plan->err_word, 0, sizeof word, st) != cudaSuccess) return FA_ERR_CUDA;
        return FA_ERR_DEVICE;
    }
    return FA_OK;
}

// ---------------------------------------------------------------------------------------
// Decode without caller-provided device buffers beyond inputs and outputs.
//
// For callers that cannot allocate device memory (see fork_attn_decode_static_scratch in
// fork_attn.h): the plan arrays and the fp32 partials live in one file-scope device array.
// Nothing here allocates.  The array is shared by every call on a device; calls that overlap
// on the GPU race on it.
namespace {

constexpr size_t kStaticScratchBytes = FA_STATIC_SCRATCH_BYTES;
static_assert(kStaticScratchBytes % fa::kAlign == 0, "whole alignment units");
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device, looked up once per device with
// that device current (the host-side name of the array is not a device address).
uint8_t *static_scratch_address() {
    static std::mutex mu;
    static uint8_t *addr[128] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<uint8_t *>(p);
    }
    return addr[dev];
}

}  // namespace

extern "C" int fork_attn_decode_static_scratch(const void *q, const void *k_pages, const void *v_pages,
                                               const fa_plan *plan, void *out, float *lse, void *stream) {
    if (!plan || !q || !k_pages || !v_pages || !out || !lse) return FA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(lse, 16))
        return FA_ERR_ALIGN;
    const size_t plan_bytes = size_t(plan->lay.total);  // a multiple of 256
    const size_t scratch = size_t(fa::scratch_bytes(plan->partial_rows));
    if (plan_bytes + scratch > kStaticScratchBytes) return FA_ERR_SCRATCH_LIMIT;
    int rc = set_smem_attr();
    if (rc != FA_OK) return rc;
    uint8_t *base = static_scratch_address();
    if (!base) return FA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the copy brings the plan arrays and a zero error word; partial rows need no clearing
    // because every one of them is written before the merge reads it
    if (cudaMemcpyAsync(base, plan->blob.data(), plan_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return FA_ERR_CUDA;
    fa::DecodeParams p;
    rc = fill_params(plan, q, k_pages, v_pages, out, lse, scratch ? base + plan_bytes : nullptr, p);
    if (rc != FA_OK) return rc;
    const fa::Layout &L = plan->lay;
    p.chunk_pages = reinterpret_cast<const int32_t *>(base + L.chunk_pages);
    p.chunks = reinterpret_cast<const fa::Chunk *>(base + L.chunks);
    p.items = reinterpret_cast<const fa::Item *>(base + L.items_rows);
    p.items_tc = reinterpret_cast<const fa::Item *>(base + L.items_tc);
    p.items_r8 = reinterpret_cast<const fa::Item *>(base + L.items_r8);
    p.rows = reinterpret_cast<const fa::RowRec *>(base + L.rows);
    p.branches = reinterpret_cast<const fa::Branch *>(base + L.branches);
    p.q_merge = reinterpret_cast<const fa::QMerge *>(base + L.q_merge);
    p.merge_bases = reinterpret_cast<const int32_t *>(base + L.merge_bases);
    p.merge_lpos = reinterpret_cast<const int32_t *>(base + L.merge_lpos);
    p.mask_words = reinterpret_cast<const uint32_t *>(base + L.mask_words);
    p.err = reinterpret_cast<int32_t *>(base);
    plan->err_word = p.err;  // fork_attn_check reads this call's error word
    return launch_all(p, plan, st, nullptr, true);  // nothing is created here
}

extern "C" int fork_attn_merge_parts(const float *part_out, const float *part_lse, int32_t n_parts, int64_t rows,
                                     void *out, int32_t out_dtype, float *lse, void *stream) {
    if (!part_out || !part_lse || !out || !lse) return FA_ERR_NULL;
    if (n_parts < 1 || rows < 0 || (out_dtype != FA_BF16 && out_dtype != FA_F32)) return FA_ERR_INVALID;
    if (!aligned(part_out, 16) || !aligned(out, 16) || !aligned(part_lse, 4) || !aligned(lse, 4)) return FA_ERR_ALIGN;
    if (rows == 0) return FA_OK;
    const int64_t blocks = (rows * 32 + fa::mergek::kThreads - 1) / fa::mergek::kThreads;
    if (blocks > INT32_MAX) return FA_ERR_INVALID;
    fa::mergek::merge_parts_kernel<<<unsigned(blocks), fa::mergek::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        part_out, part_lse, n_parts, rows, out, out_dtype, lse);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" int fork_attn_score_lse(const void *q, const void *k_pages, const fa_plan *plan, float *lse, void *stream) {
    if (!plan || !q || !k_pages || !lse) return FA_ERR_NULL;
    if (!plan->representatives) return FA_ERR_INVALID;
    if (!plan->uploaded) return FA_ERR_NOT_UPLOADED;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(lse, 16)) return FA_ERR_ALIGN;
    int rc = set_smem_attr();
    if (rc != FA_OK) return rc;
    fa::DecodeParams p;
    // V is never read: its tensor maps are encoded over the K pages
    rc = fill_params(plan, q, k_pages, k_pages, nullptr, lse, plan->dev_scratch, p);
    if (rc != FA_OK) return rc;
    if (p.n_items > 0 || p.n_items_r8 > 0) return FA_ERR_INVALID;  // representative plans run on tcgen05 only
    p.lse_only = 1;
    plan->err_word = p.err;
    return launch_all(p, plan, static_cast<cudaStream_t>(stream), nullptr, true);
}
