// api.cu -- the C ABI declared in include/dsv4.h: argument validation, the work plan,
// and the launches on the caller's stream.  No device memory is allocated here; all
// scratch lives in the caller's workspace.
#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>

#include "../../include/dsv4.h"
#include "internal.h"

namespace dsv4 {
namespace {

// Sticky per-device status word (bits kStatusBadIndex / kStatusTimeout).
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_status_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];

// Device address of the status word and the SM count of the current device.
cudaError_t device_info(unsigned **status, int *sms)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_status_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_status_word);
        if (e != cudaSuccess)
            return e;
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        g_sm_count[dev] = n;
        g_status_ptr[dev] = static_cast<unsigned *>(ptr);
    }
    if (status)
        *status = g_status_ptr[dev];
    if (sms)
        *sms = g_sm_count[dev];
    return cudaSuccess;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int kMaxWindow = 1 << 24;

// mtp_union: the plan of an MTP union call (units are a request's two tokens x 32 heads, over the
// union of the two combined lists)
bool make_plan(int num_tokens, int num_heads, int topk_width, int window, int sms, Plan *pl, bool mtp_union = false)
{
    if (num_tokens < 0 || topk_width < 0 || topk_width > kMaxTopkWidth || window < 0 || window > kMaxWindow)
        return false;
    if (num_heads != 16 && num_heads != 32 && num_heads != 64 && num_heads != 128)
        return false;
    if (mtp_union && (num_heads == 16 || num_tokens % 2 != 0))
        return false;
    Plan p{};
    // One tensor-core kernel, 64 heads per CTA (a group of 16 or 32 heads runs as a 64-head group
    // whose missing heads have zero queries and are never written), 128-key blocks, one CTA per SM.
    // Union calls: 32 heads of each of the request's two tokens per CTA.
    p.heads_per_group = mtp_union ? 32 : 64;
    p.groups = (num_heads + p.heads_per_group - 1) / p.heads_per_group;
    p.list_w = topk_width + window;
    p.cw = mtp_union ? 2 * p.list_w : p.list_w;
    const int tile = decode_tc_block_keys();
    const int units_t = mtp_union ? num_tokens / 2 : num_tokens;
    const long long units0 = (long long)(units_t > 0 ? units_t : 1) * p.groups;
    // the splits of a token form one thread-block cluster (<= 8 CTAs)
    const int split_cap = decode_tc_max_splits();
    const int max_splits = std::max(1, std::min(split_cap, (p.cw + tile - 1) / tile));
    // Choose the split count minimising (waves x time per worker): a 128-key block costs its
    // matrix products and softmax whatever its fill, the gather scales with the keys (chunks are
    // multiples of 16 keys), plus the prologue and, when split, the cluster merge.
    const int gran = 16;
    double best = 1e300;
    int best_chunk = std::max(gran, (p.cw + gran - 1) / gran * gran);
    for (int s = 1; s <= max_splits; ++s) {
        int chunk = (p.cw + s - 1) / s;
        chunk = std::max(gran, (chunk + gran - 1) / gran * gran);
        const int s_eff = std::max(1, (p.cw + chunk - 1) / chunk);
        if (s_eff > split_cap)
            continue;
        const long long units = units0 * s_eff;
        const int resident = decode_tc_resident_ctas(s_eff);
        if (resident <= 0)
            continue;
        const long long waves = (units + resident - 1) / resident;
        const int blocks = (chunk + tile - 1) / tile;
        const double per_worker = blocks + 0.25 * chunk / tile + 0.5 + (s_eff > 1 ? 0.5 : 0.0);
        const double cost = (double)waves * per_worker;
        if (cost < best - 1e-9) {
            best = cost;
            best_chunk = chunk;
        }
    }
    p.chunk = best_chunk;
    p.splits = std::max(1, (p.cw + p.chunk - 1) / p.chunk);
    p.combine_table_bits = decode_tc_table_bits(topk_width);

    size_t off = 0;
    p.off_combined = off;
    off = align_up(off + sizeof(int32_t) * (size_t)num_tokens * (size_t)p.cw, 256);
    p.off_order = off;   // the units' launch order, when the call needs one
    off = align_up(off + sizeof(int32_t) * (size_t)num_tokens * (size_t)p.groups, 256);
    if (mtp_union) {
        p.off_lists = off;
        off = align_up(off + sizeof(int32_t) * (size_t)num_tokens * (size_t)p.list_w, 256);
        p.off_lens = off;
        off = align_up(off + sizeof(int32_t) * (size_t)num_tokens, 256);
        p.off_ulist = off;
        off = align_up(off + sizeof(int32_t) * (size_t)(num_tokens / 2) * (size_t)p.cw, 256);
        p.off_ulen = off;
        off = align_up(off + sizeof(int32_t) * (size_t)(num_tokens / 2), 256);
    }
    p.total = std::max<size_t>(off, 256);
    *pl = p;
    return true;
}

dsv4_status check_combine_args(const int32_t *topk_idx, int64_t topk_stride, int32_t topk_width,
                               const int32_t *seq_lens, int32_t num_tokens, int32_t window)
{
    if (num_tokens < 0 || topk_width < 0 || window < 0 || window > kMaxWindow)
        return DSV4_ERR_INVALID_ARG;
    if (topk_width > kMaxTopkWidth)
        return DSV4_ERR_UNSUPPORTED;
    if (num_tokens > 0) {
        if (seq_lens == nullptr)
            return DSV4_ERR_INVALID_ARG;
        if (topk_width > 0 && (topk_idx == nullptr || topk_stride < topk_width))
            return DSV4_ERR_INVALID_ARG;
    }
    return DSV4_OK;
}

int g_attr_bytes[kMaxDevices][kAttrSlots];

}  // namespace

cudaError_t set_smem_once(const void *kernel, int bytes, AttrSlot slot)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_attr_bytes[dev][slot] >= bytes)
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        g_attr_bytes[dev][slot] = bytes;
    return e;
}

}  // namespace dsv4

using namespace dsv4;

extern "C" DSV4_API dsv4_status dsv4_combine_topk_swa_indices(const int32_t *topk_idx, int64_t topk_stride,
                                                     int32_t topk_width, const int32_t *topk_lens,
                                                     const int32_t *seq_lens, int32_t num_tokens, int32_t window,
                                                     int32_t *combined, int64_t combined_stride,
                                                     int32_t combined_width, int32_t *combined_lens,
                                                     dsv4_stream_t stream)
{
    dsv4_status st = check_combine_args(topk_idx, topk_stride, topk_width, seq_lens, num_tokens, window);
    if (st != DSV4_OK)
        return st;
    if ((long long)combined_width < (long long)topk_width + window)
        return DSV4_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return DSV4_OK;
    if (combined == nullptr || combined_lens == nullptr || combined_stride < combined_width)
        return DSV4_ERR_INVALID_ARG;
    cudaError_t e = launch_combine(topk_idx, topk_stride, topk_width, topk_lens, seq_lens, num_tokens, window,
                                   combined, combined_stride, combined_width, combined_lens,
                                   combine_table_bits(topk_width), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

extern "C" DSV4_API dsv4_status dsv4_combine_topk_swa_indices_compressed(
    const int32_t *topk_idx, int64_t topk_stride, int32_t topk_width, const int32_t *query_start_loc,
    const int32_t *seq_lens, const int32_t *gather_lens, int32_t num_reqs, int32_t num_tokens, int32_t region_stride,
    int32_t compressed_len, int32_t top_k, int32_t compress_ratio, int32_t window, int32_t *combined,
    int64_t combined_stride, int32_t combined_width, int32_t *combined_lens, dsv4_stream_t stream)
{
    if (num_reqs < 0 || num_tokens < 0 || topk_width < 0 || top_k < 0 || top_k > topk_width || compress_ratio < 1 ||
        window < 0 || window > kMaxWindow || region_stride < 0 || compressed_len < 0)
        return DSV4_ERR_INVALID_ARG;
    if (topk_width > kMaxTopkWidth)
        return DSV4_ERR_UNSUPPORTED;
    if ((long long)region_stride * num_reqs > INT_MAX || (long long)combined_width < (long long)top_k + window)
        return DSV4_ERR_INVALID_ARG;
    if (num_reqs == 0 || num_tokens == 0)
        return DSV4_OK;
    if (query_start_loc == nullptr || seq_lens == nullptr || gather_lens == nullptr || combined == nullptr ||
        combined_lens == nullptr || combined_stride < combined_width)
        return DSV4_ERR_INVALID_ARG;
    if (top_k > 0 && (topk_idx == nullptr || topk_stride < topk_width))
        return DSV4_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    if (device_info(&status, nullptr) != cudaSuccess)
        return DSV4_ERR_CUDA;
    cudaError_t e = launch_combine_compressed(topk_idx, topk_stride, query_start_loc, seq_lens, gather_lens, num_reqs,
                                              num_tokens, region_stride, compressed_len, top_k, compress_ratio, window,
                                              combined, combined_stride, combined_width, combined_lens, status,
                                              reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

extern "C" DSV4_API dsv4_status dsv4_selftest_wait_timeout(int64_t cycles, dsv4_stream_t stream)
{
    if (cycles < 1 || cycles > (int64_t)1 << 31)
        return DSV4_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    if (device_info(&status, nullptr) != cudaSuccess)
        return DSV4_ERR_CUDA;
    return launch_wait_selftest((long long)cycles, status, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DSV4_OK
               : DSV4_ERR_CUDA;
}

extern "C" DSV4_API dsv4_status dsv4_qnorm_rope_kv_insert(
    const void *q, int64_t q_token_stride, void *q_out, int64_t q_out_token_stride, int32_t num_tokens,
    int32_t num_heads, const float *q_norm_weight, float eps, const void *kv, int64_t kv_token_stride,
    const int64_t *positions, const int64_t *slot_mapping, const float *cos_sin_cache, int32_t max_position,
    void *kv_cache, int64_t num_slots, dsv4_stream_t stream)
{
    if (num_tokens < 0 || num_heads < 1 || num_heads > 128 || !(eps >= 0.f) || !std::isfinite(eps) ||
        max_position < 1 || num_slots < 0)
        return DSV4_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return DSV4_OK;
    const int64_t row = (int64_t)num_heads * kDim;
    auto odd = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) != 0; };
    if (q == nullptr || q_out == nullptr || kv == nullptr || positions == nullptr || slot_mapping == nullptr ||
        cos_sin_cache == nullptr || (num_slots > 0 && kv_cache == nullptr) || q_token_stride < row ||
        q_out_token_stride < row || kv_token_stride < kDim || (q_token_stride | q_out_token_stride | kv_token_stride) & 1 ||
        odd(q) || odd(q_out) || odd(kv) || (num_slots > 0 && (reinterpret_cast<uintptr_t>(kv_cache) & 15u) != 0))
        return DSV4_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    if (device_info(&status, nullptr) != cudaSuccess)
        return DSV4_ERR_CUDA;
    cudaError_t e = launch_qnorm_rope_kv_insert(q, q_token_stride, q_out, q_out_token_stride, num_tokens, num_heads,
                                                q_norm_weight, eps, kv, kv_token_stride, positions, slot_mapping,
                                                cos_sin_cache, max_position, kv_cache, num_slots, status,
                                                reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

extern "C" DSV4_API dsv4_status dsv4_topk_select(const float *scores, int64_t score_stride, int32_t score_width,
                                                 const int32_t *num_cand, int32_t num_tokens, int32_t top_k,
                                                 int32_t *topk_idx, int64_t topk_stride, int32_t *topk_lens,
                                                 dsv4_stream_t stream)
{
    if (num_tokens < 0 || top_k < 1 || score_width < 0)
        return DSV4_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return DSV4_OK;
    if (num_cand == nullptr || topk_idx == nullptr || topk_stride < top_k ||
        (score_width > 0 && (scores == nullptr || score_stride < score_width)))
        return DSV4_ERR_INVALID_ARG;
    int sms = 0;
    if (device_info(nullptr, &sms) != cudaSuccess)
        return DSV4_ERR_CUDA;
    cudaError_t e = launch_topk_select(scores, score_stride, score_width, num_cand, num_tokens, top_k, topk_idx,
                                       topk_stride, topk_lens, topk_cluster_size(num_tokens, score_width, sms),
                                       reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

extern "C" DSV4_API size_t dsv4_sparse_mla_decode_workspace_size(int32_t num_tokens, int32_t num_heads, int32_t topk_width,
                                                        int32_t window)
{
    int sms = 0;
    if (device_info(nullptr, &sms) != cudaSuccess)
        return 0;
    Plan pl;
    if (!make_plan(num_tokens, num_heads, topk_width, window, sms, &pl))
        return 0;
    return pl.total;
}

namespace {

// The decode call, with an optional record of each token's combined list (positions in list
// order and the list length) written by the decode kernel itself.
dsv4_status decode_call(const void *q, int64_t q_token_stride, const void *kv_cache, int32_t num_blocks,
                        int32_t page_block, const int32_t *block_table, int64_t bt_stride, int32_t max_blocks,
                        int32_t num_reqs, const int32_t *req_idx, const int32_t *topk_idx, int64_t topk_stride,
                        int32_t topk_width, const int32_t *topk_lens, const int32_t *seq_lens, int32_t num_tokens,
                        int32_t num_heads, int32_t window, const float *sink, float softmax_scale, void *out,
                        float *lse, void *workspace, size_t workspace_bytes, int32_t *trace, int64_t trace_stride,
                        int32_t *trace_lens, dsv4_stream_t stream, bool mtp_union = false)
{
    dsv4_status st = check_combine_args(topk_idx, topk_stride, topk_width, seq_lens, num_tokens, window);
    if (st != DSV4_OK)
        return st;
    if (num_heads != 16 && num_heads != 32 && num_heads != 64 && num_heads != 128)
        return DSV4_ERR_UNSUPPORTED;
    if (mtp_union && num_heads == 16)
        return DSV4_ERR_UNSUPPORTED;
    if (mtp_union && (num_tokens % 2 != 0 || req_idx == nullptr))
        return DSV4_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale) || softmax_scale < 0.f)   // the kernel's running max is taken on raw dot products
        return DSV4_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return DSV4_OK;
    if (q == nullptr || kv_cache == nullptr || block_table == nullptr || out == nullptr || workspace == nullptr)
        return DSV4_ERR_INVALID_ARG;
    if (q_token_stride < (int64_t)num_heads * kDim || q_token_stride % 8 != 0)
        return DSV4_ERR_INVALID_ARG;
    if (num_blocks <= 0 || page_block <= 0 || max_blocks <= 0 || num_reqs <= 0 || bt_stride < max_blocks)
        return DSV4_ERR_INVALID_ARG;
    if (req_idx == nullptr && num_reqs < num_tokens)
        return DSV4_ERR_INVALID_ARG;
    if ((long long)max_blocks * page_block > INT_MAX || (long long)num_blocks * page_block > INT_MAX)
        return DSV4_ERR_INVALID_ARG;
    if (mtp_union && (long long)num_blocks * page_block >= (1LL << 29))   // cache slots carry two mask bits above them
        return DSV4_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(workspace, 256))
        return DSV4_ERR_INVALID_ARG;

    unsigned *status = nullptr;
    int sms = 0;
    if (device_info(&status, &sms) != cudaSuccess)
        return DSV4_ERR_CUDA;
    Plan pl;
    if (!make_plan(num_tokens, num_heads, topk_width, window, sms, &pl, mtp_union))
        return DSV4_ERR_INVALID_ARG;
    if (workspace_bytes < pl.total)
        return DSV4_ERR_INVALID_ARG;

    char *ws = static_cast<char *>(workspace);
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (mtp_union) {   // every token's combined list, then each request's union list
        int32_t *lists = reinterpret_cast<int32_t *>(ws + pl.off_lists);
        int32_t *lens = reinterpret_cast<int32_t *>(ws + pl.off_lens);
        cudaError_t e = launch_combine(topk_idx, topk_stride, topk_width, topk_lens, seq_lens, num_tokens, window, lists,
                                       pl.list_w, pl.list_w, lens, combine_table_bits(topk_width), cs);
        if (e == cudaSuccess)
            e = launch_mtp_union(lists, pl.list_w, lens, seq_lens, window, req_idx, num_tokens / 2,
                                 reinterpret_cast<int32_t *>(ws + pl.off_ulist), pl.cw,
                                 reinterpret_cast<int32_t *>(ws + pl.off_ulen), topk_width, status, cs);
        if (e != cudaSuccess)
            return DSV4_ERR_CUDA;
    }
    DecodeParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.q_token_stride = q_token_stride;
    p.kv = static_cast<const uint8_t *>(kv_cache);
    p.num_blocks = num_blocks;
    p.page = page_block;
    p.block_table = block_table;
    p.bt_stride = bt_stride;
    p.max_blocks = max_blocks;
    p.num_reqs = num_reqs;
    p.req_idx = req_idx;
    p.combined = reinterpret_cast<int32_t *>(ws + pl.off_combined);
    p.cw = pl.cw;
    p.num_tokens = num_tokens;
    p.num_heads = num_heads;
    p.sink = sink;
    p.scale = softmax_scale;
    p.out = static_cast<uint16_t *>(out);
    p.lse = lse;
    p.groups = pl.groups;
    p.heads_per_group = pl.heads_per_group;
    p.splits = pl.splits;
    p.chunk = pl.chunk;
    p.status = status;
    p.topk = topk_idx;
    p.topk_stride = topk_stride;
    p.topk_width = topk_width;
    p.topk_lens = topk_lens;
    p.seq_lens = seq_lens;
    p.window = window;
    p.table_bits = pl.combine_table_bits;
    p.trace = trace;
    p.trace_stride = trace_stride;
    p.trace_lens = trace_lens;
    // Lists of different lengths over more (token, head group) units than multiprocessors: the
    // units start longest first (a one-CTA ordering kernel runs ahead of the decode).  Equal
    // lengths gain nothing from it.
    // (union calls: the union lists' lengths vary with the overlap of a request's two lists)
    p.order = nullptr;
    if (mtp_union ? (long long)(num_tokens / 2) * pl.groups > sms
                  : topk_lens != nullptr && (long long)num_tokens * pl.groups > sms)
        p.order = reinterpret_cast<int32_t *>(ws + pl.off_order);
    p.ulist = nullptr;
    p.ulist_stride = 0;
    p.ulen = nullptr;
    if (mtp_union) {
        p.ulist = reinterpret_cast<const int32_t *>(ws + pl.off_ulist);
        p.ulist_stride = pl.cw;
        p.ulen = reinterpret_cast<const int32_t *>(ws + pl.off_ulen);
    }

    // one launch: the kernel combines, decodes and merges its splits
    const cudaError_t e = launch_decode_tc(p, cs);
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

}  // namespace

extern "C" DSV4_API dsv4_status dsv4_sparse_mla_decode(const void *q, int64_t q_token_stride, const void *kv_cache,
                                              int32_t num_blocks, int32_t page_block, const int32_t *block_table,
                                              int64_t bt_stride, int32_t max_blocks, int32_t num_reqs,
                                              const int32_t *req_idx, const int32_t *topk_idx, int64_t topk_stride,
                                              int32_t topk_width, const int32_t *topk_lens, const int32_t *seq_lens,
                                              int32_t num_tokens, int32_t num_heads, int32_t window,
                                              const float *sink, float softmax_scale, void *out, float *lse,
                                              void *workspace, size_t workspace_bytes, dsv4_stream_t stream)
{
    return decode_call(q, q_token_stride, kv_cache, num_blocks, page_block, block_table, bt_stride, max_blocks,
                       num_reqs, req_idx, topk_idx, topk_stride, topk_width, topk_lens, seq_lens, num_tokens,
                       num_heads, window, sink, softmax_scale, out, lse, workspace, workspace_bytes, nullptr, 0,
                       nullptr, stream);
}

extern "C" DSV4_API dsv4_status dsv4_sparse_mla_decode_trace(
    const void *q, int64_t q_token_stride, const void *kv_cache, int32_t num_blocks, int32_t page_block,
    const int32_t *block_table, int64_t bt_stride, int32_t max_blocks, int32_t num_reqs, const int32_t *req_idx,
    const int32_t *topk_idx, int64_t topk_stride, int32_t topk_width, const int32_t *topk_lens,
    const int32_t *seq_lens, int32_t num_tokens, int32_t num_heads, int32_t window, const float *sink,
    float softmax_scale, void *out, float *lse, void *workspace, size_t workspace_bytes, int32_t *combined,
    int64_t combined_stride, int32_t combined_width, int32_t *combined_lens, dsv4_stream_t stream)
{
    if (num_tokens > 0 && (combined == nullptr || combined_lens == nullptr || combined_stride < combined_width ||
                           (long long)combined_width < (long long)topk_width + window))
        return DSV4_ERR_INVALID_ARG;
    return decode_call(q, q_token_stride, kv_cache, num_blocks, page_block, block_table, bt_stride, max_blocks,
                       num_reqs, req_idx, topk_idx, topk_stride, topk_width, topk_lens, seq_lens, num_tokens,
                       num_heads, window, sink, softmax_scale, out, lse, workspace, workspace_bytes, combined,
                       combined_stride, combined_lens, stream);
}

extern "C" DSV4_API dsv4_status dsv4_sparse_mla_decode_mtp_union(
    const void *q, int64_t q_token_stride, const void *kv_cache, int32_t num_blocks, int32_t page_block,
    const int32_t *block_table, int64_t bt_stride, int32_t max_blocks, int32_t num_reqs, const int32_t *req_idx,
    const int32_t *topk_idx, int64_t topk_stride, int32_t topk_width, const int32_t *topk_lens,
    const int32_t *seq_lens, int32_t num_tokens, int32_t num_heads, int32_t window, const float *sink,
    float softmax_scale, void *out, float *lse, void *workspace, size_t workspace_bytes, dsv4_stream_t stream)
{
    return decode_call(q, q_token_stride, kv_cache, num_blocks, page_block, block_table, bt_stride, max_blocks,
                       num_reqs, req_idx, topk_idx, topk_stride, topk_width, topk_lens, seq_lens, num_tokens,
                       num_heads, window, sink, softmax_scale, out, lse, workspace, workspace_bytes, nullptr, 0,
                       nullptr, stream, true);
}

extern "C" DSV4_API size_t dsv4_sparse_mla_decode_mtp_union_workspace_size(int32_t num_tokens, int32_t num_heads,
                                                                          int32_t topk_width, int32_t window)
{
    int sms = 0;
    if (device_info(nullptr, &sms) != cudaSuccess)
        return 0;
    Plan pl;
    if (!make_plan(num_tokens, num_heads, topk_width, window, sms, &pl, true))
        return 0;
    return pl.total;
}

extern "C" DSV4_API dsv4_status dsv4_get_device_status(dsv4_stream_t stream)
{
    unsigned *status = nullptr;
    if (device_info(&status, nullptr) != cudaSuccess)
        return DSV4_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return DSV4_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return DSV4_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpy(status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return DSV4_ERR_CUDA;
    if (word & kStatusBadIndex)
        return DSV4_ERR_BAD_INDEX;
    if (word & kStatusTimeout)
        return DSV4_ERR_TIMEOUT;
    return DSV4_OK;
}
