// noalloc.cu -- dsv4_sparse_mla_decode_noalloc: the decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at decode time: code that runs inside a
// captured or replayed pipeline whose memory was fixed up front, plug-ins whose host
// framework owns every allocation, or environments where cudaMalloc is not allowed
// between set-up and shutdown.  This entry point takes the decode's scratch (the cache
// slots of the keys past each split's first two blocks) from one static device array
// compiled into the library instead of a workspace argument.
// The array is kNoAllocScratchBytes (32 MiB) and exists on every GPU that loads the
// library until the process exits.
#include <mutex>

#include "../../include/dsv4.h"
#include "internal.h"

namespace dsv4 {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;

// The scratch array.  In host code this name only stands for the symbol: its device
// address comes from cudaGetSymbolAddress (once per device, below).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device; looked up on the first
// call per device (that first call should come before any stream capture).
cudaError_t scratch_address(void **ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace dsv4

extern "C" DSV4_API dsv4_status dsv4_sparse_mla_decode_noalloc(
    const void *q, int64_t q_token_stride, const void *kv_cache, int32_t num_blocks, int32_t page_block,
    const int32_t *block_table, int64_t bt_stride, int32_t max_blocks, int32_t num_reqs, const int32_t *req_idx,
    const int32_t *topk_idx, int64_t topk_stride, int32_t topk_width, const int32_t *topk_lens,
    const int32_t *seq_lens, int32_t num_tokens, int32_t num_heads, int32_t window, const float *sink,
    float softmax_scale, void *out, float *lse, dsv4_stream_t stream)
{
    if (num_tokens == 0)
        return dsv4_sparse_mla_decode(q, q_token_stride, kv_cache, num_blocks, page_block, block_table, bt_stride,
                                      max_blocks, num_reqs, req_idx, topk_idx, topk_stride, topk_width, topk_lens,
                                      seq_lens, num_tokens, num_heads, window, sink, softmax_scale, out, lse, nullptr,
                                      0, stream);
    void *scratch = nullptr;
    if (dsv4::scratch_address(&scratch) != cudaSuccess)
        return DSV4_ERR_CUDA;
    const size_t need = dsv4_sparse_mla_decode_workspace_size(num_tokens, num_heads, topk_width, window);
    if (need == 0)   // the arguments themselves are rejected: let the decode say how
        return dsv4_sparse_mla_decode(q, q_token_stride, kv_cache, num_blocks, page_block, block_table, bt_stride,
                                      max_blocks, num_reqs, req_idx, topk_idx, topk_stride, topk_width, topk_lens,
                                      seq_lens, num_tokens, num_heads, window, sink, softmax_scale, out, lse, scratch,
                                      dsv4::kNoAllocScratchBytes, stream);
    if (need > dsv4::kNoAllocScratchBytes)
        return DSV4_ERR_UNSUPPORTED;   // this batch needs more scratch than the static array holds
    // Every decode scratch region is fully written before it is read, so stale contents
    // from a previous call need no clearing.
    return dsv4_sparse_mla_decode(q, q_token_stride, kv_cache, num_blocks, page_block, block_table, bt_stride,
                                  max_blocks, num_reqs, req_idx, topk_idx, topk_stride, topk_width, topk_lens, seq_lens,
                                  num_tokens, num_heads, window, sink, softmax_scale, out, lse, scratch,
                                  dsv4::kNoAllocScratchBytes, stream);
}
