// internal.h -- launch interface between the C ABI (api.cu) and the kernel files.
// Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dsv4 {

// Cache entry layout (656 bytes): 512 E4M3 latent codes, 64 BF16 rope values,
// 4 UE8M0 scale bytes, 12 bytes of padding.
constexpr int kEntryBytes = 656;
constexpr int kLatent = 512;
constexpr int kRope = 64;
constexpr int kDim = 576;
constexpr int kRopeOffset = 512;
constexpr int kScaleOffset = 640;
constexpr int kScaleBlock = 128;

// Bits of the sticky device status word.
constexpr unsigned kStatusBadIndex = 1u;
constexpr unsigned kStatusTimeout = 2u;

constexpr int kMaxTopkWidth = 8192;

// Work decomposition of one decode call; computed on the host from the call's
// sizes and the device's SM count, identically by the workspace-size query.
struct Plan {
    int heads_per_group;   // heads handled by one worker (64: a group of 16 or 32 heads is padded)
    int groups;            // ceil(num_heads / heads_per_group)
    int splits;            // workers sharing one (token, head group): one thread-block cluster
    int chunk;             // combined-list entries per split
    int cw;                // row width of the workspace's slot rows (topk_width + window)
    int combine_table_bits;
    size_t off_combined, off_order, total;
    // MTP union calls: the tokens' combined lists [T, list_w] and lengths, the requests' union
    // lists [T / 2, cw] and lengths
    int list_w;
    size_t off_lists, off_lens, off_ulist, off_ulen;
};

struct DecodeParams {
    const uint16_t *q;
    int64_t q_token_stride;
    const uint8_t *kv;
    int32_t num_blocks;
    int32_t page;
    const int32_t *block_table;
    int64_t bt_stride;
    int32_t max_blocks;
    int32_t num_reqs;
    const int32_t *req_idx;
    int32_t *combined;         // [T, cw]: cache slots of the keys past each split's first two blocks
    int32_t cw;
    int32_t num_tokens;
    int32_t num_heads;
    const float *sink;
    float scale;
    uint16_t *out;             // BF16 [T, H, 512]
    float *lse;                // [T, H] or null
    int32_t groups;
    int32_t heads_per_group;
    int32_t splits;
    int32_t chunk;
    unsigned *status;
    // the combine's inputs: the kernel combines in its prologue
    const int32_t *topk;
    int64_t topk_stride;
    int32_t topk_width;
    const int32_t *topk_lens;
    const int32_t *seq_lens;
    int32_t window;
    int32_t table_bits;
    // optional record of the combined list each token's CTAs used (logical positions in
    // list order, and the list length); null in ordinary calls
    int32_t *trace;
    int64_t trace_stride;
    int32_t *trace_lens;
    // launch order of the (token, head group) units, longest estimated list first, written by
    // the ordering kernel ahead of the decode; null: index order
    int32_t *order;
    // MTP union calls: the two tokens of request r (2r, 2r + 1) share one CTA per 32 heads and the
    // union list of row r (positions with bit 29 set for token 2r's keys, bit 30 for token
    // 2r + 1's), ulen[r] entries; null in other calls
    const int32_t *ulist;
    int64_t ulist_stride;
    const int32_t *ulen;
};

// Raises a kernel's dynamic shared-memory limit to at least `bytes`, once per
// (device, kernel slot); later calls with no larger size touch no CUDA state, so a
// call made after the first one on a device is safe inside stream capture.
enum AttrSlot { kAttrCombine = 0, kAttrTc, kAttrTcLong, kAttrTcUnion, kAttrTcUnionLong, kAttrUnion, kAttrTopk,
                kAttrTopkCluster, kAttrSlots };
cudaError_t set_smem_once(const void *kernel, int bytes, AttrSlot slot);

int combine_table_bits(int topk_width);
size_t combine_smem_bytes(int table_bits, int topk_width);
// the union lists of MTP requests (tokens 2r, 2r + 1) from the tokens' combined lists
cudaError_t launch_mtp_union(const int32_t *lists, int64_t lstride, const int32_t *lens, const int32_t *seq_lens,
                             int window, const int32_t *req_idx, int num_reqs, int32_t *ulist, int64_t ustride,
                             int32_t *ulen, int topk_width, unsigned *status, cudaStream_t stream);
cudaError_t launch_combine(const int32_t *topk, int64_t topk_stride, int topk_width, const int32_t *topk_lens,
                           const int32_t *seq_lens, int num_tokens, int window, int32_t *combined,
                           int64_t combined_stride, int combined_width, int32_t *combined_lens, int table_bits,
                           cudaStream_t stream);

cudaError_t launch_combine_compressed(const int32_t *topk, int64_t topk_stride, const int32_t *qsl,
                                      const int32_t *seq_lens, const int32_t *gather_lens, int num_reqs,
                                      int num_tokens, int region_stride, int compressed_len, int top_k,
                                      int compress_ratio, int window, int32_t *combined, int64_t combined_stride,
                                      int combined_width, int32_t *combined_lens, unsigned *status,
                                      cudaStream_t stream);

// Fused Q RMSNorm + GPT-J RoPE + FP8/UE8M0 KV-cache insert (strides in BF16 elements, even).
cudaError_t launch_qnorm_rope_kv_insert(const void *q, int64_t q_stride, void *q_out, int64_t q_out_stride,
                                        int num_tokens, int num_heads, const float *norm_w, float eps,
                                        const void *kv, int64_t kv_stride, const int64_t *positions,
                                        const int64_t *slots, const float *cos_sin, int max_pos, void *cache,
                                        int64_t num_slots, unsigned *status, cudaStream_t stream);

// Top-k selection: CTAs per token row (a thread-block cluster when > 1), and the launch.
int topk_cluster_size(int num_tokens, int width, int sms);
cudaError_t launch_topk_select(const float *scores, int64_t score_stride, int width, const int32_t *num_cand,
                               int num_tokens, int top_k, int32_t *out, int64_t out_stride, int32_t *lens,
                               int cluster, cudaStream_t stream);

cudaError_t launch_decode_tc(const DecodeParams &p, cudaStream_t stream);
int decode_tc_block_keys();
cudaError_t launch_wait_selftest(long long limit, unsigned *status, cudaStream_t stream);
int decode_tc_table_bits(int topk_width);   // combine hash set of the tensor-core kernel: 2^bits 8-byte slots
int decode_tc_max_splits();
int decode_tc_resident_ctas(int splits);

}  // namespace dsv4
