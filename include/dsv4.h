/*
 * dsv4.h -- C ABI of the GB300 (sm_103a) DeepSeek-V4 sparse-MLA decode library.
 *
 * One decode step for a batch of query tokens over a paged FP8 KV cache:
 *   1. per token, merge the top-k selected positions with the sliding window
 *      (SWA), dropping invalid, non-causal, in-window and repeated entries;
 *   2. translate each logical position to a physical cache slot through the
 *      block table and gather + dequantise the 656-byte entries;
 *   3. MQA attention of all heads over those keys: logits over the 576-d key
 *      (512 latent + 64 RoPE), values = the 512-d latent, an optional per-head
 *      sink logit in the softmax normaliser;
 *   4. BF16 output [T, H, 512] and a natural-log LSE per (token, head).
 *
 * Sources of the operations (vLLM pull-request summaries):
 *   - "[ROCm] [DSv4] [Perf] Support DeepSeek v4 MTP" (vllm #43385), section
 *     "关键源码片段 / rocm.py": _combine_topk_swa_indices_kernel / combine_topk_swa_indices
 *     (top-k entries then the window [pos - swa_len + 1, pos], swa_len = min(pos + 1, W),
 *     validity test, combined_lens = topk part + swa part, 128-aligned padded width).
 *   - "feat: add DeepSeek-V4 XPU attention decode path" (vllm #42953), section
 *     "xpu_sparse_decode_fp8.py": _dequant_gather_slots_kernel (slot -> block / offset,
 *     value = e4m3 * exp2(ue8m0 - 127), negative slot -> no contribution) and
 *     xpu_sparse_decode_fp8 / triton_bf16_mla_sparse_interface (sparse MLA over the
 *     gathered keys, with per-token top-k lengths).
 *   - "Enable DeepSeek V4 and GLM-5.1 on SM120" (vllm #43477), section
 *     "flashinfer_mla_sparse_sm120.py": forward_mqa converts per-request top-k indices to
 *     physical slots through the block table and writes output [T, h, kv_lora_rank = 512];
 *     "flashinfer_sparse.py": supports_sink.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers unless stated otherwise; the caller owns
 *     all memory.  The library never allocates device memory in a call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and never synchronise it.  Kernels run on the current CUDA device.
 *   - Argument errors are detected on the host and returned before anything is
 *     enqueued.  Errors that depend on device data (an out-of-range block-table entry,
 *     an out-of-range request index) do not stop the kernels: the offending key is left
 *     out of the result and a sticky per-device status word records the error; read it
 *     with dsv4_get_device_status().
 *   - All integer sizes and strides are in elements of the array's own type.
 *
 * KV-cache entry (656 bytes; entries are token-major inside a page, page stride
 * page_block * 656 bytes):
 *   [0, 512)    512 E4M3FN latent codes (OCP FP8: bias 7, max 448, S.1111.111 = NaN)
 *   [512, 640)  64 BF16 RoPE values, little-endian
 *   [640, 644)  4 UE8M0 scale bytes; byte b scales latent dims [128 b, 128 b + 128) by 2^(byte - 127)
 *   [644, 656)  padding (not read as data)
 * The key is k = [latent * scale, rope] (576 dims); the value is v = latent * scale (512 dims).
 */
#ifndef DSV4_H_
#define DSV4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DSV4_API __attribute__((visibility("default")))
#else
#define DSV4_API
#endif

struct CUstream_st;
/* Same type as cudaStream_t. */
typedef struct CUstream_st *dsv4_stream_t;

typedef enum dsv4_status {
    DSV4_OK = 0,
    DSV4_ERR_INVALID_ARG = 1,   /* bad pointer, size, stride, alignment or workspace size */
    DSV4_ERR_BAD_INDEX = 2,     /* device status only: a block-table or request index was out of range */
    DSV4_ERR_TIMEOUT = 3,       /* device status only: a bounded wait inside a kernel gave up */
    DSV4_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    DSV4_ERR_UNSUPPORTED = 5    /* valid request this build does not implement (e.g. num_heads) */
} dsv4_status;

/*
 * dsv4_combine_topk_swa_indices -- per-token index list: kept top-k entries, then the window.
 *
 * Source: vllm #43385 "[ROCm] [DSv4] [Perf] Support DeepSeek v4 MTP", section
 * "关键源码片段 / rocm.py", _combine_topk_swa_indices_kernel.  This library reads one
 * cache region for both parts, so (where the page's kernel indexes two disjoint regions)
 * it additionally drops top-k entries that the window already covers and repeats, and
 * compacts the kept entries.
 *
 * For token t with pos = seq_lens[t] - 1 and n = min(max(topk_lens[t], 0), topk_width)
 * (n = topk_width when topk_lens is NULL):
 *   window   = [max(0, pos - window + 1), pos]   (empty when pos < 0 or window == 0)
 *   kept     = topk_idx[t][i] for i < n, in order of i, when 0 <= value <= pos, value is
 *              not inside the window, and no earlier i' < i holds the same value
 *   combined[t][0 .. L)      = kept entries, then the window positions ascending
 *   combined[t][L .. width)  = -1
 *   combined_lens[t]         = L = |kept| + window length
 *
 * Arguments:
 *   topk_idx        int32 [num_tokens, topk_width], row stride topk_stride (>= topk_width);
 *                   may be NULL when topk_width == 0.
 *   topk_width      0 .. 8192.
 *   topk_lens       int32 [num_tokens] or NULL.
 *   seq_lens        int32 [num_tokens]: causal visible length of each token (its position + 1).
 *   num_tokens      >= 0 (0 enqueues nothing).
 *   window          >= 0.
 *   combined        int32 [num_tokens, combined_width], row stride combined_stride (>= combined_width).
 *   combined_width  >= topk_width + window (callers usually round up to a multiple of 128).
 *   combined_lens   int32 [num_tokens].
 * Returns DSV4_OK, DSV4_ERR_INVALID_ARG, DSV4_ERR_UNSUPPORTED (topk_width > 8192) or DSV4_ERR_CUDA.
 */
DSV4_API dsv4_status dsv4_combine_topk_swa_indices(const int32_t *topk_idx, int64_t topk_stride, int32_t topk_width,
                                          const int32_t *topk_lens, const int32_t *seq_lens, int32_t num_tokens,
                                          int32_t window, int32_t *combined, int64_t combined_stride,
                                          int32_t combined_width, int32_t *combined_lens, dsv4_stream_t stream);

/*
 * dsv4_combine_topk_swa_indices_compressed -- per-token index lists over a compressed region
 * plus the raw window, for batches of multi-token requests (prefill chunks, speculative verify).
 *
 * Source: vllm #43385 "[ROCm] [DSv4] [Perf] Support DeepSeek v4 MTP", section
 * "关键源码片段 / rocm.py", _combine_topk_swa_indices_kernel with COMPRESS_RATIO, gather_lens
 * and query_start_loc.  Request b owns a gathered region of region_stride (M) entries:
 * compressed_len (N) compressed entries, which top-k indexes, then the raw positions from
 * gather_start = seq_lens[b] - gather_lens[b] on.  Its tokens are rows
 * [query_start_loc[b] - query_start_loc[0], query_start_loc[b + 1] - query_start_loc[0]);
 * token i of a request with query_len tokens sits at pos = seq_lens[b] - query_len + i and gets
 *   topk_len = min((pos + 1) / compress_ratio, top_k)   (0 when pos + 1 <= 0)
 *   swa_len  = min(pos + 1, window)                      (0 when pos + 1 <= 0)
 *   combined[t][k]            = M*b + topk_idx[t][k] when 0 <= topk_idx[t][k] < N, else -1
 *                               (k < topk_len; invalid entries stay in place, -1)
 *   combined[t][topk_len + j] = M*b + N + (pos - swa_len + 1 - gather_start) + j   (j < swa_len)
 *   combined[t][topk_len + swa_len .. combined_width) = -1
 *   combined_lens[t]          = topk_len + swa_len
 * The two parts index different regions, so nothing is deduplicated.  The arithmetic is 32-bit
 * two's complement, as on the page.
 *
 * Arguments:
 *   topk_idx         int32 [num_tokens, topk_width], row stride topk_stride (>= topk_width);
 *                    may be NULL when top_k == 0.
 *   query_start_loc  int32 [num_reqs + 1], non-decreasing, query_start_loc[num_reqs] -
 *                    query_start_loc[0] == num_tokens (rows no request covers are set to -1
 *                    with length 0 and flag DSV4_ERR_BAD_INDEX in the device status word).
 *   seq_lens, gather_lens  int32 [num_reqs].
 *   num_reqs         >= 0; num_tokens >= 0 (either 0 enqueues nothing).
 *   region_stride, compressed_len  >= 0, region_stride * num_reqs < 2^31.
 *   top_k            0 .. topk_width (<= 8192); compress_ratio >= 1; window >= 0.
 *   combined         int32 [num_tokens, combined_width], row stride combined_stride
 *                    (>= combined_width); combined_width >= top_k + window.
 *   combined_lens    int32 [num_tokens].
 * Returns DSV4_OK, DSV4_ERR_INVALID_ARG, DSV4_ERR_UNSUPPORTED (topk_width > 8192) or DSV4_ERR_CUDA.
 */
DSV4_API dsv4_status dsv4_combine_topk_swa_indices_compressed(
    const int32_t *topk_idx, int64_t topk_stride, int32_t topk_width, const int32_t *query_start_loc,
    const int32_t *seq_lens, const int32_t *gather_lens, int32_t num_reqs, int32_t num_tokens, int32_t region_stride,
    int32_t compressed_len, int32_t top_k, int32_t compress_ratio, int32_t window, int32_t *combined,
    int64_t combined_stride, int32_t combined_width, int32_t *combined_lens, dsv4_stream_t stream);

/*
 * dsv4_selftest_wait_timeout -- checks the bounded waits and the status path without a fault.
 *
 * Every wait of the tensor-core decode kernel on an mbarrier gives up after a limit (about two
 * seconds), records DSV4_ERR_TIMEOUT in the device status word and lets the kernel run to its
 * end, so a lost arrival never hangs the GPU.  This call launches one small kernel whose single
 * thread runs that same bounded wait, with a limit of `cycles` SM clock cycles (1 .. 2^31), on
 * an mbarrier nothing arrives on: the next dsv4_get_device_status returns DSV4_ERR_TIMEOUT and
 * the context stays usable.  Returns DSV4_OK, DSV4_ERR_INVALID_ARG or DSV4_ERR_CUDA.
 */
DSV4_API dsv4_status dsv4_selftest_wait_timeout(int64_t cycles, dsv4_stream_t stream);

/*
 * dsv4_qnorm_rope_kv_insert -- the step before the decode: normalise and rotate the queries and
 * write each token's key into the FP8 cache.
 *
 * Source: vllm #42953 "feat: add DeepSeek-V4 XPU attention decode path", section 实现拆解 4
 * (xpu_qnorm_rope_kv_fp8_insert: fused Q per-head RMSNorm, GPT-J RoPE and FP8 UE8M0 KV insert,
 * called from forward_mqa with q, kv, kv_cache, slot_mapping and positions).  The page names
 * the steps, not their formulas; this library's readings:
 *   q_out[t][h] = RoPE(q[t][h] / sqrt(mean over 576 dims of q[t][h]^2 + eps) * w)
 *   kv_cache[slot_mapping[t]] = entry(kv[t]): per 128 latent values the smallest e with
 *       448 * 2^e >= amax (0 for amax 0, clamped to [-127, 127]), E4M3 codes of x * 2^-e
 *       (nearest, ties to even), scale byte e + 127; the rotated rope part in BF16; zero padding
 * GPT-J RoPE rotates the interleaved pairs (512 + 2i, 513 + 2i), i < 32, by the angle whose
 * cosine and sine are cos_sin_cache[positions[t]][i] and [32 + i].  The arithmetic is fp32 with
 * one rounding to BF16 (queries) or E4M3/BF16 (entries) at the end.
 *
 * Arguments:
 *   q, q_out         BF16 [num_tokens, num_heads, 576], token strides in elements (even, >=
 *                    num_heads * 576); q_out may be q.  Both 4-byte aligned.
 *   num_heads        1..128; q_norm_weight fp32 [576] or NULL (all ones); eps >= 0.
 *   kv               BF16 [num_tokens, 576] (512 latent, then 64 rope), token stride even, >= 576.
 *   positions, slot_mapping  int64 [num_tokens].
 *   cos_sin_cache    fp32 [max_position, 64]: 32 cosines, then 32 sines per position.
 *   kv_cache         uint8 [num_slots, 656] (a paged cache [num_blocks, page, 656] has
 *                    num_blocks * page slots), 16-byte aligned.
 * A negative slot writes nothing (a padding token).  A slot >= num_slots, or a position outside
 * [0, max_position), writes no entry and sets DSV4_ERR_BAD_INDEX in the device status word; such
 * a token's query is normalised but not rotated.  Nothing is allocated.  Returns DSV4_OK,
 * DSV4_ERR_INVALID_ARG or DSV4_ERR_CUDA.
 */
DSV4_API dsv4_status dsv4_qnorm_rope_kv_insert(const void *q, int64_t q_token_stride, void *q_out,
                                               int64_t q_out_token_stride, int32_t num_tokens, int32_t num_heads,
                                               const float *q_norm_weight, float eps, const void *kv,
                                               int64_t kv_token_stride, const int64_t *positions,
                                               const int64_t *slot_mapping, const float *cos_sin_cache,
                                               int32_t max_position, void *kv_cache, int64_t num_slots,
                                               dsv4_stream_t stream);

/*
 * dsv4_topk_select -- each token's top-k row from its indexer scores (the step that produces
 * topk_idx for the decode).
 *
 * Source: vllm #40860 "[Model] DeepSeek V4", section 实现拆解 2 (the MLA wrapper runs the
 * Indexer ahead of the sparse attention).  The pages print no selection rule; this is the
 * plain definition.  Token t's candidates are positions [0, n), n = num_cand[t] clamped to
 * [0, score_width]; the selected set is the min(top_k, n) candidates that come first in the
 * order "larger score first, then the smaller position", where -0 equals +0 and a NaN score
 * ranks below every number.
 *   topk_idx[t][0 .. m)        the selected positions in ascending order, m = min(top_k, n)
 *   topk_idx[t][m .. top_k)    -1
 *   topk_lens[t]               m
 *
 * Arguments:
 *   scores       fp32 [num_tokens, score_width], row stride score_stride (>= score_width).
 *   num_cand     int32 [num_tokens]: candidates per token (a decode token at position pos
 *                has pos + 1 raw positions, or (pos + 1) / ratio compressed entries).
 *   num_tokens   >= 0 (0 enqueues nothing); top_k >= 1.
 *   topk_idx     int32 [num_tokens, top_k], row stride topk_stride (>= top_k).
 *   topk_lens    int32 [num_tokens], or NULL.
 * All buffers are device memory owned by the caller; nothing is allocated.  The scores are
 * read from HBM once and up to four more times from L2 (the histogram rounds and the final
 * pass).  Returns DSV4_OK, DSV4_ERR_INVALID_ARG or DSV4_ERR_CUDA.
 */
DSV4_API dsv4_status dsv4_topk_select(const float *scores, int64_t score_stride, int32_t score_width,
                                      const int32_t *num_cand, int32_t num_tokens, int32_t top_k, int32_t *topk_idx,
                                      int64_t topk_stride, int32_t *topk_lens, dsv4_stream_t stream);

/*
 * dsv4_sparse_mla_decode_workspace_size -- bytes of device workspace dsv4_sparse_mla_decode needs.
 *
 * The size depends on the arguments and on the multiprocessor count of the current
 * CUDA device (it fixes how many workers share one token's keys); query it with the
 * device that will run the decode current.  Returns 0 for arguments the decode rejects.
 */
DSV4_API size_t dsv4_sparse_mla_decode_workspace_size(int32_t num_tokens, int32_t num_heads, int32_t topk_width,
                                             int32_t window);

/*
 * dsv4_sparse_mla_decode -- one sparse-MLA decode step (combine + gather/dequant + attention).
 *
 * Sources: the three pages named at the top of this file (combine: vllm #43385 rocm.py;
 * gather + dequant + BF16 sparse MLA: vllm #42953 xpu_sparse_decode_fp8.py; block-table
 * conversion, output [T, h, 512], sinks: vllm #43477 flashinfer_mla_sparse_sm120.py).
 *
 * For each token t and head h, with K_t the token's combined index list (as
 * dsv4_combine_topk_swa_indices with this call's arguments), row r = req_idx[t] (t when
 * req_idx is NULL), and for each logical position p in K_t the cache entry at
 *     slot = block_table[r][p / page_block] * page_block + p % page_block:
 *   s_p        = softmax_scale * sum_{d < 576} q[t][h][d] * k_p[d]
 *   lse[t][h]  = ln( sum_p e^{s_p} + e^{sink[h]} )        (no sink term when sink is NULL)
 *   out[t][h]  = sum_p e^{s_p - lse[t][h]} * v_p            (BF16, round-to-nearest-even)
 * A token with no key and no sink gets out = 0 and lse = -inf.  The sink is a logit in
 * the same units as s (it is not multiplied by softmax_scale).
 *
 * Arguments:
 *   q               BF16 [num_tokens, num_heads, 576]; heads contiguous (stride 576),
 *                   tokens at stride q_token_stride (>= num_heads * 576, multiple of 8).
 *                   16-byte aligned.
 *   kv_cache        uint8 [num_blocks, page_block, 656] (layout above), 16-byte aligned.
 *   block_table     int32 [num_reqs, max_blocks], row stride bt_stride (>= max_blocks).
 *                   Entries read must lie in [0, num_blocks); others are data errors.
 *   req_idx         int32 [num_tokens]: the block-table row of each token, in [0, num_reqs);
 *                   NULL means row t (then num_reqs >= num_tokens).  Several tokens may
 *                   share a row (speculative verify: one request, several positions).
 *   topk_idx, topk_stride, topk_width, topk_lens, seq_lens, window: as in
 *                   dsv4_combine_topk_swa_indices.  seq_lens[t] - 1 must be < max_blocks *
 *                   page_block for positions the token reads; others are data errors.
 *   num_tokens      >= 0 (0 enqueues nothing).
 *   num_heads       16, 32, 64 or 128 (others: DSV4_ERR_UNSUPPORTED).
 *   sink            float32 [num_heads] or NULL.
 *   softmax_scale   finite and >= 0 (a negative scale returns DSV4_ERR_INVALID_ARG; 0 gives uniform weights).
 *   out             BF16 [num_tokens, num_heads, 512], contiguous, 16-byte aligned.
 *   lse             float32 [num_tokens, num_heads], contiguous, or NULL.
 *   workspace       device scratch of at least dsv4_sparse_mla_decode_workspace_size(...)
 *                   bytes, 256-byte aligned, not used by anything else until the work
 *                   enqueued by this call has finished.  Its contents on entry do not matter.
 *   stream          CUDA stream.
 * When topk_lens is given and num_tokens * ceil(num_heads / 64) exceeds the device's
 * multiprocessor count, the call enqueues a one-CTA ordering kernel ahead of the decode kernel,
 * so that the tokens with the longest lists start first; the results do not depend on it.
 * Returns DSV4_OK, DSV4_ERR_INVALID_ARG, DSV4_ERR_UNSUPPORTED or DSV4_ERR_CUDA.
 */
DSV4_API dsv4_status dsv4_sparse_mla_decode(const void *q, int64_t q_token_stride, const void *kv_cache, int32_t num_blocks,
                                   int32_t page_block, const int32_t *block_table, int64_t bt_stride,
                                   int32_t max_blocks, int32_t num_reqs, const int32_t *req_idx,
                                   const int32_t *topk_idx, int64_t topk_stride, int32_t topk_width,
                                   const int32_t *topk_lens, const int32_t *seq_lens, int32_t num_tokens,
                                   int32_t num_heads, int32_t window, const float *sink, float softmax_scale,
                                   void *out, float *lse, void *workspace, size_t workspace_bytes,
                                   dsv4_stream_t stream);

/*
 * dsv4_sparse_mla_decode_trace -- dsv4_sparse_mla_decode that also records, from inside the
 * decode kernel, the combined index list each token was decoded over.
 *
 * A verification aid with no counterpart on the pages: the decode kernel combines each
 * token's top-k row with its window itself (the combine of dsv4_combine_topk_swa_indices,
 * vllm #43385 rocm.py, fused into the kernel's prologue); this entry point runs exactly that
 * kernel and lets a test compare the list it built with the definition bit for bit.
 *
 * Arguments: those of dsv4_sparse_mla_decode, then
 *   combined        int32 [num_tokens, combined_width], row stride combined_stride
 *                   (>= combined_width >= topk_width + window): entries [0, L) of row t
 *                   receive the logical positions of token t's keys in list order (the
 *                   kept top-k entries, then the window ascending); entries from L on are
 *                   not written.
 *   combined_lens   int32 [num_tokens]: L of each token.
 * The decode's out and lse are written as by dsv4_sparse_mla_decode.  Returns the codes of
 * dsv4_sparse_mla_decode, and DSV4_ERR_INVALID_ARG for a missing or too narrow record.
 */
DSV4_API dsv4_status dsv4_sparse_mla_decode_trace(const void *q, int64_t q_token_stride, const void *kv_cache,
                                                 int32_t num_blocks, int32_t page_block, const int32_t *block_table,
                                                 int64_t bt_stride, int32_t max_blocks, int32_t num_reqs,
                                                 const int32_t *req_idx, const int32_t *topk_idx,
                                                 int64_t topk_stride, int32_t topk_width, const int32_t *topk_lens,
                                                 const int32_t *seq_lens, int32_t num_tokens, int32_t num_heads,
                                                 int32_t window, const float *sink, float softmax_scale, void *out,
                                                 float *lse, void *workspace, size_t workspace_bytes,
                                                 int32_t *combined, int64_t combined_stride, int32_t combined_width,
                                                 int32_t *combined_lens, dsv4_stream_t stream);

/*
 * dsv4_sparse_mla_decode_noalloc -- dsv4_sparse_mla_decode without a workspace argument.
 *
 * The pages have no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory when they decode: code replaying a pipeline whose memory was
 * fixed at set-up, plug-ins whose host framework owns every allocation, and runtimes that
 * forbid cudaMalloc between start-up and shutdown.  It computes exactly what
 * dsv4_sparse_mla_decode computes, with the same arguments except `workspace` and
 * `workspace_bytes`: the scratch comes from one static device array inside the library,
 * 32 MiB (33,554,432 bytes), which every GPU that loads the library holds until the process
 * exits.  Nothing is allocated in the call.
 *
 * - A batch whose dsv4_sparse_mla_decode_workspace_size(...) exceeds 32 MiB is rejected with
 *   DSV4_ERR_UNSUPPORTED before anything is enqueued; use dsv4_sparse_mla_decode for it.
 * - The first call on a device looks up the array's device address (cudaGetSymbolAddress);
 *   make that first call before any stream capture on that device.
 * - All calls on a device share the one array and leave their scratch in it.  Nothing in it
 *   needs to start at zero (each call writes every scratch value before reading it), but
 *   calls whose work overlaps on the GPU -- on different streams, or on one stream without
 *   ordering -- race on the array; serialise them.
 * Returns the same codes as dsv4_sparse_mla_decode, plus DSV4_ERR_UNSUPPORTED for a batch
 * too large for the array and DSV4_ERR_CUDA when the address lookup fails.
 */
DSV4_API dsv4_status dsv4_sparse_mla_decode_noalloc(const void *q, int64_t q_token_stride, const void *kv_cache,
                                                   int32_t num_blocks, int32_t page_block, const int32_t *block_table,
                                                   int64_t bt_stride, int32_t max_blocks, int32_t num_reqs,
                                                   const int32_t *req_idx, const int32_t *topk_idx,
                                                   int64_t topk_stride, int32_t topk_width, const int32_t *topk_lens,
                                                   const int32_t *seq_lens, int32_t num_tokens, int32_t num_heads,
                                                   int32_t window, const float *sink, float softmax_scale, void *out,
                                                   float *lse, dsv4_stream_t stream);

/*
 * dsv4_sparse_mla_decode_mtp_union -- dsv4_sparse_mla_decode for speculative-verify batches in
 * which the two query tokens of a request run in one tile over the union of their key lists.
 *
 * Source: "[ROCm] [DSv4] [Perf] Support DeepSeek v4 MTP" (vllm #43385), 风险 1 (MTP throughput
 * falls at high concurrency because each request's tokens gather their keys separately); the
 * per-token result is that of dsv4_sparse_mla_decode.
 *
 * Computes exactly what dsv4_sparse_mla_decode computes for the same arguments (up to the
 * order in which a token's keys are summed), with this batch layout: num_tokens is even and
 * tokens 2r and 2r + 1 are the two query tokens of request r, which share a block-table row
 * (req_idx[2r] == req_idx[2r + 1]).  Each CTA takes 32 heads of both tokens (64 tile columns)
 * and the union of the two tokens' combined lists, each key masked for the token that does not
 * list it; a CTA of dsv4_sparse_mla_decode takes 64 heads of one token.
 *
 * Arguments: those of dsv4_sparse_mla_decode, with
 *   req_idx         required (not NULL);
 *   num_tokens      even, >= 0;
 *   num_heads       32, 64 or 128 (others: DSV4_ERR_UNSUPPORTED);
 *   num_blocks * page_block < 2^29;
 *   workspace       at least dsv4_sparse_mla_decode_mtp_union_workspace_size(...) bytes.
 * A request whose two tokens name different block-table rows, or a position of 2^29 or more,
 * is a data error (recorded in the status word; the request's outputs are then not defined).
 * Enqueues the combine of every token, one union kernel (one CTA a request) and the decode
 * kernel.  Returns the codes of dsv4_sparse_mla_decode.
 */
DSV4_API dsv4_status dsv4_sparse_mla_decode_mtp_union(const void *q, int64_t q_token_stride, const void *kv_cache,
                                                     int32_t num_blocks, int32_t page_block,
                                                     const int32_t *block_table, int64_t bt_stride,
                                                     int32_t max_blocks, int32_t num_reqs, const int32_t *req_idx,
                                                     const int32_t *topk_idx, int64_t topk_stride,
                                                     int32_t topk_width, const int32_t *topk_lens,
                                                     const int32_t *seq_lens, int32_t num_tokens, int32_t num_heads,
                                                     int32_t window, const float *sink, float softmax_scale,
                                                     void *out, float *lse, void *workspace, size_t workspace_bytes,
                                                     dsv4_stream_t stream);

/*
 * dsv4_sparse_mla_decode_mtp_union_workspace_size -- bytes of device workspace
 * dsv4_sparse_mla_decode_mtp_union needs (0 for arguments it rejects); depends on the current
 * device's multiprocessor count, as dsv4_sparse_mla_decode_workspace_size.
 */
DSV4_API size_t dsv4_sparse_mla_decode_mtp_union_workspace_size(int32_t num_tokens, int32_t num_heads,
                                                               int32_t topk_width, int32_t window);

/*
 * dsv4_get_device_status -- synchronise `stream`, then read and clear the current
 * device's sticky status word.
 *
 * Returns DSV4_OK when no kernel of this library on the current device recorded a data
 * error since the last call, DSV4_ERR_BAD_INDEX or DSV4_ERR_TIMEOUT for the recorded
 * error (BAD_INDEX wins when both were recorded), or DSV4_ERR_CUDA when the
 * synchronisation or the read failed.  The word is shared by all streams of the device.
 */
DSV4_API dsv4_status dsv4_get_device_status(dsv4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSV4_H_ */
