// combine.cu -- top-k + sliding-window index combine, one CTA per query token.
//
// Follows the combine of "[ROCm] [DSv4] [Perf] Support DeepSeek v4 MTP" (vllm #43385,
// section "关键源码片段 / rocm.py", _combine_topk_swa_indices_kernel): valid top-k
// entries first in input order, then the window [pos - swa_len + 1, pos] ascending,
// swa_len = min(pos + 1, W).  With one cache region for both parts, top-k entries
// that are not causal, fall inside the window or repeat an earlier entry are
// dropped and the survivors are compacted.
//
// Design: the first-occurrence test is a shared-memory open-addressing hash set
// keyed by position that records the smallest top-k index holding each position
// (atomicCAS to claim a slot, atomicMin for the index).  Each thread owns a
// contiguous run of the top-k row, so a block-wide exclusive scan of per-thread
// survivor counts gives every survivor its output slot in input order.
#include <climits>

#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ unsigned hash_pos(int v, int bits)
{
    return ((unsigned)v * 0x9E3779B1u) >> (32 - bits);
}

__global__ void __launch_bounds__(kThreads) combine_kernel(const int32_t *__restrict__ topk, int64_t topk_stride,
                                                           int topk_width, const int32_t *__restrict__ topk_lens,
                                                           const int32_t *__restrict__ seq_lens, int window,
                                                           int32_t *__restrict__ combined, int64_t combined_stride,
                                                           int combined_width, int32_t *__restrict__ combined_lens,
                                                           int bits)
{
    // the decode kernel that follows may start its own prologue now; it reads this
    // kernel's results only after waiting for the whole grid
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ int32_t sm[];
    const int table = 1 << bits;
    int32_t *hkey = sm;           // position stored in the slot, -1 = empty
    int32_t *hmin = sm + table;   // smallest top-k index holding that position
    __shared__ int warp_sum[kThreads / 32];

    const int t = blockIdx.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int seq_len = seq_lens[t];
    const int pos = seq_len - 1;   // seq_len <= 0: nothing is visible
    int n = topk_width;
    if (topk_lens != nullptr) {
        n = topk_lens[t];
        n = n < 0 ? 0 : (n > topk_width ? topk_width : n);
    }
    // window [win_lo, pos]; top-k survivors are exactly the positions in [0, win_lo)
    const long long lo = (long long)pos - window + 1;
    const int win_lo = lo < 0 ? 0 : (int)lo;
    const int swa = seq_len > 0 ? pos - win_lo + 1 : 0;

    for (int i = tid; i < table; i += kThreads) {
        hkey[i] = -1;
        hmin[i] = INT_MAX;
    }
    __syncthreads();

    const int per = (n + kThreads - 1) / kThreads;
    const int i0 = min(n, tid * per);
    const int i1 = min(n, i0 + per);
    const int32_t *row = topk + (int64_t)t * topk_stride;
    const unsigned mask = (unsigned)table - 1u;

    for (int i = i0; i < i1; ++i) {
        const int v = row[i];
        if (v >= 0 && v < win_lo) {
            unsigned h = hash_pos(v, bits);
            while (true) {
                const int prev = atomicCAS(&hkey[h], -1, v);
                if (prev == -1 || prev == v) {
                    atomicMin(&hmin[h], i);
                    break;
                }
                h = (h + 1u) & mask;
            }
        }
    }
    __syncthreads();

    int count = 0;
    for (int i = i0; i < i1; ++i) {
        const int v = row[i];
        if (v >= 0 && v < win_lo) {
            unsigned h = hash_pos(v, bits);
            while (hkey[h] != v)
                h = (h + 1u) & mask;
            count += hmin[h] == i;
        }
    }

    // block-wide exclusive scan of the per-thread survivor counts
    int incl = count;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d)
            incl += y;
    }
    if (lane == 31)
        warp_sum[warp] = incl;
    __syncthreads();
    int warp_off = 0;
    int total = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        warp_off += w < warp ? warp_sum[w] : 0;
        total += warp_sum[w];
    }
    int o = warp_off + incl - count;

    int32_t *out = combined + (int64_t)t * combined_stride;
    for (int i = i0; i < i1; ++i) {
        const int v = row[i];
        if (v >= 0 && v < win_lo) {
            unsigned h = hash_pos(v, bits);
            while (hkey[h] != v)
                h = (h + 1u) & mask;
            if (hmin[h] == i)
                out[o++] = v;
        }
    }
    for (int k = tid; k < swa; k += kThreads)
        out[total + k] = win_lo + k;
    for (int k = total + swa + tid; k < combined_width; k += kThreads)
        out[k] = -1;
    if (tid == 0)
        combined_lens[t] = total + swa;
}

// Compressed-region combine (the page's full variant): one CTA per token row.  The CTA finds
// the request whose query range holds its row (a parallel search over query_start_loc), then
// writes the row one entry per thread at a time (coalesced top-k reads and row writes).  A row
// that no request covers is written as -1 with length 0 and flags the bad-index status.
constexpr int kCompThreads = 256;

constexpr int kCompRun = 4;   // entries per thread per pass: one 16-byte store when the row is aligned

__global__ void __launch_bounds__(kCompThreads) combine_compressed_kernel(
    const int32_t *__restrict__ topk, int64_t topk_stride, const int32_t *__restrict__ qsl,
    const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ gather_lens, int num_reqs, int region_stride,
    int compressed_len, int top_k, int compress_ratio, int window, int32_t *__restrict__ combined,
    int64_t combined_stride, int combined_width, int32_t *__restrict__ combined_lens, unsigned *status)
{
    __shared__ int req;
    const long long t = blockIdx.x;
    const int32_t *in = topk + t * topk_stride;
    // the first pass's top-k entries do not depend on the request: their loads go out first
    int x0[kCompRun];
#pragma unroll
    for (int u = 0; u < kCompRun; ++u) {
        const int k = kCompRun * threadIdx.x + u;
        x0[u] = k < top_k ? __ldg(in + k) : -1;
    }
    const long long base = qsl[0];
    if (threadIdx.x == 0)
        req = -1;
    __syncthreads();
    for (int b = threadIdx.x; b < num_reqs; b += kCompThreads)
        if (qsl[b] - base <= t && t < qsl[b + 1] - base)
            req = b;
    __syncthreads();
    const int b = req;
    int32_t *row = combined + t * combined_stride;
    const bool vec = (reinterpret_cast<uintptr_t>(row) % 16 == 0) && (combined_width % kCompRun == 0);
    int tk = 0, sw = 0;
    long long region = 0, win0 = 0;
    if (b >= 0) {
        // 64-bit intermediates, truncated to 32 bits on output (the page's arithmetic is 32-bit)
        const long long qs = qsl[b] - base;
        const long long qe = qsl[b + 1] - base;
        const long long pos = (long long)seq_lens[b] - (qe - qs) + (t - qs);
        const long long gather_start = (long long)seq_lens[b] - gather_lens[b];
        region = (long long)region_stride * b;
        if (pos + 1 > 0) {
            tk = (int)min((pos + 1) / compress_ratio, (long long)top_k);
            sw = (int)min(pos + 1, (long long)window);
        }
        win0 = region + compressed_len + (pos - sw + 1 - gather_start);
    } else if (threadIdx.x == 0) {   // no request covers this row: -1, length 0
        atomicOr(status, kStatusBadIndex);
    }
    auto entry = [&](int k, int x) -> int32_t {
        if (k < tk)
            return (x >= 0 && x < compressed_len) ? (int32_t)(region + x) : -1;
        if (k < tk + sw)
            return (int32_t)(win0 + (k - tk));
        return -1;
    };
    for (int k0 = kCompRun * threadIdx.x; k0 < combined_width; k0 += kCompRun * kCompThreads) {
        int32_t v[kCompRun];
#pragma unroll
        for (int u = 0; u < kCompRun; ++u) {
            const int k = k0 + u;
            const int x = k0 < kCompRun * kCompThreads ? x0[u] : (k < tk ? __ldg(in + k) : -1);
            v[u] = entry(k, x);
        }
        if (vec) {
            *reinterpret_cast<int4 *>(row + k0) = make_int4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
            for (int u = 0; u < kCompRun; ++u)
                if (k0 + u < combined_width)
                    row[k0 + u] = v[u];
        }
    }
    if (threadIdx.x == 0)
        combined_lens[t] = tk + sw;
}

}  // namespace

cudaError_t launch_combine_compressed(const int32_t *topk, int64_t topk_stride, const int32_t *qsl,
                                      const int32_t *seq_lens, const int32_t *gather_lens, int num_reqs,
                                      int num_tokens, int region_stride, int compressed_len, int top_k,
                                      int compress_ratio, int window, int32_t *combined, int64_t combined_stride,
                                      int combined_width, int32_t *combined_lens, unsigned *status,
                                      cudaStream_t stream)
{
    if (num_reqs <= 0 || num_tokens <= 0)
        return cudaSuccess;
    combine_compressed_kernel<<<num_tokens, kCompThreads, 0, stream>>>(
        topk, topk_stride, qsl, seq_lens, gather_lens, num_reqs, region_stride, compressed_len, top_k,
        compress_ratio, window, combined, combined_stride, combined_width, combined_lens, status);
    return cudaGetLastError();
}

int combine_table_bits(int topk_width)
{
    int bits = 6;
    while ((1 << bits) < 2 * topk_width)
        ++bits;
    return bits;
}

size_t combine_smem_bytes(int table_bits, int /*topk_width*/)
{
    return (size_t)2 * sizeof(int32_t) * ((size_t)1 << table_bits);
}

cudaError_t launch_combine(const int32_t *topk, int64_t topk_stride, int topk_width, const int32_t *topk_lens,
                           const int32_t *seq_lens, int num_tokens, int window, int32_t *combined,
                           int64_t combined_stride, int combined_width, int32_t *combined_lens, int table_bits,
                           cudaStream_t stream)
{
    if (num_tokens <= 0)
        return cudaSuccess;
    const size_t smem = combine_smem_bytes(table_bits, topk_width);
    if (smem > 48 * 1024) {
        cudaError_t e = set_smem_once(reinterpret_cast<const void *>(combine_kernel), (int)smem, kAttrCombine);
        if (e != cudaSuccess)
            return e;
    }
    combine_kernel<<<num_tokens, kThreads, smem, stream>>>(topk, topk_stride, topk_width, topk_lens, seq_lens, window,
                                                          combined, combined_stride, combined_width, combined_lens,
                                                          table_bits);
    return cudaGetLastError();
}

}  // namespace dsv4
