// mtp_union.cu -- the union key lists of MTP speculative-verify requests (a request's two
// query tokens, 2r and 2r + 1), the step ahead of the decode kernel's union mode
// ("[ROCm] [DSv4] [Perf] Support DeepSeek v4 MTP", vllm #43385, 风险 1: each request's tokens
// gather their keys separately).
#include <climits>

#include "internal.h"

namespace dsv4 {
namespace {

__device__ __forceinline__ unsigned hash_pos(int v, int bits)
{
    return ((unsigned)v * 0x9E3779B1u) >> (32 - bits);
}

// ---- MTP union: the two query tokens of request r (tokens 2r and 2r + 1) over the union of their
// combined lists.  Entry i of union row r is a position with bit 29 set when token 2r lists it and
// bit 30 when token 2r + 1 does: token 2r's list in its own order, then the positions only token
// 2r + 1 lists, in its order.  A position is in token t's list when it is one of the list's top-k
// survivors (its first len_t - swa_t entries, kept in a hash set) or inside the token's window.
constexpr int kUnionThreads = 256;
constexpr int kUnionMaxBits = 14;   // a hash set of 2^14 positions holds a top-k part of 8192
constexpr int kPosLimit = 1 << 29;  // positions carry two mask bits above them

__global__ void __launch_bounds__(kUnionThreads) mtp_union_kernel(const int32_t *__restrict__ lists, int64_t lstride,
                                                                  const int32_t *__restrict__ lens,
                                                                  const int32_t *__restrict__ seq_lens, int window,
                                                                  const int32_t *__restrict__ req_idx,
                                                                  int32_t *__restrict__ ulist, int64_t ustride,
                                                                  int32_t *__restrict__ ulen, int bits,
                                                                  unsigned *status)
{
    extern __shared__ int32_t usm[];   // the two tokens' top-k positions: two sets of 2^bits slots
    __shared__ int32_t wsum[kUnionThreads / 32];
    const int r = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int table = 1 << bits;
    const int t0 = 2 * r;
    int32_t *out = ulist + (int64_t)r * ustride;
    if (req_idx[t0] != req_idx[t0 + 1]) {   // the two tokens must read the same cache pages
        if (tid == 0) {
            ulen[r] = 0;
            atomicOr(status, kStatusBadIndex);
        }
        return;
    }
    int n[2], ntk[2], wlo[2], whi[2];   // list length, its top-k part, the window [wlo, whi]
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int s = seq_lens[t0 + k];
        const int pos = s - 1;
        const long long lo = (long long)pos - window + 1;
        wlo[k] = lo < 0 ? 0 : (int)lo;
        whi[k] = pos;
        const int swa = s > 0 ? pos - wlo[k] + 1 : 0;
        n[k] = min(max(lens[t0 + k], 0), (int)lstride);
        ntk[k] = max(0, n[k] - swa);
    }
    for (int i = tid; i < 2 * table; i += kUnionThreads)
        usm[i] = -1;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 2; ++k) {   // the top-k parts (distinct positions within a list)
        const int32_t *l = lists + (int64_t)(t0 + k) * lstride;
        int32_t *h = usm + k * table;
        for (int i = tid; i < ntk[k]; i += kUnionThreads) {
            const int v = l[i];
            unsigned s = hash_pos(v, bits);
            while (true) {
                const int prev = atomicCAS(&h[s], -1, v);
                if (prev == -1 || prev == v)
                    break;
                s = (s + 1u) & (unsigned)(table - 1);
            }
        }
    }
    __syncthreads();
    auto listed = [&](int k, int v) -> bool {   // is position v in token t0 + k's list
        if (v >= wlo[k] && v <= whi[k])
            return true;
        const int32_t *h = usm + k * table;
        unsigned s = hash_pos(v, bits);
        while (true) {
            const int x = h[s];
            if (x == v)
                return true;
            if (x == -1)
                return false;
            s = (s + 1u) & (unsigned)(table - 1);
        }
    };
    bool bad = false;
    const int32_t *l0 = lists + (int64_t)t0 * lstride;
    for (int i = tid; i < n[0]; i += kUnionThreads) {   // token 2r's list, in order
        const int v = l0[i];
        if (v >= kPosLimit) {   // no room for the mask bits: used by neither token
            bad = true;
            out[i] = v & (kPosLimit - 1);
        } else {
            out[i] = v | kPosLimit | (listed(1, v) ? 2 * kPosLimit : 0);
        }
    }
    const int32_t *l1 = lists + (int64_t)(t0 + 1) * lstride;
    int base = n[0];
    for (int i0 = 0; i0 < n[1]; i0 += kUnionThreads) {   // then what only token 2r + 1 lists, in order
        const int i = i0 + tid;
        int v = -1;
        bool add = false;
        if (i < n[1]) {
            v = l1[i];
            add = !listed(0, v);
        }
        const unsigned bal = __ballot_sync(0xffffffffu, add);
        if (lane == 0)
            wsum[warp] = __popc(bal);
        __syncthreads();
        int off = base, tot = 0;
#pragma unroll
        for (int w = 0; w < kUnionThreads / 32; ++w) {
            off += w < warp ? wsum[w] : 0;
            tot += wsum[w];
        }
        if (add) {
            const int o = off + __popc(bal & ((1u << lane) - 1u));
            if (v >= kPosLimit) {
                bad = true;
                out[o] = v & (kPosLimit - 1);
            } else {
                out[o] = v | 2 * kPosLimit;
            }
        }
        base += tot;
        __syncthreads();   // wsum is rewritten by the next step
    }
    if (bad)
        atomicOr(status, kStatusBadIndex);
    if (tid == 0)
        ulen[r] = base;
}

}  // namespace

int mtp_union_table_bits(int topk_width)
{
    int bits = 6;
    while (bits < kUnionMaxBits && (1 << bits) < 2 * topk_width)
        ++bits;
    return bits;
}

cudaError_t launch_mtp_union(const int32_t *lists, int64_t lstride, const int32_t *lens, const int32_t *seq_lens,
                             int window, const int32_t *req_idx, int num_reqs, int32_t *ulist, int64_t ustride,
                             int32_t *ulen, int topk_width, unsigned *status, cudaStream_t stream)
{
    if (num_reqs <= 0)
        return cudaSuccess;
    const int bits = mtp_union_table_bits(topk_width);
    const size_t smem = (size_t)2 * sizeof(int32_t) * ((size_t)1 << bits);
    if (smem > 48 * 1024) {
        cudaError_t e = set_smem_once(reinterpret_cast<const void *>(mtp_union_kernel), (int)smem, kAttrUnion);
        if (e != cudaSuccess)
            return e;
    }
    mtp_union_kernel<<<num_reqs, kUnionThreads, smem, stream>>>(lists, lstride, lens, seq_lens, window, req_idx, ulist,
                                                               ustride, ulen, bits, status);
    return cudaGetLastError();
}

}  // namespace dsv4
