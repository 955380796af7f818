// topk.cu -- top-k selection from indexer scores: the step that produces each token's top-k
// row ("[Model] DeepSeek V4", vllm #40860, 实现拆解 2: the MLA wrapper runs the Indexer ahead
// of the sparse attention).  The pages print no selection rule; this kernel computes the
// plain definition: row t's candidates are positions [0, n), n = num_cand[t] clamped to
// [0, width]; the selected set is the min(K, n) candidates first in the order "larger score
// first, then smaller position" (-0 equal to +0, NaN below every number); the row lists the
// selected positions ascending, then -1; lens[t] = min(K, n).
//
// One thread-block cluster of CL CTAs per token row (CL = 1 when the rows alone fill the
// GPU), each CTA a contiguous segment of the row.  Scores become order-preserving 32-bit
// keys; three histogram rounds (11, 11 and 10 bits from the top) find the K-th largest key
// v* and how many keys equal to v* the selection takes.  Each round every CTA builds its
// segment's histogram in shared memory, then reduces one slice of the bins across the
// cluster through distributed shared memory; the owner of the slice holding the K-th key
// broadcasts the digit.  A last pass over the row in position order writes every position
// with key > v* and the first ones with key == v*.  The first pass reads the scores from
// HBM; the later ones normally hit L2.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkBins = 2048;          // 11-bit digits
constexpr int kTkItems = 8;            // final pass: consecutive positions per thread
constexpr int kTkTile = kTkThreads * kTkItems;

struct TopkParams {
    const float *scores;
    int64_t score_stride;
    int32_t width;
    const int32_t *num_cand;
    int32_t top_k;
    int32_t *out;
    int64_t out_stride;
    int32_t *lens;
    int32_t cluster;
};

// Order-preserving key: larger score -> larger key; -0 and +0 share a key; NaN -> 0, below
// every number (-inf maps to 0x007FFFFF).
__device__ __forceinline__ uint32_t order_key(float x)
{
    if (x != x)
        return 0u;
    uint32_t u = __float_as_uint(x);
    if ((u << 1) == 0u)
        u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void cluster_barrier()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t remote_addr(const void *p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(r)
                 : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_remote(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_remote(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Inclusive prefix sum over the CTA's threads; `total` gets the sum of all.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t *wsum, uint32_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += y;
    }
    if (lane == 31)
        wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < kTkWarps ? wsum[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        if (lane < kTkWarps)
            wsum[lane] = w;
    }
    __syncthreads();
    const uint32_t r = v + (warp > 0 ? wsum[warp - 1] : 0u);
    total = wsum[kTkWarps - 1];
    __syncthreads();   // wsum is reused by the next scan
    return r;
}

__global__ void __launch_bounds__(kTkThreads) topk_select_kernel(const TopkParams p)
{
    __shared__ uint32_t hist[kTkBins];     // this CTA's histogram of the round
    __shared__ uint32_t slice[kTkBins];    // this CTA's slice of the cluster-wide histogram
    __shared__ uint32_t sums[8];           // slice totals of every CTA of the cluster
    __shared__ uint32_t bcast[2];          // the round's digit and remaining count
    __shared__ uint32_t cnt[8][2];         // final pass: (> v*, == v*) counts per CTA
    __shared__ uint32_t wsum[kTkWarps];

    const int tid = threadIdx.x;
    const int CL = p.cluster;
    const uint32_t rank = CL > 1 ? cluster_rank() : 0u;
    // a word into the shared memory of CTA `r` of the cluster (plain store without a cluster)
    auto put = [&](uint32_t *local, int r, uint32_t v) {
        if (CL > 1)
            st_remote(remote_addr(local, (uint32_t)r), v);
        else
            *local = v;
    };
    const int64_t t = blockIdx.x / CL;
    int64_t n = p.num_cand[t];
    n = n < 0 ? 0 : (n > p.width ? p.width : n);
    const int64_t K = p.top_k;
    const int64_t m = n < K ? n : K;
    int32_t *orow = p.out + t * p.out_stride;
    if (rank == 0 && tid == 0 && p.lens)
        p.lens[t] = (int32_t)m;

    if (n <= K) {   // every candidate is selected: positions 0..n-1, then -1
        for (int64_t i = (int64_t)rank * kTkThreads + tid; i < K; i += (int64_t)CL * kTkThreads)
            orow[i] = i < n ? (int32_t)i : -1;
        return;
    }

    const float *row = p.scores + t * p.score_stride;
    const int64_t seg = ((n + CL - 1) / CL + 3) / 4 * 4;   // a multiple of 4: 16-byte loads stay aligned
    const int64_t lo = min(n, (int64_t)rank * seg);
    const int64_t hi = min(n, lo + seg);
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;

    // ---- three digit rounds: find the K-th largest key
    uint32_t prefix = 0u, pmask = 0u, rem = (uint32_t)m;
#pragma unroll 1
    for (int round = 0; round < 3; ++round) {
        const int shift = round == 0 ? 21 : (round == 1 ? 10 : 0);
        const int nb = round == 2 ? 1024 : 2048;
        const uint32_t dmask = (uint32_t)nb - 1u;
        for (int i = tid; i < nb; i += kTkThreads)
            hist[i] = 0u;
        __syncthreads();
        auto count = [&](float x) {
            const uint32_t k = order_key(x);
            if ((k & pmask) == prefix)
                atomicAdd(&hist[(k >> shift) & dmask], 1u);
        };
        if (vec) {
            const float4 *r4 = reinterpret_cast<const float4 *>(row + lo);
            const int64_t n4 = (hi - lo) / 4;
#pragma unroll 4
            for (int64_t i = tid; i < n4; i += kTkThreads) {
                const float4 v = __ldg(r4 + i);
                count(v.x);
                count(v.y);
                count(v.z);
                count(v.w);
            }
            for (int64_t i = lo + 4 * n4 + tid; i < hi; i += kTkThreads)
                count(__ldg(row + i));
        } else {
#pragma unroll 4
            for (int64_t i = lo + tid; i < hi; i += kTkThreads)
                count(__ldg(row + i));
        }
        if (CL > 1)
            cluster_barrier();   // every segment's histogram is complete
        else
            __syncthreads();
        // this CTA's slice of the bins, summed over the cluster
        const int per = (nb + CL - 1) / CL;
        const int s_lo = min(nb, (int)rank * per);
        const int s_hi = min(nb, s_lo + per);
        uint32_t part = 0u;
        for (int b = s_lo + tid; b < s_hi; b += kTkThreads) {
            uint32_t s = hist[b];
            for (int r = 0; r < CL; ++r)
                if (r != (int)rank)
                    s += ld_remote(remote_addr(&hist[b], (uint32_t)r));
            slice[b - s_lo] = s;
            part += s;
        }
        uint32_t tot;
        block_scan(part, wsum, tot);
        if (tid < CL)
            put(&sums[rank], tid, tot);
        if (CL > 1)
            cluster_barrier();   // slice totals everywhere
        else
            __syncthreads();
        // the slice holding the rem-th largest key (higher ranks hold higher bins)
        uint32_t above = 0u;
        int owner = 0;
        for (int r = CL - 1; r >= 0; --r) {
            if (above + sums[r] >= rem) {
                owner = r;
                break;
            }
            above += sums[r];
        }
        if ((int)rank == owner) {
            // thread i takes the i-th group of c bins counted from the top of the slice
            const int len = s_hi - s_lo;
            const int c = (len + kTkThreads - 1) / kTkThreads;
            const int g_hi = len - tid * c;
            const int g_lo = max(0, g_hi - c);
            uint32_t gs = 0u;
            for (int b = g_lo; b < g_hi; ++b)
                gs += slice[b];
            uint32_t gtot;
            const uint32_t incl = block_scan(gs, wsum, gtot);
            uint32_t a = above + incl - gs;   // keys in bins above this group
            if (g_lo < g_hi && a < rem && rem <= a + gs) {
                for (int b = g_hi - 1; b >= g_lo; --b) {
                    if (a + slice[b] >= rem) {
                        for (int r = 0; r < CL; ++r) {
                            put(&bcast[0], r, (uint32_t)(s_lo + b));
                            put(&bcast[1], r, rem - a);
                        }
                        break;
                    }
                    a += slice[b];
                }
            }
        }
        if (CL > 1)
            cluster_barrier();   // the digit is known everywhere; remote reads of hist are over
        else
            __syncthreads();
        prefix |= bcast[0] << shift;
        pmask |= dmask << shift;
        rem = bcast[1];
    }
    const uint32_t vstar = prefix;   // the K-th largest key; rem keys equal to it are taken

    // ---- counts of this segment, then the output offsets of every segment
    uint32_t g = 0u, e = 0u;
    for (int64_t i = lo + tid; i < hi; i += kTkThreads) {
        const uint32_t k = order_key(__ldg(row + i));
        g += k > vstar;
        e += k == vstar;
    }
    uint32_t gtot, etot;
    block_scan(g, wsum, gtot);
    block_scan(e, wsum, etot);
    if (tid < CL) {
        put(&cnt[rank][0], tid, gtot);
        put(&cnt[rank][1], tid, etot);
    }
    if (CL > 1)
        cluster_barrier();
    else
        __syncthreads();
    uint32_t G = 0u, E = 0u;   // keys > v* and == v* before this segment
    for (int r = 0; r < (int)rank; ++r) {
        G += cnt[r][0];
        E += cnt[r][1];
    }
    // ---- position-ordered compaction: the output index of a selected position is
    // (keys > v* before it) + min(keys == v* before it, rem)
#pragma unroll 1
    for (int64_t base = lo; base < hi; base += kTkTile) {
        const int64_t i0 = base + (int64_t)tid * kTkItems;
        uint32_t keys[kTkItems];
        uint32_t pk = 0u;   // (> v*) << 16 | (== v*) among this thread's positions
#pragma unroll
        for (int j = 0; j < kTkItems; ++j) {
            keys[j] = i0 + j < hi ? order_key(__ldg(row + i0 + j)) : 0u;
            const bool in = i0 + j < hi;
            pk += (in && keys[j] > vstar) ? 0x10000u : ((in && keys[j] == vstar) ? 1u : 0u);
        }
        uint32_t ptot;
        const uint32_t excl = block_scan(pk, wsum, ptot) - pk;
        uint32_t gb = G + (excl >> 16), eb = E + (excl & 0xFFFFu);
#pragma unroll
        for (int j = 0; j < kTkItems; ++j) {
            if (i0 + j >= hi)
                break;
            if (keys[j] > vstar) {
                orow[gb + min(eb, rem)] = (int32_t)(i0 + j);
                ++gb;
            } else if (keys[j] == vstar) {
                if (eb < rem)
                    orow[gb + eb] = (int32_t)(i0 + j);
                ++eb;
            }
        }
        G += ptot >> 16;
        E += ptot & 0xFFFFu;
    }
}

}  // namespace

int topk_cluster_size(int num_tokens, int width, int sms)
{
    int cl = 1;
    while (cl < 8 && (long long)num_tokens * (cl + 1) <= sms && (long long)(cl + 1) * 4096 <= width)
        ++cl;
    return cl;
}

cudaError_t launch_topk_select(const float *scores, int64_t score_stride, int width, const int32_t *num_cand,
                               int num_tokens, int top_k, int32_t *out, int64_t out_stride, int32_t *lens,
                               int cluster, cudaStream_t stream)
{
    if (num_tokens <= 0)
        return cudaSuccess;
    if (cluster < 1 || cluster > 8 || top_k < 1)
        return cudaErrorInvalidValue;
    TopkParams p{scores, score_stride, width, num_cand, top_k, out, out_stride, lens, cluster};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)num_tokens * cluster));
    cfg.blockDim = dim3(kTkThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 1 : 0;
    void *args[] = {&p};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(topk_select_kernel), args);
}

}  // namespace dsv4
