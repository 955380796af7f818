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
// v* and how many keys equal to v* the selection takes.  For each round every CTA builds its
// segment's histogram in shared memory, sums one slice of the bins over the cluster through
// distributed shared memory and writes the sums into every CTA; each CTA then finds the digit
// itself (two cluster barriers a round).  Round 0 reads the scores from HBM with 16-byte loads issued four deep and keeps
// the segment's keys in shared memory (up to 40960 keys a CTA).  One pass over the cached
// keys then lists the keys of round 0's bin with their positions (up to 128 a warp chunk, 256 in
// a whole-row CTA whose shared memory has room) and
// counts the keys above it; rounds 1 and 2 and the per-chunk counts work on that list alone
// (a segment with more candidates, i.e. many equal keys, rescans its keys instead).  The
// compaction walks the segment in position order, one contiguous chunk per warp with warp
// scans only, and writes every position with key > v* and the first ones with key == v*.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace dsv4 {
namespace {

// CTA size: 1024 threads when a row has a CTA to itself, 512 in clusters (two CTAs fit an SM,
// so a cluster's CTAs find room inside one GPC)
constexpr int kTkThreadsRow = 1024;
constexpr int kTkThreadsCluster = 512;
constexpr int kTkBins = 2048;          // 11-bit digits
constexpr int kTkCacheKeys = 40960;    // keys of a segment kept in shared memory (160 KB)
constexpr int kTkStep = 32 * 8;        // compaction: a warp takes 8 consecutive positions per lane
constexpr int kTkCandWarp = 128;       // candidates (keys in round 0's bin) a warp chunk keeps in shared memory,
constexpr int kTkCandWarpWide = 256;   // or, for whole-row CTAs whose shared memory has room, this many
constexpr int kTkRowDynMax = 204800;   // dynamic shared memory of a whole-row CTA (with its 17 KB static: < 227 KB)

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
    int32_t cache;   // keys of shared-memory cache per CTA (0: no cache; every segment fits otherwise)
    int32_t cand;    // entries of a warp's candidate list (kTkCandWarp or kTkCandWarpWide)
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

// Inclusive prefix sum over the CTA's NT threads; `total` gets the sum of all.
template <int NT>
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t *wsum, uint32_t &total)
{
    constexpr int kTkWarps = NT / 32;
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

// Visits every key of the segment row[lo, hi): from the shared-memory cache (kc[i - lo]) when
// `cached`, else from global memory, storing it into the cache when `fill`.  Loads are issued
// four deep before any key is used.  f(key) must not synchronise.
template <int NT, class F>
__device__ __forceinline__ void visit_keys(const float *row, int64_t lo, int64_t hi, bool vec, uint32_t *kc,
                                           bool cached, bool fill, F f)
{
    const int tid = threadIdx.x;
    const int64_t len = hi - lo;
    const int64_t n4 = len / 4;
    if (cached) {
        const uint4 *k4 = reinterpret_cast<const uint4 *>(kc);
        for (int64_t b = 0; b < n4; b += 4 * NT) {
            uint4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t i = b + j * NT + tid;
                v[j] = i < n4 ? k4[i] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (b + j * NT + tid < n4) {
                    f(v[j].x);
                    f(v[j].y);
                    f(v[j].z);
                    f(v[j].w);
                }
        }
        for (int64_t i = 4 * n4 + tid; i < len; i += NT)
            f(kc[i]);
        return;
    }
    if (vec) {
        const float4 *r4 = reinterpret_cast<const float4 *>(row + lo);
        for (int64_t b = 0; b < n4; b += 4 * NT) {
            float4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t i = b + j * NT + tid;
                v[j] = i < n4 ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t i = b + j * NT + tid;
                if (i < n4) {
                    const uint4 k = make_uint4(order_key(v[j].x), order_key(v[j].y), order_key(v[j].z),
                                               order_key(v[j].w));
                    if (fill)
                        reinterpret_cast<uint4 *>(kc)[i] = k;
                    f(k.x);
                    f(k.y);
                    f(k.z);
                    f(k.w);
                }
            }
        }
    } else {
        for (int64_t b = 0; b < 4 * n4; b += 4 * NT) {
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t i = b + j * NT + tid;
                v[j] = i < 4 * n4 ? __ldg(row + lo + i) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t i = b + j * NT + tid;
                if (i < 4 * n4) {
                    const uint32_t k = order_key(v[j]);
                    if (fill)
                        kc[i] = k;
                    f(k);
                }
            }
        }
    }
    for (int64_t i = 4 * n4 + tid; i < len; i += NT) {
        const uint32_t k = order_key(__ldg(row + lo + i));
        if (fill)
            kc[i] = k;
        f(k);
    }
}

template <int NT>
__global__ void __launch_bounds__(NT) topk_select_kernel(const TopkParams p)
{
    constexpr int kTkThreads = NT;
    constexpr int kTkWarps = NT / 32;
    __shared__ uint32_t hist[kTkBins];     // this CTA's histogram of the round
    __shared__ uint32_t slice[kTkBins];    // the cluster-wide histogram (clusters of more than one CTA)
    __shared__ uint32_t bcast[2];          // the round's digit and remaining count
    __shared__ uint32_t cnt[8][2];         // (> v*, == v*) counts per CTA
    __shared__ uint32_t wsum[kTkWarps];
    __shared__ uint32_t wsure[kTkWarps];     // keys above round 0's bin per warp chunk
    __shared__ uint32_t wcnt[kTkWarps][2];   // (> v*, == v*) counts per warp chunk
    __shared__ uint32_t wncand[kTkWarps];    // candidates per warp chunk
    // [p.cache keys][cand x warps candidate keys][cand x warps positions][a bit per cached position]
    extern __shared__ uint4 dyn4[];
    uint32_t *kc = reinterpret_cast<uint32_t *>(dyn4);
    uint32_t *ckey = kc + p.cache;
    const int cap = p.cand;                // entries of a warp's candidate list
    uint32_t *cpos = ckey + cap * kTkWarps;
    uint32_t *bm = cpos + cap * kTkWarps;  // the selected positions of the segment (with the cache)

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int CL = p.cluster;
    const uint32_t rank = CL > 1 ? cluster_rank() : 0u;
    // a word into the shared memory of CTA `r` of the cluster (plain store without a cluster)
    auto put = [&](uint32_t *local, int r, uint32_t v) {
        if (CL > 1)
            st_remote(remote_addr(local, (uint32_t)r), v);
        else
            *local = v;
    };
    auto sync_all = [&]() {
        if (CL > 1)
            cluster_barrier();
        else
            __syncthreads();
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
    const bool cache = p.cache > 0;
    const int len = (int)(hi - lo);
    // warp w owns the chunk [c_lo, c_hi) of the segment (a multiple of 128 positions long, so that
    // chunks start on a bitmap word)
    const int cw = ((len + kTkWarps - 1) / kTkWarps + 127) / 128 * 128;
    const int c_lo = min(len, warp * cw);
    const int c_hi = min(len, c_lo + cw);
    auto key_at = [&](int i) -> uint32_t { return cache ? kc[i] : order_key(__ldg(row + lo + i)); };

    // The digit of a round: the cluster-wide histogram of the round (this CTA's part in
    // `hist`) decides which bin holds the rem-th largest key; rem becomes its rank in the bin.
    uint32_t rem = (uint32_t)m;
    auto find_digit = [&](int nb) -> uint32_t {
        sync_all();   // every segment's histogram is complete
        const uint32_t *bins = hist;
        if (CL > 1) {
            // this CTA sums its slice of the bins over the cluster and writes the sums into every
            // CTA's copy of the cluster-wide histogram (`slice`)
            const int per = (nb + CL - 1) / CL;
            const int s_lo = min(nb, (int)rank * per);
            const int s_hi = min(nb, s_lo + per);
            for (int b = s_lo + tid; b < s_hi; b += kTkThreads) {
                uint32_t v[8];
#pragma unroll
                for (int r = 0; r < 8; ++r)   // every remote load in flight before the sum
                    v[r] = (r < CL && r != (int)rank) ? ld_remote(remote_addr(&hist[b], (uint32_t)r)) : 0u;
                uint32_t sm = hist[b];
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    sm += v[r];
                for (int r = 0; r < CL; ++r)
                    put(&slice[b], r, sm);
            }
            cluster_barrier();   // the cluster-wide histogram is in every CTA; remote reads of hist are over
            bins = slice;
        }
        // every CTA finds the digit itself: thread i takes the i-th group of c bins from the top
        const int c = (nb + kTkThreads - 1) / kTkThreads;
        const int g_hi = nb - tid * c;
        const int g_lo = max(0, g_hi - c);
        uint32_t gs = 0u;
        for (int b = g_lo; b < g_hi; ++b)
            gs += bins[b];
        uint32_t gtot;
        const uint32_t incl = block_scan<NT>(gs, wsum, gtot);
        uint32_t a = incl - gs;   // keys in bins above this group
        if (g_lo < g_hi && a < rem && rem <= a + gs) {
            for (int b = g_hi - 1; b >= g_lo; --b) {
                if (a + bins[b] >= rem) {
                    bcast[0] = (uint32_t)b;
                    bcast[1] = rem - a;
                    break;
                }
                a += bins[b];
            }
        }
        __syncthreads();
        rem = bcast[1];
        return bcast[0];
    };

    // ---- round 0 (top 11 bits) over every key; the keys go to the shared-memory cache
    for (int i = tid; i < kTkBins; i += kTkThreads)
        hist[i] = 0u;
    if (cache)
        for (int i = tid; i < (len + 31) / 32; i += kTkThreads)
            bm[i] = 0u;
    __syncthreads();
    visit_keys<NT>(row, lo, hi, vec, kc, false, cache, [&](uint32_t k) { atomicAdd(&hist[k >> 21], 1u); });
    const uint32_t d0 = find_digit(kTkBins);
    uint32_t prefix = d0 << 21, pmask = 0xFFE00000u;

    // ---- the keys in round 0's bin become candidates (key, position), each warp listing those
    // of its chunk in position order; keys above the bin are selected whatever the later rounds
    // find: they are counted, and (with the cache) marked in the bitmap
    uint32_t sure = 0u, nw = 0u;   // per warp (the same in every lane): keys above the bin, candidates so far
    uint32_t *wkey = ckey + warp * cap;
    uint32_t *wpos = cpos + warp * cap;
    const uint32_t below = (1u << lane) - 1u;
    for (int i0 = c_lo; i0 < c_hi; i0 += 128) {   // lane l takes positions i0 + 32 j + l: a bitmap word is a ballot
        const bool full = cache && i0 + 128 <= c_hi;
        uint32_t k[4];
        if (full) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                k[j] = kc[i0 + 32 * j + lane];
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + 32 * j + lane;
                k[j] = i < c_hi ? key_at(i) : 0u;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + 32 * j + lane;
            const bool in = full || i < c_hi;
            const uint32_t dg = k[j] >> 21;
            const uint32_t bu = __ballot_sync(0xffffffffu, in && dg > d0);
            const uint32_t bc = __ballot_sync(0xffffffffu, in && dg == d0);
            sure += (uint32_t)__popc(bu);
            if (bc != 0u) {   // candidates in position order: (j, lane) is position order within the 128
                if ((bc >> lane) & 1u) {
                    const uint32_t slot = nw + (uint32_t)__popc(bc & below);
                    if (slot < (uint32_t)cap) {
                        wkey[slot] = k[j];
                        wpos[slot] = (uint32_t)i;
                    }
                }
                nw += (uint32_t)__popc(bc);
            }
            if (cache && lane == j && i0 + 32 * j < c_hi)
                bm[(i0 >> 5) + j] = bu;
        }
    }
    if (lane == 0) {
        wsure[warp] = sure;
        wncand[warp] = nw;
    }
    __syncthreads();
    bool listed = true;   // else (many equal keys in one chunk) the rounds rescan the segment
    for (int w = 0; w < kTkWarps; ++w)
        listed = listed && wncand[w] <= (uint32_t)cap;

    // ---- rounds 1 (next 11 bits) and 2 (last 10 bits)
#pragma unroll 1
    for (int round = 1; round < 3; ++round) {
        const int shift = round == 1 ? 10 : 0;
        const int nb = round == 1 ? 2048 : 1024;
        const uint32_t dmask = (uint32_t)nb - 1u;
        for (int i = tid; i < nb; i += kTkThreads)
            hist[i] = 0u;
        __syncthreads();
        auto count = [&](uint32_t k) {
            if ((k & pmask) == prefix)
                atomicAdd(&hist[(k >> shift) & dmask], 1u);
        };
        if (listed) {   // every warp its own list
            const uint32_t nwc = wncand[warp];
            for (uint32_t c = lane; c < nwc; c += 32)
                count(wkey[c]);
        } else {
            visit_keys<NT>(row, lo, hi, vec, kc, cache, false, count);
        }
        const uint32_t d = find_digit(nb);
        prefix |= d << shift;
        pmask |= dmask << shift;
    }
    const uint32_t vstar = prefix;   // the K-th largest key; rem keys equal to it are taken

    // ---- (> v*, == v*) per warp chunk, then per segment and the segments' offsets
    {
        uint32_t ng = 0u, ne = 0u;
        if (listed) {   // the warp's own list, plus the keys above round 0's bin
            const uint32_t nwc = wncand[warp];
            for (uint32_t c = lane; c < nwc; c += 32) {
                const uint32_t k = wkey[c];
                ng += k > vstar ? 1u : 0u;
                ne += k == vstar ? 1u : 0u;
            }
        } else {
            for (int i = c_lo + lane; i < c_hi; i += 32) {
                const uint32_t k = key_at(i);
                ng += k > vstar ? 1u : 0u;
                ne += k == vstar ? 1u : 0u;
            }
        }
        ng = __reduce_add_sync(0xffffffffu, ng);
        ne = __reduce_add_sync(0xffffffffu, ne);
        if (lane == 0) {
            wcnt[warp][0] = ng + (listed ? wsure[warp] : 0u);
            wcnt[warp][1] = ne;
        }
    }
    __syncthreads();
    // every warp scans the chunk counts: lane w holds chunk w's
    uint32_t gt_local, eq_local, wg, we;
    {
        uint32_t g = lane < kTkWarps ? wcnt[lane][0] : 0u;
        uint32_t e = lane < kTkWarps ? wcnt[lane][1] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t yg = __shfl_up_sync(0xffffffffu, g, o);
            const uint32_t ye = __shfl_up_sync(0xffffffffu, e, o);
            if (lane >= o) {
                g += yg;
                e += ye;
            }
        }
        gt_local = __shfl_sync(0xffffffffu, g, 31);
        eq_local = __shfl_sync(0xffffffffu, e, 31);
        wg = __shfl_sync(0xffffffffu, g, (warp + 31) & 31);   // inclusive sum of chunks before this warp's
        we = __shfl_sync(0xffffffffu, e, (warp + 31) & 31);
        if (warp == 0) {
            wg = 0u;
            we = 0u;
        }
    }
    if (tid < CL) {
        put(&cnt[rank][0], tid, gt_local);
        put(&cnt[rank][1], tid, eq_local);
    }
    sync_all();
    uint32_t G = 0u, E = 0u;   // keys > v* and == v* before this segment
    for (int r = 0; r < (int)rank; ++r) {
        G += cnt[r][0];
        E += cnt[r][1];
    }

    if (listed && cache) {
        // ---- the candidates above v*, and those equal to it that the budget reaches (in position
        // order: the rank among equal keys before them in the row), join the bitmap
        uint32_t eseen = E + we;
        const uint32_t nwc = wncand[warp];
        for (uint32_t b0 = 0; b0 < nwc; b0 += 32) {
            const uint32_t c = b0 + lane;
            const bool in = c < nwc;
            const uint32_t k = in ? wkey[c] : 0u;
            const bool gt = in && k > vstar;
            const bool eq = in && k == vstar;
            const uint32_t bal = __ballot_sync(0xffffffffu, eq);
            const uint32_t rank = eseen + (uint32_t)__popc(bal & ((1u << lane) - 1u));
            if (gt || (eq && rank < rem)) {
                const uint32_t pos = wpos[c];
                atomicOr(&bm[pos >> 5], 1u << (pos & 31));
            }
            eseen += (uint32_t)__popc(bal);
        }
        __syncthreads();
        // ---- the bitmap in position order: thread t takes words [t q, t q + q)
        const int words = (len + 31) / 32;
        const int q = (words + kTkThreads - 1) / kTkThreads;
        const int w_lo = min(words, tid * q);
        const int w_hi = min(words, w_lo + q);
        uint32_t nsel = 0u;
        for (int wi = w_lo; wi < w_hi; ++wi)
            nsel += (uint32_t)__popc(bm[wi]);
        uint32_t stot;
        uint32_t o = G + min(E, rem) + block_scan<NT>(nsel, wsum, stot) - nsel;
        for (int wi = w_lo; wi < w_hi; ++wi) {
            uint32_t x = bm[wi];
            while (x != 0u) {
                const int bit = __ffs(x) - 1;
                orow[o++] = (int32_t)(lo + 32 * wi + bit);
                x &= x - 1u;
            }
        }
        return;
    }

    // ---- position-ordered compaction over this warp's chunk: the output index of a selected
    // position is (keys > v* before it) + min(keys == v* before it, rem)
    uint32_t gb = G + wg, eb = E + we;   // keys > v* and == v* before this lane's next positions
    for (int s0 = c_lo; s0 < c_hi; s0 += kTkStep) {
        const int i0 = s0 + lane * 8;
        uint32_t keys[8];
        if (cache && i0 + 8 <= c_hi) {
            const uint4 a0 = *reinterpret_cast<const uint4 *>(kc + i0);
            const uint4 a1 = *reinterpret_cast<const uint4 *>(kc + i0 + 4);
            keys[0] = a0.x; keys[1] = a0.y; keys[2] = a0.z; keys[3] = a0.w;
            keys[4] = a1.x; keys[5] = a1.y; keys[6] = a1.z; keys[7] = a1.w;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                keys[j] = i0 + j < c_hi ? key_at(i0 + j) : 0u;
        }
        uint32_t q = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            q += (i0 + j < c_hi && keys[j] > vstar) ? 0x10000u
                                                   : ((i0 + j < c_hi && keys[j] == vstar) ? 1u : 0u);
        uint32_t incl = q;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        const uint32_t step_tot = __shfl_sync(0xffffffffu, incl, 31);
        if (q != 0u) {
            const uint32_t excl = incl - q;
            uint32_t g = gb + (excl >> 16), e = eb + (excl & 0xFFFFu);
#pragma unroll
            for (int j = 0; j < 8; ++j) {   // one predicated store a key: index g + min(e, rem) either way
                const bool in = i0 + j < c_hi;
                const bool gt = in && keys[j] > vstar;
                const bool eq = in && keys[j] == vstar;
                if (gt || (eq && e < rem))
                    orow[g + min(e, rem)] = (int32_t)(lo + i0 + j);
                g += gt ? 1u : 0u;
                e += eq ? 1u : 0u;
            }
        }
        gb += step_tot >> 16;
        eb += step_tot & 0xFFFFu;
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
    if (cluster < 1 || cluster > 8 || top_k < 1 || width < 0)
        return cudaErrorInvalidValue;
    // every segment's keys in shared memory when the longest segment fits the cache
    const long long seg_max = (((long long)width + cluster - 1) / cluster + 3) / 4 * 4;
    const int cache = seg_max <= kTkCacheKeys ? (int)seg_max : 0;
    const int warps = (cluster > 1 ? kTkThreadsCluster : kTkThreadsRow) / 32;
    const int bm_bytes = cache ? 4 * ((cache + 31) / 32) : 0;
    // whole-row CTAs take the longer candidate lists where they fit (a CTA has the SM to itself);
    // clustered CTAs keep the short ones, so that two of them still share an SM
    const int cand = (cluster == 1 && 4 * cache + 8 * kTkCandWarpWide * warps + bm_bytes <= kTkRowDynMax)
                         ? kTkCandWarpWide
                         : kTkCandWarp;
    const int smem = 4 * cache + 8 * cand * warps + bm_bytes;
    const void *kernel = cluster > 1 ? reinterpret_cast<const void *>(topk_select_kernel<kTkThreadsCluster>)
                                     : reinterpret_cast<const void *>(topk_select_kernel<kTkThreadsRow>);
    const int smem_max = 4 * kTkCacheKeys + 8 * kTkCandWarp * 32 + 4 * (kTkCacheKeys / 32);
    cudaError_t e = set_smem_once(kernel, cluster > 1 ? smem_max : (smem_max > kTkRowDynMax ? smem_max : kTkRowDynMax),
                                  cluster > 1 ? kAttrTopkCluster : kAttrTopk);
    if (e != cudaSuccess)
        return e;
    TopkParams p{scores, score_stride, width, num_cand, top_k, out, out_stride, lens, cluster, cache, cand};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)num_tokens * cluster));
    cfg.blockDim = dim3(cluster > 1 ? kTkThreadsCluster : kTkThreadsRow);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 1 : 0;
    void *args[] = {&p};
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

}  // namespace dsv4
