// decode_simt.cu -- CUDA-core sparse-MLA decode for low head counts (16 or 32 heads per worker).
//
// One CTA (256 threads) handles one (token, head group, split): a contiguous
// range of the token's combined index list.  Per tile of 32 keys it
//   1. turns logical positions into cache byte offsets through the block table
//      (the per-request logical -> physical conversion of "Enable DeepSeek V4 and
//      GLM-5.1 on SM120", vllm #43477, flashinfer_mla_sparse_sm120.py),
//   2. gathers the 656-byte entries with 16-byte loads and dequantises them
//      (latent = e4m3 * 2^(ue8m0 - 127), rope = BF16 as stored; the dequant of
//      "feat: add DeepSeek-V4 XPU attention decode path", vllm #42953,
//      _dequant_gather_slots_kernel) into fp32 shared memory,
//   3. computes the head x key logits on CUDA cores, updates an online softmax
//      (running max / running sum per head) and accumulates P.V in registers.
// At the end it either normalises (one split: sink folded into the normaliser,
// BF16 out, natural-log LSE) or stores the unnormalised partial for the merge.
// The cache slots of tile i + 2 are resolved, and the raw entries of tile i + 1 loaded into
// registers, while tile i is computed; the softmax runs on all threads (the threads of a head
// are one group of lanes and keep its running max and sum in registers).  Each key costs
// 2 * 16..32 * 1088 fp32 FLOPs against 656 bytes: on CUDA cores the kernel is bound by the
// FMA rate, not by the gather.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;        // keys per tile
constexpr int kRow = 580;        // padded fp32 row (576 + 4): conflict-free per-head row reads
constexpr int kScoreRow = kTile + 1;

__device__ __forceinline__ float ue8m0_to_float(unsigned e)
{
    // 2^(e - 127): the float with exponent field e (e = 0 gives the subnormal 2^-127)
    if (e == 0xFFu)
        return __int_as_float(0x7FC00000);
    if (e == 0u)
        return __int_as_float(0x00400000);
    return __int_as_float((int)(e << 23));
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float *dst)
{
    const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f;
        f.x = __uint_as_float(w[i] << 16);
        f.y = __uint_as_float(w[i] & 0xFFFF0000u);
        *reinterpret_cast<float2 *>(dst + 2 * i) = f;
    }
}

__device__ __forceinline__ void e4m3x16_to_f32(const uint4 v, float scale, float *dst)
{
    const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFFu), __NV_E4M3);
        const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
        const float2 a = __half22float2(__half2(lo));
        const float2 b = __half22float2(__half2(hi));
        float4 f;
        f.x = a.x * scale;
        f.y = a.y * scale;
        f.z = b.x * scale;
        f.w = b.y * scale;
        *reinterpret_cast<float4 *>(dst + 4 * i) = f;
    }
}

// Cache slot of logical position idx of block-table row `row` (-1, and the bad-index bit in the
// status word, when the position or its page is outside the table or the cache).
__device__ __forceinline__ int slot_of(const DecodeParams &p, int row, int idx, int phys)
{
    if (idx < 0 || phys < 0 || phys >= p.num_blocks) {
        atomicOr(p.status, kStatusBadIndex);
        return -1;
    }
    return phys * p.page + (idx - (idx / p.page) * p.page);
}

__device__ __forceinline__ int page_of(const DecodeParams &p, int row, int idx)
{
    const int blk = idx >= 0 ? idx / p.page : -1;
    return (idx >= 0 && blk < p.max_blocks) ? __ldg(p.block_table + (int64_t)row * p.bt_stride + blk) : -1;
}

template <int HG>
__global__ void __launch_bounds__(kThreads, 1) decode_simt_kernel(const DecodeParams p)
{
    static_assert(HG == 16 || HG == 32, "head group");
    constexpr int TPH = kThreads / HG;          // threads per head in the softmax and P.V stages
    constexpr int NV4 = kLatent / (4 * TPH);    // float4 accumulators per thread
    constexpr int KPL = HG / 8;                 // keys per lane in the logit stage
    constexpr int KPT = kTile / TPH;            // keys per thread in the softmax
    constexpr int kPieces = 40;                 // 16-byte data pieces of an entry (32 latent, 8 rope)
    constexpr int kLoads = kTile * kPieces / kThreads;
    static_assert(kTile * kPieces % kThreads == 0, "gather pieces per thread");

    extern __shared__ __align__(16) float smem[];
    float *qs = smem;                 // [HG][kRow]
    float *ks = qs + HG * kRow;       // [kTile][kRow]
    float *ss = ks + kTile * kRow;    // [HG][kScoreRow]
    __shared__ int ring[3][kTile];    // cache slots of tiles i, i+1, i+2 (slot -1: no key)

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int unit = blockIdx.x;
    const int split = unit % p.splits;
    const int group = (unit / p.splits) % p.groups;
    const int t = unit / (p.splits * p.groups);
    const int h0 = group * HG;

    asm volatile("griddepcontrol.wait;" ::: "memory");   // combined lists from the combine kernel
    const int L = p.lens[t];
    const int kbeg = split * p.chunk;
    const int kend = min(L, kbeg + p.chunk);
    const int ntiles = kend > kbeg ? (kend - kbeg + kTile - 1) / kTile : 0;
    const int row = p.req_idx ? p.req_idx[t] : t;
    const bool row_ok = row >= 0 && row < p.num_reqs;
    if (!row_ok && tid == 0 && kend > kbeg)
        atomicOr(p.status, kStatusBadIndex);
    const int32_t *crow = p.combined + (int64_t)t * p.cw;

    // slots of tiles 0 and 1 (one round trip through the combined list and the block table)
    if (tid < 2 * kTile) {
        const int k = kbeg + tid;
        int sl = -1;
        if (row_ok && k < kend) {
            const int idx = crow[k];
            sl = slot_of(p, row, idx, page_of(p, row, idx));
        }
        ring[tid / kTile][tid % kTile] = sl;
    }
    // Q (BF16) -> fp32 rows
    for (int i = tid; i < HG * (kDim / 8); i += kThreads) {
        const int h = i / (kDim / 8);
        const int c = i % (kDim / 8);
        const uint4 v = *reinterpret_cast<const uint4 *>(p.q + (int64_t)t * p.q_token_stride + (int64_t)(h0 + h) * kDim + 8 * c);
        bf16x8_to_f32(v, qs + h * kRow + 8 * c);
    }
    const int ph = tid / TPH;   // head of this thread in the softmax and P.V stages
    const int pg = tid % TPH;
    float m_run = -INFINITY, l_run = 0.f;   // the head's running max and row sum (same in its TPH threads)
    float4 acc[NV4];
#pragma unroll
    for (int i = 0; i < NV4; ++i)
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();

    // the raw pieces of the next tile, in registers: piece c = tid + kThreads u is piece c % 40 of row c / 40
    uint4 raw[kLoads];
    unsigned rsc[kLoads];
    auto load_tile = [&](const int *sl) {
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
            const int c = tid + kThreads * u;
            const int s = sl[c / kPieces];
            const int j = c % kPieces;
            raw[u] = make_uint4(0u, 0u, 0u, 0u);
            rsc[u] = 0u;
            if (s >= 0) {
                const uint8_t *e = p.kv + (int64_t)s * kEntryBytes;
                raw[u] = __ldg(reinterpret_cast<const uint4 *>(e + 16 * j));
                if (j < 32)
                    rsc[u] = __ldg(reinterpret_cast<const unsigned *>(e + kScaleOffset));
            }
        }
    };
    if (ntiles > 0)
        load_tile(ring[0]);

    for (int it = 0; it < ntiles; ++it) {
        const int k0 = kbeg + it * kTile;
        const int nk = min(kTile, kend - k0);
        const int *sl = ring[it % 3];
        // tile it + 2: its positions now, its pages after the dequant, its slots after the logits
        int idx2 = -1, pg2 = -1;
        const bool has2 = warp == 0 && row_ok && k0 + 2 * kTile + lane < kend;
        if (has2)
            idx2 = crow[k0 + 2 * kTile + lane];
        // 1. dequantise the registers into the key tile (rows without a key are zeros)
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
            const int c = tid + kThreads * u;
            const int r = c / kPieces;
            const int j = c % kPieces;
            float *dst = ks + r * kRow + (j < 32 ? 16 * j : kLatent + 8 * (j - 32));
            if (j < 32)
                e4m3x16_to_f32(raw[u], ue8m0_to_float((rsc[u] >> (8 * (j >> 3))) & 0xFFu), dst);
            else
                bf16x8_to_f32(raw[u], dst);
        }
        if (has2)
            pg2 = page_of(p, row, idx2);
        __syncthreads();
        if (it + 1 < ntiles)
            load_tile(ring[(it + 1) % 3]);
        // 2. logits: lane -> head, each lane KPL keys of this warp's four
        {
            const int h = lane % HG;
            const int kb = 4 * warp + (lane / HG) * KPL;
            const float *qr = qs + h * kRow;
            float a[KPL];
#pragma unroll
            for (int k = 0; k < KPL; ++k)
                a[k] = 0.f;
#pragma unroll 4
            for (int d = 0; d < kDim; d += 4) {
                const float4 qv = *reinterpret_cast<const float4 *>(qr + d);
#pragma unroll
                for (int k = 0; k < KPL; ++k) {
                    const float4 kv = *reinterpret_cast<const float4 *>(ks + (kb + k) * kRow + d);
                    a[k] = fmaf(qv.x, kv.x, a[k]);
                    a[k] = fmaf(qv.y, kv.y, a[k]);
                    a[k] = fmaf(qv.z, kv.z, a[k]);
                    a[k] = fmaf(qv.w, kv.w, a[k]);
                }
            }
#pragma unroll
            for (int k = 0; k < KPL; ++k) {
                const int j = kb + k;
                ss[h * kScoreRow + j] = (j < nk && sl[j] >= 0) ? a[k] * p.scale : -INFINITY;
            }
        }
        if (warp == 0 && k0 + 2 * kTile < kend)   // ring slot of tile it - 1, done with
            ring[(it + 2) % 3][lane] = has2 ? slot_of(p, row, idx2, pg2) : -1;
        __syncthreads();
        // 3. online softmax: the TPH threads of head ph (one warp) take KPT keys each
        {
            float *sr = ss + ph * kScoreRow + pg * KPT;
            float sv[KPT];
            float mt = -INFINITY;
#pragma unroll
            for (int u = 0; u < KPT; ++u) {
                sv[u] = sr[u];
                mt = fmaxf(mt, sv[u]);
            }
#pragma unroll
            for (int o = TPH / 2; o > 0; o >>= 1)
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
            const float mn = fmaxf(m_run, mt);
            float alpha = 1.f, sum = 0.f;
            if (mn != -INFINITY) {
                alpha = expf(m_run - mn);
#pragma unroll
                for (int u = 0; u < KPT; ++u) {
                    const float e = expf(sv[u] - mn);
                    sr[u] = e;
                    sum += e;
                }
            } else {
#pragma unroll
                for (int u = 0; u < KPT; ++u)
                    sr[u] = 0.f;
            }
#pragma unroll
            for (int o = TPH / 2; o > 0; o >>= 1)
                sum += __shfl_xor_sync(0xffffffffu, sum, o);
            l_run = l_run * alpha + sum;
            m_run = mn;
            __syncwarp();
            // 4. O = alpha * O + P.V
#pragma unroll
            for (int i = 0; i < NV4; ++i) {
                acc[i].x *= alpha;
                acc[i].y *= alpha;
                acc[i].z *= alpha;
                acc[i].w *= alpha;
            }
            const float *pr = ss + ph * kScoreRow;
            for (int j = 0; j < nk; ++j) {
                const float pj = pr[j];
                const float *vr = ks + j * kRow + 4 * pg;
#pragma unroll
                for (int i = 0; i < NV4; ++i) {
                    const float4 v = *reinterpret_cast<const float4 *>(vr + 4 * TPH * i);
                    acc[i].x = fmaf(pj, v.x, acc[i].x);
                    acc[i].y = fmaf(pj, v.y, acc[i].y);
                    acc[i].z = fmaf(pj, v.z, acc[i].z);
                    acc[i].w = fmaf(pj, v.w, acc[i].w);
                }
            }
        }
        __syncthreads();
    }

    const int h = h0 + ph;
    const float m = m_run;
    const float l = l_run;
    if (p.splits == 1) {
        float mf = m;
        float lf = l;
        if (p.sink != nullptr) {
            const float sk = p.sink[h];
            mf = fmaxf(m, sk);
            lf = (m == -INFINITY ? 0.f : l * expf(m - mf)) + expf(sk - mf);
        }
        const float f = (lf > 0.f && m != -INFINITY) ? expf(m - mf) / lf : 0.f;
        uint16_t *o = p.out + ((int64_t)t * p.num_heads + h) * kLatent + 4 * pg;
#pragma unroll
        for (int i = 0; i < NV4; ++i) {
            const __nv_bfloat162 a = __floats2bfloat162_rn(acc[i].x * f, acc[i].y * f);
            const __nv_bfloat162 b = __floats2bfloat162_rn(acc[i].z * f, acc[i].w * f);
            uint2 u;
            u.x = *reinterpret_cast<const unsigned *>(&a);
            u.y = *reinterpret_cast<const unsigned *>(&b);
            *reinterpret_cast<uint2 *>(o + 4 * TPH * i) = u;
        }
        if (pg == 0 && p.lse != nullptr)
            p.lse[(int64_t)t * p.num_heads + h] = lf > 0.f ? mf + logf(lf) : -INFINITY;
    } else {
        const int64_t slot = ((int64_t)unit * HG + ph);
        float *o = p.part_o + slot * kLatent + 4 * pg;
#pragma unroll
        for (int i = 0; i < NV4; ++i)
            *reinterpret_cast<float4 *>(o + 4 * TPH * i) = acc[i];
        if (pg == 0) {
            p.part_ml[2 * slot] = m;
            p.part_ml[2 * slot + 1] = l;
        }
    }
}

template <int HG>
cudaError_t launch_simt(const DecodeParams &p, cudaStream_t stream)
{
    const size_t smem = sizeof(float) * ((size_t)HG * kRow + (size_t)kTile * kRow + (size_t)HG * kScoreRow);
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(decode_simt_kernel<HG>), (int)smem,
                                  HG == 16 ? kAttrSimt16 : kAttrSimt32);
    if (e != cudaSuccess)
        return e;
    const long long grid = (long long)p.num_tokens * p.groups * p.splits;
    return launch_after_previous(reinterpret_cast<const void *>(decode_simt_kernel<HG>), (unsigned)grid, kThreads,
                                 smem, stream, p);
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeParams &p, cudaStream_t stream)
{
    if (p.num_tokens <= 0)
        return cudaSuccess;
    if (p.heads_per_group == 16)
        return launch_simt<16>(p, stream);
    if (p.heads_per_group == 32)
        return launch_simt<32>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace dsv4
