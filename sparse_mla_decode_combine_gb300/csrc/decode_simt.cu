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
// At 16-32 heads the logits are a thin product (<= 32 x 576 per key) that the
// CUDA cores keep up with; the kernel is bound by the gather.
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

template <int HG>
__global__ void __launch_bounds__(kThreads, 1) decode_simt_kernel(const DecodeParams p)
{
    static_assert(HG == 16 || HG == 32, "head group");
    constexpr int TPH = kThreads / HG;          // threads per head in the P.V stage
    constexpr int NV4 = kLatent / (4 * TPH);    // float4 accumulators per thread
    constexpr int KPL = HG / 8;                 // keys per lane in the logit stage

    extern __shared__ __align__(16) float smem[];
    float *qs = smem;                 // [HG][kRow]
    float *ks = qs + HG * kRow;       // [kTile][kRow]
    float *ss = ks + kTile * kRow;    // [HG][kScoreRow]
    __shared__ long long rowoff[kTile];
    __shared__ float rscale[kTile][4];
    __shared__ float s_alpha[HG], s_m[HG], s_l[HG];

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
    const int row = p.req_idx ? p.req_idx[t] : t;
    const bool row_ok = row >= 0 && row < p.num_reqs;
    if (!row_ok && tid == 0 && kend > kbeg)
        atomicOr(p.status, kStatusBadIndex);

    // Q (BF16) -> fp32 rows
    for (int i = tid; i < HG * (kDim / 8); i += kThreads) {
        const int h = i / (kDim / 8);
        const int c = i % (kDim / 8);
        const uint4 v = *reinterpret_cast<const uint4 *>(p.q + (int64_t)t * p.q_token_stride + (int64_t)(h0 + h) * kDim + 8 * c);
        bf16x8_to_f32(v, qs + h * kRow + 8 * c);
    }
    if (tid < HG) {
        s_m[tid] = -INFINITY;
        s_l[tid] = 0.f;
    }
    const int ph = tid / TPH;   // head of this thread in the P.V stage
    const int pg = tid % TPH;
    float4 acc[NV4];
#pragma unroll
    for (int i = 0; i < NV4; ++i)
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();

    for (int k0 = kbeg; k0 < kend; k0 += kTile) {
        const int nk = min(kTile, kend - k0);
        // 1. logical position -> cache byte offset, and the row's four scales
        if (tid < kTile) {
            long long off = -1;
            if (tid < nk && row_ok) {
                const int idx = p.combined[(int64_t)t * p.cw + k0 + tid];
                const int blk = idx >= 0 ? idx / p.page : -1;
                int phys = -1;
                if (idx >= 0 && blk < p.max_blocks)
                    phys = p.block_table[(int64_t)row * p.bt_stride + blk];
                if (phys >= 0 && phys < p.num_blocks)
                    off = ((long long)phys * p.page + (idx - blk * p.page)) * kEntryBytes;
                else
                    atomicOr(p.status, kStatusBadIndex);
            }
            rowoff[tid] = off;
            unsigned sw = 0;
            if (off >= 0)
                sw = __ldg(reinterpret_cast<const unsigned *>(p.kv + off + kScaleOffset));
#pragma unroll
            for (int b = 0; b < 4; ++b)
                rscale[tid][b] = ue8m0_to_float((sw >> (8 * b)) & 0xFFu);
        }
        __syncthreads();
        // 2. gather + dequantise: 40 data chunks of 16 bytes per row (32 latent, 8 rope)
        for (int c = tid; c < kTile * 40; c += kThreads) {
            const int r = c / 40;
            const int j = c % 40;
            const long long off = rowoff[r];
            float *dst = ks + r * kRow + (j < 32 ? 16 * j : kLatent + 8 * (j - 32));
            const int nv = j < 32 ? 16 : 8;
            if (off < 0) {
                for (int e = 0; e < nv; e += 4)
                    *reinterpret_cast<float4 *>(dst + e) = make_float4(0.f, 0.f, 0.f, 0.f);
                continue;
            }
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.kv + off + 16 * j));
            if (j < 32)
                e4m3x16_to_f32(v, rscale[r][j >> 3], dst);
            else
                bf16x8_to_f32(v, dst);
        }
        __syncthreads();
        // 3. logits: lane -> head, each lane KPL keys of this warp's four
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
                ss[h * kScoreRow + j] = (j < nk && rowoff[j] >= 0) ? a[k] * p.scale : -INFINITY;
            }
        }
        __syncthreads();
        // 4. online softmax update, one thread per head
        if (tid < HG) {
            float *sr = ss + tid * kScoreRow;
            const float mo = s_m[tid];
            float mt = -INFINITY;
            for (int j = 0; j < kTile; ++j)
                mt = fmaxf(mt, sr[j]);
            const float mn = fmaxf(mo, mt);
            float alpha = 1.f;
            float sum = 0.f;
            if (mn == -INFINITY) {
                for (int j = 0; j < kTile; ++j)
                    sr[j] = 0.f;
            } else {
                alpha = expf(mo - mn);
                for (int j = 0; j < kTile; ++j) {
                    const float e = expf(sr[j] - mn);
                    sr[j] = e;
                    sum += e;
                }
            }
            s_l[tid] = s_l[tid] * alpha + sum;
            s_m[tid] = mn;
            s_alpha[tid] = alpha;
        }
        __syncthreads();
        // 5. O = alpha * O + P.V
        {
            const float al = s_alpha[ph];
#pragma unroll
            for (int i = 0; i < NV4; ++i) {
                acc[i].x *= al;
                acc[i].y *= al;
                acc[i].z *= al;
                acc[i].w *= al;
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
    const float m = s_m[ph];
    const float l = s_l[ph];
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
