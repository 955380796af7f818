// insert.cu -- fused Q per-head RMSNorm + GPT-J RoPE + FP8/UE8M0 KV-cache insert: the step that
// runs before the decode ("feat: add DeepSeek-V4 XPU attention decode path", vllm #42953,
// 实现拆解 4: xpu_qnorm_rope_kv_fp8_insert, called from forward_mqa with q, kv, kv_cache,
// slot_mapping and positions).  The page names the steps; this kernel computes:
//   q_out[t][h] = RoPE_pos(q[t][h] / sqrt(mean(q[t][h]^2) + eps) * w)      (576 dims, one rounding)
//   kv_cache[slot_mapping[t]] = the 656-byte entry of kv[t]: per 128 latent values the smallest
//       UE8M0 exponent e with 448 * 2^e >= amax, E4M3 codes of x * 2^-e (nearest, ties to even),
//       the GPT-J-rotated rope part in BF16, zero padding
// where GPT-J RoPE rotates the interleaved pairs (512 + 2i, 513 + 2i) by the angle whose cosine
// and sine are cos_sin[pos][i] and cos_sin[pos][32 + i].  A negative slot writes nothing; a slot
// past the cache or a position outside the table writes nothing and sets the bad-index bit (the
// query is then normalised but not rotated).
//
// One CTA per token: warps 0..15 take the query heads, four at a time (their loads all in flight
// before any use), lane l holding the BF16 pairs l + 32 j (j < 9; j = 8 is the rope part, pair
// i = l) so a pair never leaves its lane; warp 16 builds the cache entry.  fp32 arithmetic
// throughout, IEEE division and square root.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kInsQWarps = 16;
constexpr int kInsHeadsIter = 4;   // heads a warp has in flight at once
constexpr int kInsThreads = 32 * (kInsQWarps + 1);
constexpr int kPairs = kDim / 2;   // 288 BF16 pairs per head; pairs 256.. are the rope part

struct InsertParams {
    const uint32_t *q;          // BF16 pairs
    int64_t q_stride;           // pairs per token
    uint32_t *q_out;
    int64_t q_out_stride;
    int32_t num_heads;
    const float *norm_w;        // [576] or null
    float eps;
    const uint32_t *kv;         // BF16 pairs [T][288]
    int64_t kv_stride;          // pairs per token
    const int64_t *positions;
    const int64_t *slots;
    const float *cos_sin;       // [max_pos][64]
    int32_t max_pos;
    uint8_t *cache;
    int64_t num_slots;
    unsigned *status;
};

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v)
{
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t pack_rn_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Smallest integer e with 448 * 2^e >= amax (0 for amax 0), clamped to [-127, 127].  For
// amax in [2^k, 2^(k+1)) the answer is k - 8 or k - 7; one exact comparison decides.
__device__ __forceinline__ int ue8m0_exponent(float amax)
{
    if (!(amax > 0.f))
        return 0;
    int e = ilogbf(amax) - 8;
    if (ldexpf(448.f, e) < amax)
        ++e;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

__global__ void __launch_bounds__(kInsThreads) qnorm_rope_kv_insert_kernel(const InsertParams p)
{
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t pos = p.positions[t];
    const bool rot = pos >= 0 && pos < p.max_pos;
    float c = 1.f, s = 0.f;   // this lane's rope pair i = lane
    if (rot) {
        c = __ldg(p.cos_sin + pos * 64 + lane);
        s = __ldg(p.cos_sin + pos * 64 + 32 + lane);
    } else if (threadIdx.x == 0) {
        atomicOr(p.status, kStatusBadIndex);
    }

    if (warp < kInsQWarps) {
        float w[18];   // the norm weight of this lane's 18 dims (pairs lane + 32 j)
#pragma unroll
        for (int j = 0; j < 9; ++j) {
            const int d = 2 * (lane + 32 * j);
            w[2 * j] = p.norm_w ? __ldg(p.norm_w + d) : 1.f;
            w[2 * j + 1] = p.norm_w ? __ldg(p.norm_w + d + 1) : 1.f;
        }
        for (int h0 = warp; h0 < p.num_heads; h0 += kInsHeadsIter * kInsQWarps) {
            uint32_t x[kInsHeadsIter][9];
#pragma unroll
            for (int k = 0; k < kInsHeadsIter; ++k) {   // every head's loads in flight before any use
                const int h = h0 + k * kInsQWarps;
                const uint32_t *a = p.q + t * p.q_stride + (int64_t)h * kPairs;
#pragma unroll
                for (int j = 0; j < 9; ++j)
                    x[k][j] = h < p.num_heads ? __ldg(a + lane + 32 * j) : 0u;
            }
#pragma unroll
            for (int k = 0; k < kInsHeadsIter; ++k) {
                const int h = h0 + k * kInsQWarps;
                if (h >= p.num_heads)
                    break;
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < 9; ++j) {
                    const float2 v = unpack_bf16x2(x[k][j]);
                    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, ss));
                }
                ss = warp_sum(ss);
                const float r = 1.f / sqrtf(ss / (float)kDim + p.eps);
                uint32_t *o = p.q_out + t * p.q_out_stride + (int64_t)h * kPairs;
#pragma unroll
                for (int j = 0; j < 9; ++j) {
                    const float2 v = unpack_bf16x2(x[k][j]);
                    float y0 = v.x * r * w[2 * j], y1 = v.y * r * w[2 * j + 1];
                    if (j == 8) {
                        const float u0 = y0 * c - y1 * s;
                        const float u1 = y0 * s + y1 * c;
                        y0 = u0;
                        y1 = u1;
                    }
                    o[lane + 32 * j] = pack_rn_bf16x2(y0, y1);
                }
            }
        }
        return;
    }

    // ---- warp 16: the cache entry of this token's key
    const int64_t slot = p.slots[t];
    if (slot < 0)
        return;
    if (slot >= p.num_slots || !rot) {   // (a bad position was flagged above)
        if (lane == 0 && slot >= p.num_slots)
            atomicOr(p.status, kStatusBadIndex);
        return;
    }
    uint32_t x[9];
#pragma unroll
    for (int j = 0; j < 9; ++j)
        x[j] = __ldg(p.kv + t * p.kv_stride + lane + 32 * j);
    uint8_t *e = p.cache + slot * kEntryBytes;
    uint32_t scales = 0u;
#pragma unroll
    for (int b = 0; b < 4; ++b) {   // latent block b = pairs 64 b .. 64 b + 63 = j in {2 b, 2 b + 1}
        const float2 v0 = unpack_bf16x2(x[2 * b]), v1 = unpack_bf16x2(x[2 * b + 1]);
        const float amax = warp_max(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v1.x), fabsf(v1.y))));
        const int ex = ue8m0_exponent(amax);
        scales |= (uint32_t)(ex + 127) << (8 * b);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const float2 v = jj == 0 ? v0 : v1;
            const __nv_fp8x2_storage_t codes =
                __nv_cvt_float2_to_fp8x2(make_float2(ldexpf(v.x, -ex), ldexpf(v.y, -ex)), __NV_SATFINITE, __NV_E4M3);
            *reinterpret_cast<uint16_t *>(e + 2 * (lane + 32 * (2 * b + jj))) = (uint16_t)codes;
        }
    }
    {
        const float2 v = unpack_bf16x2(x[8]);
        const float u0 = v.x * c - v.y * s;
        const float u1 = v.x * s + v.y * c;
        *reinterpret_cast<uint32_t *>(e + kRopeOffset + 4 * lane) = pack_rn_bf16x2(u0, u1);
    }
    if (lane < 4)   // scale bytes, then the 12 padding bytes
        *reinterpret_cast<uint32_t *>(e + kScaleOffset + 4 * lane) = lane == 0 ? scales : 0u;
}

}  // namespace

cudaError_t launch_qnorm_rope_kv_insert(const void *q, int64_t q_stride, void *q_out, int64_t q_out_stride,
                                        int num_tokens, int num_heads, const float *norm_w, float eps,
                                        const void *kv, int64_t kv_stride, const int64_t *positions,
                                        const int64_t *slots, const float *cos_sin, int max_pos, void *cache,
                                        int64_t num_slots, unsigned *status, cudaStream_t stream)
{
    if (num_tokens <= 0)
        return cudaSuccess;
    InsertParams p{reinterpret_cast<const uint32_t *>(q),
                   q_stride / 2,
                   reinterpret_cast<uint32_t *>(q_out),
                   q_out_stride / 2,
                   num_heads,
                   norm_w,
                   eps,
                   reinterpret_cast<const uint32_t *>(kv),
                   kv_stride / 2,
                   positions,
                   slots,
                   cos_sin,
                   max_pos,
                   reinterpret_cast<uint8_t *>(cache),
                   num_slots,
                   status};
    qnorm_rope_kv_insert_kernel<<<num_tokens, kInsThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dsv4
