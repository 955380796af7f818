// merge.cu -- log-sum-exp merge of split-KV partial results.
//
// When one (token, head group) is split over several workers, each worker w
// leaves its running max m_w, running sum l_w = sum_{j in w} e^{s_j - m_w} and the
// unnormalised O_w = sum_{j in w} e^{s_j - m_w} v_j.  The merge forms
//   m   = max(max_w m_w, sink)
//   Z   = sum_w l_w e^{m_w - m} + e^{sink - m}     (sink term only when a sink is given)
//   out = (sum_w e^{m_w - m} O_w) / Z  -> BF16,     lse = m + ln Z
// i.e. the softmax normaliser of the whole key set with the sink counted once.
// One CTA of 128 threads per (token, head); each thread owns four output dims.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxSplits = 64;

__global__ void __launch_bounds__(kThreads) merge_kernel(const DecodeParams p)
{
    __shared__ float s_w[kMaxSplits];
    __shared__ float s_f;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // partials from the decode kernel
    const int t = blockIdx.x / p.num_heads;
    const int h = blockIdx.x % p.num_heads;
    const int group = h / p.heads_per_group;
    const int hh = h % p.heads_per_group;
    const int tid = threadIdx.x;
    const int64_t unit0 = ((int64_t)t * p.groups + group) * p.splits;

    if (tid == 0) {
        float m = -INFINITY;
        for (int s = 0; s < p.splits; ++s)
            m = fmaxf(m, p.part_ml[2 * ((unit0 + s) * p.heads_per_group + hh)]);
        const float mk = m;
        float sk = 0.f;
        if (p.sink != nullptr) {
            sk = p.sink[h];
            m = fmaxf(m, sk);
        }
        float z = 0.f;
        for (int s = 0; s < p.splits; ++s) {
            const int64_t slot = (unit0 + s) * p.heads_per_group + hh;
            const float ms = p.part_ml[2 * slot];
            const float ls = p.part_ml[2 * slot + 1];
            const float w = ms == -INFINITY ? 0.f : expf(ms - m);
            s_w[s] = w;
            z += ls * w;
        }
        if (p.sink != nullptr)
            z += expf(sk - m);
        s_f = (z > 0.f && mk != -INFINITY) ? 1.f / z : 0.f;
        if (p.lse != nullptr)
            p.lse[(int64_t)t * p.num_heads + h] = z > 0.f ? m + logf(z) : -INFINITY;
    }
    __syncthreads();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < p.splits; ++s) {
        const float w = s_w[s];
        if (w == 0.f)
            continue;
        const int64_t slot = (unit0 + s) * p.heads_per_group + hh;
        const float4 v = *reinterpret_cast<const float4 *>(p.part_o + slot * kLatent + 4 * tid);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    const float f = s_f;
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc.x * f, acc.y * f);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc.z * f, acc.w * f);
    uint2 u;
    u.x = *reinterpret_cast<const unsigned *>(&a);
    u.y = *reinterpret_cast<const unsigned *>(&b);
    *reinterpret_cast<uint2 *>(p.out + ((int64_t)t * p.num_heads + h) * kLatent + 4 * tid) = u;
}

}  // namespace

int merge_max_splits() { return kMaxSplits; }

cudaError_t launch_merge(const DecodeParams &p, cudaStream_t stream)
{
    if (p.num_tokens <= 0 || p.splits <= 1)
        return cudaSuccess;
    if (p.splits > kMaxSplits)
        return cudaErrorInvalidValue;
    const long long grid = (long long)p.num_tokens * p.num_heads;
    return launch_after_previous(reinterpret_cast<const void *>(merge_kernel), (unsigned)grid, kThreads, 0, stream, p);
}

}  // namespace dsv4
