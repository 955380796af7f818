// decode_tc.cu -- tensor-core (tcgen05 / TMEM) sparse-MLA decode, 64 heads per CTA.
//
// Operation (per token t, head h, over the token's combined key list K_t):
//   s_p = scale * q_h . k_p  (576 dims),  out_h = sum_p softmax(s)_p v_p  (512 dims)
// with the gather/dequant of "feat: add DeepSeek-V4 XPU attention decode path"
// (vllm #42953, _dequant_gather_slots_kernel: value = e4m3 * 2^(ue8m0 - 127), rope
// as stored) and the per-request block-table conversion and [T, h, 512] output of
// "Enable DeepSeek V4 and GLM-5.1 on SM120" (vllm #43477, flashinfer_mla_sparse_sm120.py).
//
// Shape of the contraction.  All heads share one key set (MQA), so a token is a
// pair of dense products: S = Q K^T (64 x 576 x keys) and O = P V (64 x keys x 512).
// With 64 heads the head dimension is too short to fill a 128-row tcgen05 tile, so
// both products run transposed, keys and value dims on the M side:
//   S^T[128 keys x 64 heads]   = K_tile[128 x 576] . Q^T          (A = K tile, K-major)
//   O^T[128 dv x 64 heads] += V^T[128 dv x 128 keys] . P^T        (A = K tile, MN-major)
// One BF16 K tile in shared memory (128-byte swizzle, 8-row atoms, 64-dim column
// chunks) is read by both: as K-major A for S^T (rows = keys) and, without any
// copy, as MN-major A for O^T (rows of the same atoms = keys along K, the 64
// contiguous dims along M).  S^T, O^T (four 128-dv tiles) and per-lane partial row
// sums live in TMEM (512 columns).
//
// CTA = 512 threads, one (token, 64-head group, split):
//   warp 0       tcgen05.alloc/dealloc; lane 0 issues the MMAs and commits
//   warps 1-15   workers: 16-byte streaming loads of the next block's entries into
//                registers while the current block computes, then the exact dequant
//                (E4M3 -> f16 -> f32 * 2^(e-127) -> BF16) into the swizzled K tile;
//                warps 1-3 also look up cache slots two blocks ahead
//   warps 4-11   also the softmax: lane i of a warp owns TMEM lane i of its quadrant
//                (key i of the block in S^T, a value dim in O^T), two warps per
//                quadrant split the 64 heads; per-head block maxima with
//                redux.sync.max.f32, lazy rescaling (only when a head's max grows by
//                more than 2^8), P^T (BF16) into shared memory, row sums in TMEM
// When a token's keys are split over S CTAs (S <= 8), the S CTAs form a thread-block
// cluster: each stages its partial in its own shared memory and, after a cluster
// barrier, every CTA merges a slice of the heads by reading its peers' partials
// through distributed shared memory.
// Every mbarrier wait is bounded; a wait that runs out records DSV4_ERR_TIMEOUT in
// the status word and the CTA finishes without waiting again.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kThreads = 512;
constexpr int kBK = 128;                 // keys per block = MMA M
constexpr int kNH = 64;                  // heads per CTA = MMA N
constexpr int kChunks = 9;               // 576 dims / 64
constexpr int kQBytes = kChunks * kNH * 128;     // 73728
constexpr int kKBytes = kChunks * kBK * 128;     // 147456
constexpr int kChunkBytes = kBK * 128;           // 16384 (one 64-dim column chunk of the K tile)
constexpr int kQChunkBytes = kNH * 128;          // 8192
constexpr int kWorkers = 480;                    // warps 1-15: loads + dequant (and softmax on warps 4-11)
constexpr int kDataPieces = 40;                  // 16-byte pieces per entry holding data (32 latent + 8 rope)
constexpr int kRowGroups = kWorkers / kDataPieces;     // 12: worker w owns piece w % 40 of rows w / 40 + 12 i
constexpr int kRowsPerLoader = (kBK + kRowGroups - 1) / kRowGroups;   // 11
constexpr int kSoftWarps = 8;            // two per TMEM lane quadrant, 32 heads each
constexpr int kSoftThreads = 32 * kSoftWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;            // S^T: 64 columns
constexpr uint32_t kColO = 64;           // O^T: 4 tiles x 64 columns
constexpr uint32_t kColL = 320;          // per-lane partial row sums: 64 columns
constexpr float kRescaleLog2 = 8.0f;
constexpr long long kWaitCycles = 4000000000LL;
constexpr int kMaxSplits = 8;            // portable cluster size

// small shared region (after Q and the K tile)
constexpr int kOffSlots = 0;             // int [3][128]
constexpr int kOffScale = 1536;          // uint [128]
constexpr int kOffRed = 2048;            // float [4][64]
constexpr int kOffMrun = 3072;           // float [64]
constexpr int kOffMc = 3328;             // float [64]
constexpr int kOffAlpha = 3584;          // float [64]
constexpr int kOffFin = 3840;            // float [64]
constexpr int kOffBars = 4096;           // u64 [3]
constexpr int kOffTmem = 4128;           // u32
constexpr int kOffFlags = 4136;          // int [2]
constexpr int kSmallBytes = 4160;
constexpr int kSmemBytes = kQBytes + kKBytes + kSmallBytes + 1024;   // + alignment slack
constexpr int kQLoads = kNH * (kDim / 8) / kThreads;                 // 9 16-byte Q pieces per thread

// instruction descriptors (kind::f16): D f32, A/B bf16, M = 128, N = 64
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kNH >> 3) << 17) |
                                ((uint32_t)(kBK >> 4) << 24);
constexpr uint32_t kIdescQK = kIdescBase;                           // A, B K-major
constexpr uint32_t kIdescPV = kIdescBase | (1u << 15) | (1u << 16);  // A, B MN-major

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// byte offset of 16-byte unit u (0..7) of row r inside a 128-byte-swizzled [rows x 128 B] region
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t u)
{
    return (r >> 3) * 1024u + (r & 7u) * 128u + ((u ^ (r & 7u)) << 4);
}

// shared-memory matrix descriptor: 128-byte swizzle, fixed version bits for tcgen05
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// try_wait with a suspend-time hint: the thread sleeps until the phase completes or the
// hint (ns) elapses, instead of spinning on shared memory
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity), "r"(200000u)
                 : "memory");
    return ok != 0;
}

// Bounded wait on one phase of an mbarrier by a single thread.  After any timeout in
// the CTA (abort flag set) waits return at once, so the CTA still reaches its end.
__device__ __forceinline__ void mbar_wait_one(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              unsigned *status)
{
    if (*abort_flag)
        return;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitCycles) {
            *abort_flag = 1;
            atomicOr(status, kStatusTimeout);
            return;
        }
        if (*abort_flag)
            return;
    }
}

// Warp-wide wait: lane 0 polls, the warp then proceeds together.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned *status)
{
    if ((threadIdx.x & 31) == 0)
        mbar_wait_one(bar, parity, abort_flag, status);
    __syncwarp();
}

__device__ __forceinline__ void named_bar(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float warp_max(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ float ue8m0_to_float(unsigned e)
{
    if (e == 0xFFu)
        return __int_as_float(0x7FC00000);
    if (e == 0u)
        return __int_as_float(0x00400000);
    return __int_as_float((int)(e << 23));
}

// two E4M3 codes (low byte = first element) -> BF16x2 of code * scale (exact for in-range values)
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two, float scale)
{
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    const float2 f = __half22float2(__half2(hr));
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y * scale), "f"(f.x * scale));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint16_t bf16_bits(float v)
{
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<const uint16_t *>(&b);
}

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- thread-block cluster: the splits of one (token, head group) merge over distributed shared memory
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Split-KV merge inside a cluster of S = splits CTAs (one per split of a token's keys).
// Every CTA has staged, in its own shared memory, its running max m_s (natural-log
// units, s_m[h]) and row sum l_s (s_l[h]) per head and its unnormalised O_s as fp32
// [64 heads][512] (s_o).  After a cluster barrier the CTA of rank r merges heads
// [r*hp, (r+1)*hp) (hp = ceil(64 / S)), reading all S partials through distributed
// shared memory with the loads of all splits in flight together:
//   m = max(max_s m_s, sink), Z = sum_s l_s e^{m_s - m} + e^{sink - m},
//   out = sum_s e^{m_s - m} O_s / Z  (BF16),  lse = m + ln Z.
__device__ void cluster_merge_pull(const DecodeParams &p, int t, int h0, int rank, uint32_t s_m, uint32_t s_l,
                                   uint32_t s_o, float *wts)
{
    const int S = p.splits;
    const int hp = (kNH + S - 1) / S;
    const int hb = rank * hp;
    const int he = min(kNH, hb + hp);
    const int tid = threadIdx.x;
    if (tid < he - hb) {
        const int h = hb + tid;
        float ms[kMaxSplits], ls[kMaxSplits];
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s) {
            ms[s] = s < S ? ld_cluster_f32(map_to_rank(s_m + 4u * h, s)) : -INFINITY;
            ls[s] = s < S ? ld_cluster_f32(map_to_rank(s_l + 4u * h, s)) : 0.f;
        }
        float m = -INFINITY;
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s)
            m = fmaxf(m, ms[s]);
        const float mk = m;
        float sk = 0.f;
        if (p.sink != nullptr) {
            sk = p.sink[h0 + h];
            m = fmaxf(m, sk);
        }
        float z = 0.f;
        float w[kMaxSplits];
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s) {
            w[s] = ms[s] == -INFINITY ? 0.f : expf(ms[s] - m);
            z += ls[s] * w[s];
        }
        if (p.sink != nullptr)
            z += expf(sk - m);
        const float f = (z > 0.f && mk != -INFINITY) ? 1.f / z : 0.f;
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s)
            wts[tid * 10 + s] = w[s] * f;
        wts[tid * 10 + 8] = z > 0.f ? m + logf(z) : -INFINITY;
    }
    __syncthreads();
    uint32_t peer[kMaxSplits];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s)
        peer[s] = s < S ? map_to_rank(s_o, s) : 0u;
    for (int i = tid; i < (he - hb) * (kLatent / 4); i += kThreads) {
        const int hl = i / (kLatent / 4);
        const int c = i % (kLatent / 4);
        const uint32_t off = (uint32_t)((hb + hl) * kLatent + 4 * c) * 4u;
        float4 v[kMaxSplits];
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s)
            v[s] = (s < S && wts[hl * 10 + s] != 0.f) ? ld_cluster_v4(peer[s] + off) : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s) {
            const float ws = wts[hl * 10 + s];
            acc.x = fmaf(ws, v[s].x, acc.x);
            acc.y = fmaf(ws, v[s].y, acc.y);
            acc.z = fmaf(ws, v[s].z, acc.z);
            acc.w = fmaf(ws, v[s].w, acc.w);
        }
        uint2 u;
        u.x = pack_bf16x2(acc.x, acc.y);
        u.y = pack_bf16x2(acc.z, acc.w);
        const int h = h0 + hb + hl;
        *reinterpret_cast<uint2 *>(p.out + ((int64_t)t * p.num_heads + h) * kLatent + 4 * c) = u;
        if (c == 0 && p.lse != nullptr)
            p.lse[(int64_t)t * p.num_heads + h] = wts[hl * 10 + 8];
    }
}

// Logical position of key `k` of block `b` -> cache slot (phys_block * page + offset), or -1.
__device__ __forceinline__ int slot_of(const DecodeParams &p, int t, int row, bool row_ok, int kbeg, int kend, int b,
                                       int k)
{
    const int i = kbeg + b * kBK + k;
    if (i >= kend || !row_ok)
        return -1;
    const int idx = p.combined[(int64_t)t * p.cw + i];
    const int blk = idx >= 0 ? idx / p.page : -1;
    int phys = -1;
    if (idx >= 0 && blk < p.max_blocks)
        phys = p.block_table[(int64_t)row * p.bt_stride + blk];
    if (phys < 0 || phys >= p.num_blocks) {
        atomicOr(p.status, kStatusBadIndex);
        return -1;
    }
    return phys * p.page + (idx - blk * p.page);
}

__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int unit = blockIdx.x;
    const int split = unit % p.splits;   // = rank in the cluster when splits > 1
    const int group = (unit / p.splits) % p.groups;
    const int t = unit / (p.splits * p.groups);
    const int h0 = group * kNH;

    // Q does not depend on the combine kernel: its loads go out before waiting for it
    uint4 qv[kQLoads];
#pragma unroll
    for (int j = 0; j < kQLoads; ++j) {
        const int i = tid + kThreads * j;
        const int h = i / (kDim / 8);
        const int c = i % (kDim / 8);
        qv[j] = __ldg(reinterpret_cast<const uint4 *>(p.q + (int64_t)t * p.q_token_stride + (int64_t)(h0 + h) * kDim +
                                                       8 * c));
    }

    // ---- shared memory carve-up (1024-byte aligned base for the swizzled tiles)
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sQ = base;
    const uint32_t sK = base + kQBytes;
    const uint32_t sP = sK + 8 * kChunkBytes;   // P^T reuses the rope column chunk once S^T is done
    uint8_t *small = gbase + kQBytes + kKBytes;
    int *slots = reinterpret_cast<int *>(small + kOffSlots);
    unsigned *scal = reinterpret_cast<unsigned *>(small + kOffScale);
    float *red = reinterpret_cast<float *>(small + kOffRed);
    float *mrun = reinterpret_cast<float *>(small + kOffMrun);
    float *mcs = reinterpret_cast<float *>(small + kOffMc);
    float *alpha = reinterpret_cast<float *>(small + kOffAlpha);   // at the end: this split's max per head
    float *fin = reinterpret_cast<float *>(small + kOffFin);       // at the end: this split's row sum per head
    const uint32_t bar_s = smem_u32(small + kOffBars);
    const uint32_t bar_p = bar_s + 8;
    const uint32_t bar_o = bar_s + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(small + kOffTmem);
    volatile int *flags = reinterpret_cast<volatile int *>(small + kOffFlags);   // [0] abort, [1] rescale block tag
    float *wts = reinterpret_cast<float *>(gbase + 40960);   // merge weights (Q region, idle at the end)
    float *o_stage = reinterpret_cast<float *>(gbase + kQBytes);   // partial O [64][512] fp32 (K tile region)

    grid_dependency_wait();   // combined lists and lengths are ready

    const int L = p.lens[t];
    const int kbeg = split * p.chunk;
    const int kend = min(L, kbeg + p.chunk);
    const int nkeys = max(0, kend - kbeg);
    const int nblocks = (nkeys + kBK - 1) / kBK;
    const int row = p.req_idx ? p.req_idx[t] : t;
    const bool row_ok = row >= 0 && row < p.num_reqs;
    const float c2 = p.scale * 1.4426950408889634f;   // logits in log2 units per raw dot product
    if (!row_ok && tid == 0 && nkeys > 0)
        atomicOr(p.status, kStatusBadIndex);

    if (nblocks == 0) {   // no key in this split
        if (p.splits == 1) {   // zero output, LSE from the sink alone
            if (tid < kNH && p.lse)
                p.lse[(int64_t)t * p.num_heads + h0 + tid] = p.sink ? p.sink[h0 + tid] : -INFINITY;
            for (int i = tid; i < kNH * kLatent / 8; i += kThreads) {
                const int h = i / (kLatent / 8);
                const int d = i % (kLatent / 8);
                *reinterpret_cast<uint4 *>(p.out + ((int64_t)t * p.num_heads + h0 + h) * kLatent + 8 * d) =
                    make_uint4(0, 0, 0, 0);
            }
            return;
        }
        if (tid < kNH) {   // an empty partial: weight 0 in the merge, its O is never read
            alpha[tid] = -INFINITY;
            fin[tid] = 0.f;
        }
        cluster_sync();   // every split has staged its partial
        cluster_merge_pull(p, t, h0, split, smem_u32(alpha), smem_u32(fin), sK, wts);
        cluster_sync();   // peers have finished reading this CTA's shared memory
        return;
    }

    const bool is_mma = warp == 0;
    const bool is_soft = warp >= 4 && warp < 4 + kSoftWarps;
    const int wk = tid - 32;                              // worker index 0..479 (warps 1-15)
    const int stid = tid - 128;                           // softmax thread index 0..255 (warps 4-11)
    const int quad = warp & 3;                            // TMEM lane quadrant of this warp
    const int hh = (warp - 4) >> 2;                       // softmax: head half (heads 32 hh .. 32 hh + 31)
    const int key = quad * 32 + lane;                     // softmax: key of the block / value dim of a tile

    if (tid == 0) {
        mbar_init(bar_s, 1);
        mbar_init(bar_p, kSoftWarps);
        mbar_init(bar_o, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        flags[0] = 0;
        flags[1] = 0;
    }
    if (tid < kNH)
        mrun[tid] = -INFINITY;
    if (is_mma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // cache slots of blocks 0 and 1, one lookup per thread
    if (tid < 2 * kBK)
        slots[tid] = slot_of(p, t, row, row_ok, kbeg, kend, tid / kBK, tid % kBK);
    // Q (64 heads x 576 dims) -> swizzled K-major B operand
#pragma unroll
    for (int j = 0; j < kQLoads; ++j) {
        const int i = tid + kThreads * j;
        const int h = i / (kDim / 8);
        const int c = i % (kDim / 8);
        st_shared_v4(sQ + (c >> 3) * kQChunkBytes + sw128(h, c & 7), qv[j].x, qv[j].y, qv[j].z, qv[j].w);
    }
    fence_async_smem();
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);   // this warp's TMEM lanes

    if (is_mma) {
        // descriptors: 128-byte swizzle; K-major S^T operands advance 32 B per 16-dim step and one
        // column chunk per 64 dims; MN-major P.V operands advance 2 KB per 16 keys
        const uint64_t qk_a = sdesc(sK, 16, 1024);
        const uint64_t qk_b = sdesc(sQ, 16, 1024);
        const uint64_t pv_a = sdesc(sK, kChunkBytes, 1024);
        const uint64_t pv_b = sdesc(sP, 1024, 1024);   // one 64-head group along N: LBO unused, kept = SBO
        for (int b = 0; b < nblocks; ++b) {
            const uint32_t ph = (uint32_t)(b & 1);
            named_bar(3, kThreads);   // K tile of block b complete
            if (lane == 0) {
                tc_after();
#pragma unroll
                for (int ch = 0; ch < kChunks; ++ch) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma(tmem + kColS, qk_a + (uint64_t)((ch * kChunkBytes + 32 * k) >> 4),
                             qk_b + (uint64_t)((ch * kQChunkBytes + 32 * k) >> 4), kIdescQK, (ch | k) != 0 ? 1u : 0u);
                }
                umma_commit(bar_s);
                mbar_wait_one(bar_p, ph, flags, p.status);
                tc_after();
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        umma(tmem + kColO + 64 * m, pv_a + (uint64_t)((2 * m * kChunkBytes + kk * 2048) >> 4),
                             pv_b + (uint64_t)((kk * 2048) >> 4), kIdescPV, (b > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(bar_o);
            }
            __syncwarp();
        }
    } else {
        // ---- workers.  Worker wk owns 16-byte piece pc = wk % 40 of rows rg, rg + 12, ... of every
        // block (pieces 0-31 latent, 32-39 rope); workers 0-127 also fetch the scale word of row wk.
        const int pc = wk % kDataPieces;
        const int rg = wk / kDataPieces;
        const bool latent = pc < 32;
        const int chunk = latent ? pc >> 2 : 8;
        const uint32_t u0 = latent ? (uint32_t)(pc & 3) * 2u : (uint32_t)(pc - 32);
        const bool odd = latent && (chunk & 1);   // neighbouring chunks store their two units in opposite order
        const int scale_shift = 8 * (pc >> 3);
        uint4 pre[kRowsPerLoader];
        unsigned pre_scale = 0;
        auto issue_loads = [&](int b) {
            const int *sl = slots + (b % 3) * kBK;
#pragma unroll
            for (int it = 0; it < kRowsPerLoader; ++it) {
                const int r = rg + kRowGroups * it;
                const int sidx = r < kBK ? sl[r] : -1;
                pre[it] = sidx >= 0 ? ld_stream(p.kv + (int64_t)sidx * kEntryBytes + 16 * pc) : make_uint4(0, 0, 0, 0);
            }
            if (wk < kBK) {
                const int sidx = sl[wk];
                pre_scale = sidx >= 0 ? __ldg(reinterpret_cast<const unsigned *>(p.kv + (int64_t)sidx * kEntryBytes +
                                                                                  kScaleOffset))
                                      : 0u;
            }
        };
        issue_loads(0);
        for (int b = 0; b < nblocks; ++b) {
            const uint32_t ph = (uint32_t)(b & 1);
            if (b > 0)
                mbar_wait(bar_o, ph ^ 1u, flags, p.status);   // P.V has drained the tile
            if (wk < kBK)
                scal[wk] = pre_scale;
            named_bar(2, kWorkers);
            // the row addresses are recomputed each block (an opaque copy of rg stops the compiler
            // from hoisting 22 of them into registers for the whole loop)
            int rgb = rg;
            asm volatile("" : "+r"(rgb));
#pragma unroll
            for (int it = 0; it < kRowsPerLoader; ++it) {
                const int r = rgb + kRowGroups * it;
                if (r >= kBK)
                    continue;
                const uint32_t rowbase = sK + (uint32_t)chunk * kChunkBytes + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u;
                const uint4 v = pre[it];
                if (latent) {
                    const float sc = ue8m0_to_float((scal[r] >> scale_shift) & 0xFFu);
                    const uint32_t a0 = e4m3x2_to_bf16x2(v.x, sc), a1 = e4m3x2_to_bf16x2(v.x >> 16, sc);
                    const uint32_t a2 = e4m3x2_to_bf16x2(v.y, sc), a3 = e4m3x2_to_bf16x2(v.y >> 16, sc);
                    const uint32_t b0 = e4m3x2_to_bf16x2(v.z, sc), b1 = e4m3x2_to_bf16x2(v.z >> 16, sc);
                    const uint32_t b2 = e4m3x2_to_bf16x2(v.w, sc), b3 = e4m3x2_to_bf16x2(v.w >> 16, sc);
                    const uint32_t uf = u0 + (odd ? 1u : 0u);
                    const uint32_t us = u0 + (odd ? 0u : 1u);
                    st_shared_v4(rowbase + ((uf ^ (uint32_t)(r & 7)) << 4), odd ? b0 : a0, odd ? b1 : a1,
                                 odd ? b2 : a2, odd ? b3 : a3);
                    st_shared_v4(rowbase + ((us ^ (uint32_t)(r & 7)) << 4), odd ? a0 : b0, odd ? a1 : b1,
                                 odd ? a2 : b2, odd ? a3 : b3);
                } else {
                    st_shared_v4(rowbase + ((u0 ^ (uint32_t)(r & 7)) << 4), v.x, v.y, v.z, v.w);
                }
            }
            fence_async_smem();
            named_bar(3, kThreads);   // K tile of block b complete
            if (b + 1 < nblocks)
                issue_loads(b + 1);
            if (warp < 4 && b + 2 < nblocks) {
                for (int k = tid - 32; k < kBK; k += 96)
                    slots[((b + 2) % 3) * kBK + k] = slot_of(p, t, row, row_ok, kbeg, kend, b + 2, k);
            }
            if (!is_soft)
                continue;
            // ---- softmax of block b (warps 4-11; this warp: lanes of its quadrant, heads 32hh..32hh+31)
            mbar_wait(bar_s, ph, flags, p.status);
            tc_after();
            const bool kv = (b * kBK + key < nkeys) && slots[(b % 3) * kBK + key] >= 0;
            const uint32_t colS = kColS + 32 * hh;
            {   // per-head maxima of this block over the 32 keys of the quadrant; lane j keeps head j
                float mine = -INFINITY;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t s[16];
                    tmem_ld16(lane_base + colS + 16 * half, s);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float m = warp_max(kv ? __uint_as_float(s[j]) : -INFINITY);
                        mine = lane == 16 * half + j ? m : mine;
                    }
                }
                red[quad * kNH + 32 * hh + lane] = mine;
            }
            named_bar(1, kSoftThreads);
            if (stid < kNH) {
                const int h = stid;
                const float mb = fmaxf(fmaxf(red[h], red[kNH + h]), fmaxf(red[2 * kNH + h], red[3 * kNH + h]));
                const float mo = mrun[h];
                float mn = mo;
                float a = 1.f;
                if (mo == -INFINITY) {
                    mn = mb;
                } else if (mb > mo && (mb - mo) * c2 > kRescaleLog2) {
                    mn = mb;
                    a = exp2f((mo - mb) * c2);
                    flags[1] = b + 1;
                }
                mrun[h] = mn;
                mcs[h] = mn == -INFINITY ? 0.f : mn * c2;
                alpha[h] = a;
            }
            named_bar(1, kSoftThreads);
            if (flags[1] == b + 1) {   // some head's max grew past the threshold: rescale O^T and row sums
                uint32_t x[16];
#pragma unroll 1
                for (int m = 0; m < 10; ++m) {   // four O^T tiles, then the row sums, 16 columns at a time
                    const uint32_t col = ((m >> 1) < 4 ? kColO + 64 * (m >> 1) : kColL) + 32 * hh + 16 * (m & 1);
                    tmem_ld16(lane_base + col, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        x[j] = __float_as_uint(__uint_as_float(x[j]) * alpha[32 * hh + 16 * (m & 1) + j]);
                    tmem_st16(lane_base + col, x);
                }
            }
            // P = 2^(s*c - m*c) -> BF16 P^T row `key`; row sums accumulate per lane in TMEM
#pragma unroll 1
            for (int hq = 0; hq < 2; ++hq) {   // 16 heads at a time
                const int hb = 32 * hh + 16 * hq;
                uint32_t sv[16], l[16];
                tmem_ld16(lane_base + kColS + hb, sv);
                if (b > 0)
                    tmem_ld16(lane_base + kColL + hb, l);
                tmem_ld_wait();
                uint32_t pk[8];
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const float p0 = kv ? exp2f(fmaf(__uint_as_float(sv[j]), c2, -mcs[hb + j])) : 0.f;
                    const float p1 = kv ? exp2f(fmaf(__uint_as_float(sv[j + 1]), c2, -mcs[hb + j + 1])) : 0.f;
                    l[j] = __float_as_uint((b > 0 ? __uint_as_float(l[j]) : 0.f) + p0);
                    l[j + 1] = __float_as_uint((b > 0 ? __uint_as_float(l[j + 1]) : 0.f) + p1);
                    pk[j >> 1] = pack_bf16x2(p0, p1);
                }
                tmem_st16(lane_base + kColL + hb, l);
                st_shared_v4(sP + sw128(key, hb >> 3), pk[0], pk[1], pk[2], pk[3]);
                st_shared_v4(sP + sw128(key, (hb >> 3) + 1), pk[4], pk[5], pk[6], pk[7]);
            }
            tmem_st_wait();
            fence_async_smem();
            tc_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_p);
        }
    }

    mbar_wait(bar_o, (uint32_t)((nblocks - 1) & 1), flags, p.status);
    tc_after();

    // ---- epilogue: row sums across lanes; normalised output, or the partial staged for the merge
    float *lred = reinterpret_cast<float *>(gbase);   // Q region is free: [128 lanes][65]
    if (is_soft) {
        {
            uint32_t l[32];
            tmem_ld32(lane_base + kColL + 32 * hh, l);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j)
                lred[key * 65 + 32 * hh + j] = __uint_as_float(l[j]);
        }
        named_bar(1, kSoftThreads);
        if (stid < kNH) {
            const int h = stid;
            float acc[8];
#pragma unroll
            for (int a = 0; a < 8; ++a)
                acc[a] = 0.f;
#pragma unroll 2
            for (int k = 0; k < kBK; k += 8) {
#pragma unroll
                for (int a = 0; a < 8; ++a)
                    acc[a] += lred[(k + a) * 65 + h];
            }
            const float lsum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
            const float m = mrun[h];
            const float ms = m == -INFINITY ? -INFINITY : m * p.scale;   // natural-log units
            if (p.splits == 1) {
                float M = ms;
                float Z = lsum;
                if (p.sink != nullptr) {
                    const float sk = p.sink[h0 + h];
                    M = fmaxf(ms, sk);
                    Z = (ms == -INFINITY ? 0.f : lsum * expf(ms - M)) + expf(sk - M);
                }
                fin[h] = (Z > 0.f && ms != -INFINITY) ? expf(ms - M) / Z : 0.f;
                if (p.lse)
                    p.lse[(int64_t)t * p.num_heads + h0 + h] = Z > 0.f ? M + logf(Z) : -INFINITY;
            } else {
                alpha[h] = ms;
                fin[h] = ms == -INFINITY ? 0.f : lsum;
            }
        }
        named_bar(1, kSoftThreads);
        uint32_t x[32];
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
            const int dv = 128 * m + key;
            tmem_ld32(lane_base + kColO + 64 * m + 32 * hh, x);
            tmem_ld_wait();
            if (p.splits == 1) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int h = 32 * hh + j;
                    p.out[((int64_t)t * p.num_heads + h0 + h) * kLatent + dv] = bf16_bits(__uint_as_float(x[j]) * fin[h]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    o_stage[(32 * hh + j) * kLatent + dv] = __uint_as_float(x[j]);
            }
        }
    }
    tc_before();
    __syncthreads();
    tc_after();
    if (is_mma)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    if (p.splits > 1) {
        cluster_sync();   // every split has staged its partial
        cluster_merge_pull(p, t, h0, split, smem_u32(alpha), smem_u32(fin), sK, wts);
        cluster_sync();   // peers have finished reading this CTA's shared memory
    }
}

}  // namespace

int decode_tc_chunk_keys() { return kBK; }
int decode_tc_max_splits() { return kMaxSplits; }

// Concurrently resident CTAs of the decode kernel when launched in clusters of `splits`
// (whole clusters must fit inside one GPC); cached per device.
int decode_tc_resident_ctas(int splits)
{
    static int cache[64][kMaxSplits + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || splits < 1 || splits > kMaxSplits)
        return 0;
    if (cache[dev][splits] > 0)
        return cache[dev][splits];
    if (set_smem_once(reinterpret_cast<const void *>(decode_tc_kernel), kSmemBytes, kAttrTc) != cudaSuccess)
        return 0;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int n = sms;
    if (splits > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(splits * sms);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = splits;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, reinterpret_cast<const void *>(decode_tc_kernel), &cfg) !=
            cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        n = clusters * splits;
    }
    cache[dev][splits] = n;
    return n;
}

cudaError_t launch_decode_tc(const DecodeParams &p, cudaStream_t stream)
{
    if (p.num_tokens <= 0)
        return cudaSuccess;
    if (p.heads_per_group != kNH || p.chunk % kBK != 0 || p.splits < 1 || p.splits > kMaxSplits)
        return cudaErrorInvalidValue;
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(decode_tc_kernel), kSmemBytes, kAttrTc);
    if (e != cudaSuccess)
        return e;
    const long long grid = (long long)p.num_tokens * p.groups * p.splits;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)p.splits;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.splits > 1 ? 2 : 1;
    void *args[] = {const_cast<DecodeParams *>(&p)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(decode_tc_kernel), args);
}

}  // namespace dsv4
