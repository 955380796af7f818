// decode_tc.cu -- tensor-core (tcgen05 / TMEM) sparse-MLA decode, 64 heads per CTA, with the
// top-k + sliding-window index combine fused into its prologue.
//
// Operation (per token t, head h, over the token's combined key list K_t):
//   s_p = scale * q_h . k_p  (576 dims),  out_h = sum_p softmax(s)_p v_p  (512 dims)
// with the combine of "[ROCm] [DSv4] [Perf] Support DeepSeek v4 MTP" (vllm #43385,
// _combine_topk_swa_indices_kernel: kept top-k entries in input order, then the window
// ascending), the gather/dequant of "feat: add DeepSeek-V4 XPU attention decode path"
// (vllm #42953, _dequant_gather_slots_kernel: value = e4m3 * 2^(ue8m0 - 127), rope as
// stored) and the per-request block-table conversion and [T, h, 512] output of "Enable
// DeepSeek V4 and GLM-5.1 on SM120" (vllm #43477, flashinfer_mla_sparse_sm120.py).
//
// Shape of the contraction.  All heads share one key set (MQA), so a token is a pair of
// dense products: S = Q K^T (64 x 576 x keys) and O = P V (64 x keys x 512).  With 64
// heads the head dimension is too short to fill a 128-row tcgen05 tile, so both products
// run transposed, keys and value dims on the M side:
//   S^T[128 keys x 64 heads]   = K_tile[128 x 576] . Q^T          (A = K tile, K-major)
//   O^T[128 dv x 64 heads] += V^T[128 dv x 128 keys] . P^T        (A = K tile, MN-major)
// One BF16 K tile in shared memory (128-byte swizzle, 8-row atoms, nine 64-dim column
// chunks) is read by both: as K-major A for S^T and, without a copy, as MN-major A for O^T.
// S^T (two accumulators over column chunks 0-4 and 5-8, summed by the softmax), O^T (four
// 128-dv tiles) and per-lane partial row sums live in TMEM (448 of 512 columns).
//
// CTA = 19 warps, one (token, 64-head group, split): lane 0 of warps 0, 17 and 18 issue the
// MMAs (warp 0: S^T over chunks 0-4 and O^T tiles 0-1; warp 17: S^T over chunks 5-8; warp 18:
// O^T tiles 2-3), warps 1-16 do everything else.  A token with 16 or 32 heads is one group
// whose missing heads have zero queries: their columns of the products are computed and
// dropped, never written out.  Prologue: the CTA combines its token's top-k row with the window
// (shared-memory hash set for first occurrences, ballot scan for the output order), keeps the
// entries of its own split and resolves them through the block-table row (cached in shared
// memory) to cache slots: blocks 0 and 1 straight into shared memory, later blocks into the
// workspace.  Per 128-key block:
//   dequant   each worker thread owns a quarter of one row of the tile (the rows of a warp
//             differ in row % 8 and spread over the tile), holds the row's 16-byte pieces
//             in registers (loaded during the previous block) and writes the exact BF16
//             values chunk by chunk; chunk c of block b+1 is written as soon as the P.V
//             product of block b has released it; rows past the split's keys are zeros
//   S^T       the MMAs of column chunks 0-5 are issued once every worker warp has written
//             them, those of chunks 6-8 after, so the product trails the dequant
//   softmax   all 16 warps: warp w reads TMEM lanes 32 (w % 4).. (its keys) for heads
//             16 ((w - 1) / 4)..; per-head block maxima with redux.sync, one barrier to share
//             them between the four warps of a head slice, which then each keep the running
//             max in registers; lazy rescaling (only when a head's max grows by more than
//             2^8), P^T (BF16) into shared memory, row sums in TMEM
//   O^T       up to 32 MMAs (only the 16-key steps that hold keys), committed per 128-dv tile
//             so the next block's dequant can start
// When a token's keys are split over S CTAs (S <= 8), the S CTAs form a thread-block
// cluster: after a cluster barrier each pushes its fp32 partial straight from TMEM into the
// shared memory of the CTA that owns each head slice (distributed shared memory), and after
// a second barrier every CTA merges its slice locally.
// Every mbarrier wait is bounded; a wait that runs out records DSV4_ERR_TIMEOUT in the
// status word and the CTA finishes without waiting again.
#include <climits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kThreads = 608;             // warp 0: MMA issue; warps 1-16: workers; warps 17, 18: MMA issue
constexpr int kSIssuerB = 17;            // S^T over column chunks 5-8 (a second accumulator)
constexpr int kPVIssuerB = 18;           // O^T tiles 2 and 3
constexpr int kWorkers = 512;
constexpr int kBK = 128;                 // keys per block = MMA M
constexpr int kNH = 64;                  // heads per CTA = MMA N
constexpr int kChunks = 9;               // 576 dims / 64
constexpr int kQBytes = kChunks * kNH * 128;     // 73728
constexpr int kKBytes = kChunks * kBK * 128;     // 147456
constexpr int kChunkBytes = kBK * 128;           // 16384 (one 64-dim column chunk of the K tile)
constexpr int kQChunkBytes = kNH * 128;          // 8192
constexpr int kHeadSlots = 2 * kBK;      // cache slots of blocks 0 and 1, found in the prologue
constexpr int kPassLoads = 4;            // combine: top-k entries per thread loaded up front
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;            // S^T: 64 columns
constexpr uint32_t kColO = 64;           // O^T: 4 tiles x 64 columns
constexpr uint32_t kColL = 320;          // per-lane partial row sums: 64 columns
constexpr uint32_t kColSb = 384;         // S^T over column chunks 5-8: 64 columns (added to kColS's)
constexpr float kRescaleLog2 = 8.0f;
constexpr long long kWaitCycles = 4000000000LL;
constexpr int kMaxSplits = 8;            // portable cluster size
// MTP union lists: a position below 2^29, bit 29 set when the request's first token lists it,
// bit 30 when its second does; the union kernel writes them and cache slots (below 2^29 as
// well) carry the same bits through the decode
constexpr int kUnionMaskShift = 29;
constexpr int kUnionPosMask = (1 << kUnionMaskShift) - 1;

// small shared region (after Q and the K tile)
constexpr int kOffSlots = 0;             // int [3][128]: cache slots of blocks b, b+1, b+2
constexpr int kOffRed = 1536;            // float [2][4][64]: per-quadrant head maxima, by block parity
constexpr int kOffMrun = 3584;           // float [64]
constexpr int kOffAlpha = 3840;          // float [64]
constexpr int kOffFin = 4096;            // float [64]
constexpr int kOffWsum = 4352;           // int [4][32]
constexpr int kOffBars = 4864;           // u64: bar_s, bar_p, bar_pv[4], bar_grp[2]
constexpr int kOffTmem = 4936;           // u32
constexpr int kOffFlags = 4944;          // int [2]
constexpr int kSmallBytes = 4992;
constexpr int kBtOffset = 2 * 4 * 2 * kMaxTopkWidth;   // block-table cache in the K tile region, after the hash set
constexpr int kBtCache = (kKBytes - kBtOffset) / 4;    // entries
constexpr int kSmemBytes = kQBytes + kKBytes + kSmallBytes + 1024;   // + alignment slack
constexpr int kQLoads = kNH * (kDim / 8) / kWorkers;                 // 9 16-byte Q pieces per worker
constexpr int kGroups = 2;               // S^T is issued in 2 groups: column chunks 0-5, then 6-8
static_assert(kNH * (kDim / 8) % kWorkers == 0, "Q pieces per worker");
static_assert(kKBytes >= kNH * kLatent * (int)sizeof(float), "partial O fits the K tile");

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
__device__ __noinline__ void mbar_wait_one(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned *status,
                                           long long limit = kWaitCycles)
{
    if (*abort_flag)
        return;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            atomicOr(status, kStatusTimeout);
            return;
        }
        if (*abort_flag)
            return;
    }
}

// Warp-wide wait: every lane of the warp waits itself (measured faster than one polling lane
// handing over through __syncwarp).
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned *status)
{
    mbar_wait_one(bar, parity, abort_flag, status);
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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
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

// 16-byte asynchronous copy global -> shared (L2 only); `bytes` < 16 fills the rest with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
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

// two E4M3 codes (low byte = first element) -> BF16x2 of code * scale through the hardware
// conversion (exact for every code and scale)
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two, float scale)
{
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    const float2 f = __half22float2(__half2(hr));
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y * scale), "f"(f.x * scale));
    return r;
}

// The hardware-conversion form of dequant16_store below, kept out of line: it only runs
// for pieces holding the NaN code or a scale past 2^7.
__device__ __noinline__ void dequant16_store_convert(uint4 v, uint32_t se, uint32_t a0, uint32_t a1)
{
    const float sc = ue8m0_to_float(se);
    st_shared_v4(a0, e4m3x2_to_bf16x2(v.x, sc), e4m3x2_to_bf16x2(v.x >> 16, sc), e4m3x2_to_bf16x2(v.y, sc),
                 e4m3x2_to_bf16x2(v.y >> 16, sc));
    st_shared_v4(a1, e4m3x2_to_bf16x2(v.z, sc), e4m3x2_to_bf16x2(v.z >> 16, sc), e4m3x2_to_bf16x2(v.w, sc),
                 e4m3x2_to_bf16x2(v.w >> 16, sc));
}

// 16 E4M3 codes times 2^(se - 127) -> 16 BF16, elements 0-7 to shared address a0 and 8-15 to a1.
// An E4M3 code s.eeee.mmm placed as the BF16 pattern s.0000eeee.mmm0000 is its value times
// 2^-120 for normal and subnormal codes alike (both formats put the binary point the same
// way; only the exponent biases, 7 and 127, differ).  One BF16 multiply by 2^(se - 7) then
// gives the value exactly rounded.  The NaN code (magnitude 0x7F) and scales past 2^7
// (se > 134, whose factor has no BF16 form) take the hardware conversion instead.
__device__ __forceinline__ void dequant16_store(uint4 v, uint32_t se, uint32_t a0, uint32_t a1)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t t[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        t[2 * i] = __byte_perm(w[i], 0u, 0x1404);       // [0, c0, 0, c1]
        t[2 * i + 1] = __byte_perm(w[i], 0u, 0x3424);   // [0, c2, 0, c3]
    }
    uint32_t bad = se > 134u ? 1u : 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        bad |= ((w[i] & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;   // a byte with magnitude 0x7F
    if (bad == 0u) {
        uint32_t f = (se + 120u) << 7;
        f |= f << 16;
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t x = (t[i] & 0x80008000u) | ((t[i] & 0x7F007F00u) >> 4);
            asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(x), "r"(f));
        }
        st_shared_v4(a0, o[0], o[1], o[2], o[3]);
        st_shared_v4(a1, o[4], o[5], o[6], o[7]);
    } else {
        dequant16_store_convert(v, se, a0, a1);
    }
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

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_v2(uint32_t addr, float a, float b)
{
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}

// Split-KV merge inside a cluster of S = splits CTAs (one per split of a token's keys).
// The CTA of rank r owns heads [r*hp, (r+1)*hp) (hp = ceil(64 / S)).  Every split s has
// pushed, into each owner's shared memory, its running max m_s (natural-log units) and row
// sum l_s for the owner's heads (stat[s][hl] = (m_s, l_s)) and its unnormalised fp32 O_s for
// them (recv[s][hl][512]).  After the cluster barrier the owner forms
//   m = max(max_s m_s, sink), Z = sum_s l_s e^{m_s - m} + e^{sink - m},
//   out = sum_s e^{m_s - m} O_s / Z  (BF16),  lse = m + ln Z,
// skipping splits without keys (weight 0, whatever their slots hold).
// kUnion: column c of the tile is head h0 + c % 32 of token t + c / 32 (MTP union calls); else
// head h0 + c of token t.
template <bool kUnion>
__device__ __noinline__ void cluster_merge_local(uint16_t *out, float *lse, const float *sink, int num_heads, int S,
                                                 int t, int h0, int rank, const float *recv, const float *stat,
                                                 float *wts)
{
    const int hp = (kNH + S - 1) / S;
    const int hb = rank * hp;
    const int nh = max(0, min(kUnion ? kNH : min(kNH, num_heads - h0), hb + hp) - hb);   // owned heads that exist
    const int tid = threadIdx.x;
    if (tid < nh) {
        const int h = hb + tid;
        float m = -INFINITY;
        for (int s = 0; s < S; ++s)
            m = fmaxf(m, stat[2 * (s * hp + tid)]);
        const float mk = m;
        float sk = 0.f;
        if (sink != nullptr) {
            sk = sink[kUnion ? h0 + (h & 31) : h0 + h];
            m = fmaxf(m, sk);
        }
        float z = 0.f;
        for (int s = 0; s < S; ++s) {
            const float ms = stat[2 * (s * hp + tid)];
            const float w = ms == -INFINITY ? 0.f : expf(ms - m);
            wts[tid * 10 + s] = w;
            z += stat[2 * (s * hp + tid) + 1] * w;
        }
        if (sink != nullptr)
            z += expf(sk - m);
        const float f = (z > 0.f && mk != -INFINITY) ? 1.f / z : 0.f;
        for (int s = 0; s < S; ++s)
            wts[tid * 10 + s] *= f;
        wts[tid * 10 + 8] = z > 0.f ? m + logf(z) : -INFINITY;
    }
    __syncthreads();
    const int items = nh * (kLatent / 4);   // 16-byte pieces of the slice
    for (int i = tid; i < items; i += kThreads) {
        const int hl = i / (kLatent / 4);
        const int c = i % (kLatent / 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < S; ++s) {
            const float ws = wts[hl * 10 + s];
            if (ws != 0.f) {
                const float4 v = *reinterpret_cast<const float4 *>(recv + ((size_t)(s * hp + hl)) * kLatent + 4 * c);
                acc.x = fmaf(ws, v.x, acc.x);
                acc.y = fmaf(ws, v.y, acc.y);
                acc.z = fmaf(ws, v.z, acc.z);
                acc.w = fmaf(ws, v.w, acc.w);
            }
        }
        uint2 o;
        o.x = pack_bf16x2(acc.x, acc.y);
        o.y = pack_bf16x2(acc.z, acc.w);
        const int col = hb + hl;
        const int64_t row = kUnion ? (int64_t)(t + (col >> 5)) * num_heads + h0 + (col & 31)
                                   : (int64_t)t * num_heads + h0 + col;
        *reinterpret_cast<uint2 *>(out + row * kLatent + 4 * c) = o;
        if (c == 0 && lse != nullptr)
            lse[row] = wts[hl * 10 + 8];
    }
}

// Pushes the (m, l) pair of head h (0..63) of split `split` to the head's owner in the cluster.
__device__ __forceinline__ void push_stat(uint32_t stat_s, int S, int split, int h, float m, float l)
{
    const int hp = (kNH + S - 1) / S;
    const int r = h / hp;
    const uint32_t off = (uint32_t)(2 * (split * hp + (h - r * hp))) * 4u;
    st_cluster_v2(map_to_rank(stat_s + off, (uint32_t)r), m, l);
}

// Logical position -> cache slot (phys_block * page + offset) through the token's
// block-table row; -1 (and the bad-index status bit) when the table has no valid block.
__device__ __forceinline__ int slot_of_position(const DecodeParams &p, int row, int idx, const int *bt_s,
                                                bool bt_cached)
{
    const int blk = idx / p.page;
    int phys = -1;
    if (blk < p.max_blocks)
        phys = bt_cached ? bt_s[blk] : p.block_table[(int64_t)row * p.bt_stride + blk];
    if (phys < 0 || phys >= p.num_blocks) {
        atomicOr(p.status, kStatusBadIndex);
        return -1;
    }
    return phys * p.page + (idx - blk * p.page);
}

// L2 prefetch of the cache entry of position idx (through the cached block-table row); no
// status is recorded here, the combine resolves the same position again.
__device__ __forceinline__ void prefetch_entry(const DecodeParams &p, int idx, const int *bt_s)
{
    const int blk = idx / p.page;
    if (blk >= p.max_blocks)
        return;
    const int phys = bt_s[blk];
    if (phys < 0 || phys >= p.num_blocks)
        return;
    const int64_t slot = (int64_t)phys * p.page + (idx - blk * p.page);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.kv + slot * kEntryBytes), "r"((uint32_t)kEntryBytes)
                 : "memory");
}

__device__ __forceinline__ unsigned hash_pos(int v, int bits) { return ((unsigned)v * 0x9E3779B1u) >> (32 - bits); }

constexpr int kHashBitsMax = 14;                       // 2^14 slots of 8 bytes: the K tile region before the block table
constexpr unsigned long long kHashEmpty = ~0ull;
static_assert((8 << kHashBitsMax) <= kBtOffset, "combine hash table fits before the block-table cache");

// The slot of position v holds (v << 32) | smallest top-k index seen for v.  Returns the slot;
// the first writer of a position claims the slot with one CAS, a repeat lowers the index.
__device__ __forceinline__ unsigned hash_insert(unsigned long long *tab, int bits, int v, int i)
{
    const unsigned long long want = ((unsigned long long)(unsigned)v << 32) | (unsigned)i;
    unsigned h = hash_pos(v, bits);
    while (true) {
        const unsigned long long prev = atomicCAS(&tab[h], kHashEmpty, want);
        if (prev == kHashEmpty)
            return h;
        if ((unsigned)(prev >> 32) == (unsigned)v) {
            atomicMin(&tab[h], want);
            return h;
        }
        h = (h + 1u) & ((1u << bits) - 1u);
    }
}

// kRide: the next block's entries are loaded during the dequant, each chunk group's pieces once the
// group is written (worth it when a CTA runs many blocks), instead of in one burst after it.
// kUnion: an MTP union call (unit = request and 32-head group; column c of the tile is head
// h0 + c % 32 of token t + c / 32, t = 2 * request; keys come from the request's union list,
// each masked for the token that does not list it).
template <bool kRide, bool kUnion>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int split = blockIdx.x % p.splits;   // = rank in the cluster when splits > 1
    const bool is_mma = warp == 0;
    const bool is_worker = warp >= 1 && warp <= 16;
    const bool is_issuer = is_mma || warp == kSIssuerB || warp == kPVIssuerB;
    const int wid = tid - 32;            // worker index 0..511 (warps 1-16)

    // ---- shared memory carve-up (1024-byte aligned base for the swizzled tiles)
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sQ = base;
    const uint32_t sK = base + kQBytes;
    const uint32_t sP = sK + 8 * kChunkBytes;   // P^T reuses the rope column chunk once S^T is done
    uint8_t *small = gbase + kQBytes + kKBytes;
    int *slots = reinterpret_cast<int *>(small + kOffSlots);
    float *red = reinterpret_cast<float *>(small + kOffRed);
    float *mrun = reinterpret_cast<float *>(small + kOffMrun);
    float *alpha = reinterpret_cast<float *>(small + kOffAlpha);   // at the end: this split's max per head
    float *fin = reinterpret_cast<float *>(small + kOffFin);       // at the end: this split's row sum per head
    int *wsum = reinterpret_cast<int *>(small + kOffWsum);
    const uint32_t bar_s = smem_u32(small + kOffBars);   // S^T of the block complete
    const uint32_t bar_p = bar_s + 8;                    // P^T and row sums of the block written (16 warps)
    const uint32_t bar_pv = bar_s + 16;                  // [4] O^T tiles 0..m of the block complete
    const uint32_t bar_grp = bar_s + 48;                 // [2] column chunks 0-5, then 6-8 of the K tile written
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(small + kOffTmem);
    volatile int *flags = reinterpret_cast<volatile int *>(small + kOffFlags);   // [0] abort, [1] rescale block tag
    int *hkey = reinterpret_cast<int *>(gbase + kQBytes);          // combine hash set (K tile region)

    // ---- set-up that reads no input, ahead of the wait for the previous grid: barriers, TMEM,
    // the combine's empty hash set
    if (tid == 0) {
        mbar_init(bar_s, 2);   // both S^T accumulators committed
        mbar_init(bar_p, kWorkers / 32);
        for (int m = 0; m < 4; ++m)
            mbar_init(bar_pv + 8 * m, 1);
        for (int g = 0; g < kGroups; ++g)
            mbar_init(bar_grp + 8 * g, kWorkers / 32);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        flags[0] = 0;
        flags[1] = 0;
    }
    if (is_mma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // (position, top-k index) pairs, 64 bits a slot, at most a quarter full
    const int bits = p.table_bits;
    const int table = 1 << bits;
    unsigned long long *htab = reinterpret_cast<unsigned long long *>(hkey);
    for (int i = tid; i < table; i += kThreads)
        htab[i] = kHashEmpty;
    if (tid < kHeadSlots)
        slots[tid] = -1;
    tc_before();

    // every input may come from the previous kernel in the stream; the next kernel may be
    // scheduled now (it waits for this grid's results itself)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // this cluster's (token, head group): the ordering kernel's choice, else index order
    const int cl = blockIdx.x / p.splits;
    const int unit = p.order != nullptr ? p.order[cl] : cl;
    const int group = unit % p.groups;
    const int t = kUnion ? 2 * (unit / p.groups) : unit / p.groups;
    const int h0 = group * (kUnion ? kNH / 2 : kNH);
    // heads of the group that exist (16 or 32 heads: the rest are zero); all 64 columns in union calls
    const int nhv = kUnion ? kNH : min(kNH, p.num_heads - h0);
    // output row of tile column c
    auto out_row = [&](int c) -> int64_t {
        return kUnion ? (int64_t)(t + (c >> 5)) * p.num_heads + h0 + (c & 31) : (int64_t)t * p.num_heads + h0 + c;
    };

    // ---- early loads: the token's sizes and top-k run first (the combine waits on them), then Q,
    // copied asynchronously into its tile (the combine works in the K tile region)
    const int seq_len = kUnion ? 0 : p.seq_lens[t];   // union calls take their keys from the union list
    const int W = p.topk_width;
    int n = kUnion ? 0 : W;
    if (!kUnion && p.topk_lens != nullptr) {
        n = p.topk_lens[t];
        n = n < 0 ? 0 : (n > W ? W : n);
    }
    const int row = p.req_idx ? p.req_idx[t] : t;
    const bool row_ok = row >= 0 && row < p.num_reqs;
    // the token's block-table row -> shared memory, read alongside the top-k row
    int *bt_s = reinterpret_cast<int *>(gbase + kQBytes + kBtOffset);
    const bool bt_cached = p.max_blocks <= kBtCache;
    if (row_ok && bt_cached) {
        const int32_t *bt_row = p.block_table + (int64_t)row * p.bt_stride;
        for (int i = tid; i < p.max_blocks; i += kThreads)
            bt_s[i] = __ldg(bt_row + i);
    }
    const int32_t *trow = p.topk + (int64_t)t * p.topk_stride;
    const int npass = (n + kThreads - 1) / kThreads;   // the combine visits entry pass * kThreads + tid
    int tv[kPassLoads];
#pragma unroll
    for (int u = 0; u < kPassLoads; ++u)
        tv[u] = u < npass && u * kThreads + tid < n ? __ldg(trow + u * kThreads + tid) : -1;
    if (is_worker) {   // Q -> swizzled K-major B operand (zeros for heads that do not exist)
#pragma unroll
        for (int j = 0; j < kQLoads; ++j) {
            const int i = wid + kWorkers * j;
            const int h = i / (kDim / 8);
            const int c = i % (kDim / 8);
            if constexpr (kUnion)
                cp_async16(sQ + (c >> 3) * kQChunkBytes + sw128(h, c & 7),
                           p.q + (int64_t)(t + (h >> 5)) * p.q_token_stride + (int64_t)(h0 + (h & 31)) * kDim + 8 * c,
                           16u);
            else
                cp_async16(sQ + (c >> 3) * kQChunkBytes + sw128(h, c & 7),
                           p.q + (int64_t)t * p.q_token_stride + (int64_t)(h0 + min(h, nhv - 1)) * kDim + 8 * c,
                           h < nhv ? 16u : 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }

    // ---- fused combine (kept top-k entries in input order, then the window ascending):
    // window [win_lo, pos]; the top-k survivors are the first occurrences of positions in [0, win_lo)
    const int pos = seq_len - 1;   // seq_len <= 0: nothing is visible
    const long long lo = (long long)pos - p.window + 1;
    const int win_lo = lo < 0 ? 0 : (int)lo;
    const int swa = seq_len > 0 ? pos - win_lo + 1 : 0;
    __syncthreads();
    // first occurrence of each position: the smallest top-k index holding it; the entries of
    // the first passes remember their slot
    unsigned hs_slot[kPassLoads];
#pragma unroll
    for (int u = 0; u < kPassLoads; ++u)
        hs_slot[u] = (tv[u] >= 0 && tv[u] < win_lo) ? hash_insert(htab, bits, tv[u], u * kThreads + tid) : 0u;
#pragma unroll 1
    for (int ps = kPassLoads; ps < npass; ++ps) {
        const int i = ps * kThreads + tid;
        const int v = i < n ? __ldg(trow + i) : -1;
        if (v >= 0 && v < win_lo)
            hash_insert(htab, bits, v, i);
    }
    __syncthreads();
    const int kbeg = split * p.chunk;
    const int klim = kbeg + p.chunk;
    // the first two blocks' entries start towards L2 now, while the combine finishes: the rank of
    // an entry is taken as its input index (exact unless earlier entries are dropped), the window
    // as following all n top-k entries
    if (row_ok && bt_cached) {
        const int plim = min(klim, kbeg + 2 * kBK);
#pragma unroll
        for (int u = 0; u < kPassLoads; ++u) {
            const int i = u * kThreads + tid;
            if (tv[u] >= 0 && tv[u] < win_lo && i >= kbeg && i < plim)
                prefetch_entry(p, tv[u], bt_s);
        }
        for (int j = max(0, kbeg - n) + tid; j < swa && n + j < plim; j += kThreads)
            prefetch_entry(p, win_lo + j, bt_s);
    }
    // survivors in input order: ballots of up to four passes, one barrier, then every thread
    // ranks its entries; the ones of this split resolve to cache slots
    int32_t *slot_row = p.combined + (int64_t)t * p.cw;   // cache slots of blocks >= 2 of this split
    int total = 0;
#pragma unroll 1
    for (int pg = 0; pg < npass; pg += kPassLoads) {
        unsigned bal[kPassLoads];
        int vg[kPassLoads];
#pragma unroll
        for (int u = 0; u < kPassLoads; ++u) {
            bal[u] = 0;
            vg[u] = -1;
            if (pg + u >= npass)
                continue;
            const int i = (pg + u) * kThreads + tid;
            const int v = pg == 0 ? tv[u] : (i < n ? __ldg(trow + i) : -1);
            vg[u] = v;
            bool keep = false;
            if (v >= 0 && v < win_lo) {
                unsigned h;
                if (pg == 0) {
                    h = hs_slot[u];
                } else {
                    h = hash_pos(v, bits);
                    while ((unsigned)(htab[h] >> 32) != (unsigned)v)
                        h = (h + 1u) & (unsigned)(table - 1);
                }
                keep = (unsigned)htab[h] == (unsigned)i;
            }
            bal[u] = __ballot_sync(0xffffffffu, keep);
            if (lane == 0)
                wsum[32 * u + warp] = __popc(bal[u]);
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kPassLoads; ++u) {
            if (pg + u >= npass)
                continue;
            int rank = total + __popc(bal[u] & ((1u << lane) - 1u));
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) {
                rank += w < warp ? wsum[32 * u + w] : 0;
                total += wsum[32 * u + w];
            }
            if (((bal[u] >> lane) & 1u) && rank >= kbeg && rank < klim && p.trace != nullptr && group == 0)
                p.trace[(int64_t)t * p.trace_stride + rank] = vg[u];
            if (((bal[u] >> lane) & 1u) && row_ok && rank >= kbeg && rank < klim) {
                const int sl = slot_of_position(p, row, vg[u], bt_s, bt_cached);
                if (rank - kbeg < kHeadSlots)
                    slots[rank - kbeg] = sl;
                else
                    slot_row[rank] = sl;
            }
        }
        if (pg + kPassLoads < npass)
            __syncthreads();   // wsum is rewritten by the next group of passes
    }

    const int L = kUnion ? max(0, min(p.ulen[t >> 1], p.cw)) : total + swa;
    const int kend = min(L, klim);
    const int nkeys = max(0, kend - kbeg);
    const int nblocks = (nkeys + kBK - 1) / kBK;
    if (!row_ok && tid == 0 && nkeys > 0)
        atomicOr(p.status, kStatusBadIndex);
    if (p.trace != nullptr && group == 0) {   // the window part of the list, and its length
        for (int i = max(kbeg, total) + tid; i < kend; i += kThreads)
            p.trace[(int64_t)t * p.trace_stride + i] = win_lo + (i - total);
        if (split == 0 && tid == 0)
            p.trace_lens[t] = L;
    }
    if (kUnion && row_ok) {   // this split's part of the request's union list: slots carry the token masks
        const int32_t *urow = p.ulist + (int64_t)(t >> 1) * p.ulist_stride;
        for (int i = kbeg + tid; i < kend; i += kThreads) {
            const int e = urow[i];
            const int pos_e = e & kUnionPosMask;
            int sl = e >= 0 ? slot_of_position(p, row, pos_e, bt_s, bt_cached) : -1;
            sl = sl >= 0 ? (sl | (((e >> kUnionMaskShift) & 3) << kUnionMaskShift)) : -1;
            if (i - kbeg < kHeadSlots) {
                slots[i - kbeg] = sl;
                if (sl >= 0 && bt_cached)
                    prefetch_entry(p, pos_e, bt_s);
            } else {
                slot_row[i] = sl;
            }
        }
    } else if (row_ok) {   // the window part of this split
        for (int i = max(kbeg, total) + tid; i < kend; i += kThreads) {
            const int sl = slot_of_position(p, row, win_lo + (i - total), bt_s, bt_cached);
            if (i - kbeg < kHeadSlots)
                slots[i - kbeg] = sl;
            else
                slot_row[i] = sl;
        }
    }

    if (nblocks == 0) {   // no key in this split
        asm volatile("cp.async.wait_all;" ::: "memory");   // the Q copy lands before the merge overlays Q
        if (is_mma) {   // TMEM back (its address is visible after the combine's barriers)
            tc_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*tmem_slot), "r"(kTmemCols)
                         : "memory");
        }
        if (p.splits == 1) {   // zero output, LSE from the sink alone
            if (tid < nhv && p.lse)
                p.lse[kUnion ? out_row(tid) : (int64_t)t * p.num_heads + h0 + tid] =
                    p.sink ? p.sink[kUnion ? h0 + (tid & 31) : h0 + tid] : -INFINITY;
            for (int i = tid; i < nhv * kLatent / 8; i += kThreads) {
                const int h = i / (kLatent / 8);
                const int d = i % (kLatent / 8);
                const int64_t orow = kUnion ? out_row(h) : (int64_t)t * p.num_heads + h0 + h;
                *reinterpret_cast<uint4 *>(p.out + orow * kLatent + 8 * d) = make_uint4(0, 0, 0, 0);
            }
            return;
        }
        cluster_sync();   // every split is past its matrix products: partials may land
        if (tid < kNH)    // an empty partial: weight 0 in the merge, its O is never read
            push_stat(smem_u32(gbase), p.splits, split, tid, -INFINITY, 0.f);
        cluster_sync();   // every partial has landed
        cluster_merge_local<kUnion>(p.out, p.lse, p.sink, p.num_heads, p.splits, t, h0, split,
                            reinterpret_cast<const float *>(gbase + kQBytes), reinterpret_cast<const float *>(gbase),
                            reinterpret_cast<float *>(gbase + 1024));
        return;
    }

    const int quad = warp & 3;                            // TMEM lane quadrant of this warp
    const int hs = 16 * ((warp - 1) >> 2);                // workers: first of this warp's 16 heads
    const int key = quad * 32 + lane;                     // softmax: key of the block / value dim of a tile
    // dequant: lane l of worker warp ww takes quarter l % 4 of row 8 ((ww - l / 4) mod 16) + l / 4, so a
    // warp's 8 rows differ in row % 8 (no bank conflicts in the swizzled stores) and the first rows of a
    // block spread over all warps
    const int qtr = lane & 3;
    const int rrow = 8 * (((warp - 1) - (lane >> 2)) & 15) + (lane >> 2);
    const float c2 = p.scale * 1.4426950408889634f;      // logits in log2 units per raw dot product

    if (is_worker)
        asm volatile("cp.async.wait_all;" ::: "memory");   // this thread's Q pieces have landed
    fence_async_smem();
    tc_before();
    __syncthreads();   // slots of blocks 0/1, Q, barriers, TMEM address; the hash set is dead
    tc_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);   // this warp's TMEM lanes

    if (is_issuer) {
        // descriptors: 128-byte swizzle; K-major S^T operands advance 32 B per 16-dim step and one
        // column chunk per 64 dims; MN-major P.V operands advance 2 KB per 16 keys.  Three threads
        // issue, each its own chain (one thread issues a tcgen05.mma about every 70 cycles, more than
        // an M128 N64 K16 product takes the tensor pipe): warp 0 S^T over chunks 0-4 and O^T tiles
        // 0-1, warp 17 S^T over chunks 5-8 (a second accumulator, summed by the softmax), warp 18 O^T
        // tiles 2-3.
        const uint64_t qk_a = sdesc(sK, 16, 1024);
        const uint64_t qk_b = sdesc(sQ, 16, 1024);
        const uint64_t pv_a = sdesc(sK, kChunkBytes, 1024);
        const uint64_t pv_b = sdesc(sP, 1024, 1024);   // one 64-head group along N: LBO unused, kept = SBO
        const bool do_s = warp == 0 || warp == kSIssuerB;
        const bool do_pv = warp == 0 || warp == kPVIssuerB;
        const int c_lo = warp == kSIssuerB ? 5 : 0;             // S^T column chunks of this thread
        const int c_hi = warp == kSIssuerB ? kChunks : 5;
        const uint32_t s_col = warp == kSIssuerB ? kColSb : kColS;
        const int m_lo = warp == kPVIssuerB ? 2 : 0;            // O^T tiles of this thread
        for (int b = 0; b < nblocks; ++b) {
            const uint32_t ph = (uint32_t)(b & 1);
            if (lane == 0) {
                if (do_s) {
#pragma unroll
                    for (int g = 0; g < kGroups; ++g) {
                        if (6 * g >= c_hi || (g == 0 ? 6 : kChunks) <= c_lo)
                            continue;   // no chunk of this thread in group g
                        mbar_wait_one(bar_grp + 8 * g, ph, flags, p.status);   // chunks of group g written
                        tc_after();
#pragma unroll
                        for (int c = 0; c < kChunks; ++c) {
                            if (c < max(c_lo, 6 * g) || c >= min(c_hi, g == 0 ? 6 : kChunks))
                                continue;
                            const uint64_t a = qk_a + (uint64_t)((c * kChunkBytes) >> 4);
                            const uint64_t bq = qk_b + (uint64_t)((c * kQChunkBytes) >> 4);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                umma(tmem + s_col, a + (uint64_t)(2 * k), bq + (uint64_t)(2 * k), kIdescQK,
                                     (c != c_lo || k != 0) ? 1u : 0u);
                        }
                    }
                    umma_commit(bar_s);
                }
                if (do_pv) {
                    mbar_wait_one(bar_p, ph, flags, p.status);   // P^T of block b written
                    tc_after();
                    const int ksteps = min(kBK / 16, (nkeys - b * kBK + 15) / 16);   // 16-key steps holding keys
                    // loops kept rolled: a small issuer body is fetched faster (instruction fetch is
                    // the kernel's main stall, and a CTA runs this code only once a block)
#pragma unroll 1
                    for (int m = m_lo; m < m_lo + 2; ++m) {
                        const uint64_t a = pv_a + (uint64_t)((2 * m * kChunkBytes) >> 4);
#pragma unroll 1
                        for (int kk = 0; kk < ksteps; ++kk)
                            umma(tmem + kColO + 64 * m, a + (uint64_t)(kk * 128), pv_b + (uint64_t)(kk * 128),
                                 kIdescPV, (b > 0 || kk > 0) ? 1u : 0u);
                        umma_commit(bar_pv + 8 * m);   // releases K chunks 2m, 2m+1 (tile 3: also P^T)
                    }
                }
            }
            __syncwarp();
        }
    } else {
        // registers for the next block: 8 latent pieces, 2 rope pieces and the scale word of row rrow
        uint4 pre[10];
        uint32_t pre_sw = 0;
        bool pre_ok = false;
        auto issue_loads = [&](int b) {
            const int sidx = slots[(b % 3) * kBK + rrow];
            pre_ok = sidx >= 0;
            if (pre_ok) {
                const uint8_t *e = p.kv + (int64_t)(kUnion ? sidx & kUnionPosMask : sidx) * kEntryBytes;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    pre[c] = ld_stream(e + 64 * c + 16 * qtr);
                pre[8] = ld_stream(e + kRopeOffset + 16 * qtr);
                pre[9] = ld_stream(e + kRopeOffset + 64 + 16 * qtr);
                pre_sw = __ldg(reinterpret_cast<const unsigned *>(e + kScaleOffset));
            }
        };
        issue_loads(0);
        float m_run = -INFINITY;   // running max (logit units) of head hs + lane % 16

        for (int b = 0; b < nblocks; ++b) {
            const uint32_t ph = (uint32_t)(b & 1);
            // ---- dequant of block b into the K tile, chunk by chunk (zeros for rows without a key)
            {
                const uint32_t rb = sK + (uint32_t)(rrow >> 3) * 1024u + (uint32_t)(rrow & 7) * 128u;
                const uint32_t x7 = (uint32_t)(rrow & 7);
                const uint32_t u0 = (((uint32_t)(2 * qtr)) ^ x7) << 4;
                const uint32_t u1 = (((uint32_t)(2 * qtr + 1)) ^ x7) << 4;
                const uint8_t *enext = p.kv;   // kRide: the next block's entry of row rrow
                bool ok_next = false;
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    if (b > 0 && c < 8 && (c & 1) == 0)
                        mbar_wait(bar_pv + 8 * (c >> 1), ph ^ 1u, flags, p.status);   // P.V of block b-1 released it
                    if (kRide && c == 0 && b + 1 < nblocks) {   // (after the first wait: the slots of b + 1 are visible)
                        const int sidx = slots[((b + 1) % 3) * kBK + rrow];
                        ok_next = sidx >= 0;
                        enext = p.kv + (int64_t)(ok_next ? (kUnion ? sidx & kUnionPosMask : sidx) : 0) * kEntryBytes;
                    }
                    const uint32_t cb = rb + (uint32_t)c * kChunkBytes;
                    if (!pre_ok) {
                        const uint32_t ua = c < 8 ? u0 : ((((uint32_t)qtr) ^ x7) << 4);
                        const uint32_t ub = c < 8 ? u1 : ((((uint32_t)qtr + 4u) ^ x7) << 4);
                        st_shared_v4(cb + ua, 0u, 0u, 0u, 0u);
                        st_shared_v4(cb + ub, 0u, 0u, 0u, 0u);
                    } else if (c < 8) {
                        dequant16_store(pre[c], (pre_sw >> (8 * (c >> 1))) & 0xFFu, cb + u0, cb + u1);
                    } else {   // rope units qtr and qtr + 4, as stored
                        st_shared_v4(cb + ((((uint32_t)qtr) ^ x7) << 4), pre[8].x, pre[8].y, pre[8].z, pre[8].w);
                        st_shared_v4(cb + ((((uint32_t)qtr + 4u) ^ x7) << 4), pre[9].x, pre[9].y, pre[9].z,
                                     pre[9].w);
                    }
                    if (kRide && ok_next && (c == 5 || c == 8)) {
                        // once a chunk group is written, the next block's pieces of that group take its
                        // registers (chunks 0-5, then 6-8)
#pragma unroll
                        for (int cc = 0; cc < kChunks; ++cc) {
                            if (cc > c || (c == 8 && cc < 6))
                                continue;
                            if (cc < 8) {
                                pre[cc] = ld_stream(enext + 64 * cc + 16 * qtr);
                            } else {
                                pre[8] = ld_stream(enext + kRopeOffset + 16 * qtr);
                                pre[9] = ld_stream(enext + kRopeOffset + 64 + 16 * qtr);
                            }
                        }
                    }
                    if (c == 5 || c == kChunks - 1) {
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(bar_grp + 8 * (c == 5 ? 0 : 1));
                    }
                }
                if (kRide) {
                    if (ok_next)   // the next block's scale word, once this block's scales are used
                        pre_sw = __ldg(reinterpret_cast<const unsigned *>(enext + kScaleOffset));
                    pre_ok = ok_next;
                }
            }
            // ---- next block's entries into registers (in one burst unless they rode along); cache
            // slots of block b + 2 (stored below)
            if (!kRide && b + 1 < nblocks)
                issue_loads(b + 1);
            // cache slots of block b + 2: eight per worker warp (lanes 0-7), spread over all warps
            const int ns = 8 * (warp - 1) + lane;
            int next_slot = -1;
            if (lane < 8 && b + 2 < nblocks) {
                const int i = kbeg + (b + 2) * kBK + ns;
                if (i < kend)
                    next_slot = slot_row[i];
            }

            // ---- softmax of block b: this warp's 32 keys (TMEM lanes) x 16 heads
            mbar_wait(bar_s, ph, flags, p.status);
            tc_after();
            bool kv;
            if constexpr (kUnion) {   // warps 1-8 hold the first token's heads, 9-16 the second's
                const int ksl = slots[(b % 3) * kBK + key];
                kv = (b * kBK + key < nkeys) && ksl >= 0 && ((ksl >> (kUnionMaskShift + ((warp - 1) >> 3))) & 1);
            } else {
                kv = (b * kBK + key < nkeys) && slots[(b % 3) * kBK + key] >= 0;
            }
            float *redb = red + (b & 1) * 4 * kNH;
            {   // per-head maxima over this warp's keys; lane j keeps head hs + j
                float mine = -INFINITY;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t sa[8], sb[8];
                    tmem_ld8(lane_base + kColS + hs + 8 * half, sa);
                    tmem_ld8(lane_base + kColSb + hs + 8 * half, sb);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        sa[j] = __float_as_uint(__uint_as_float(sa[j]) + __uint_as_float(sb[j]));
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float m = warp_max(kv ? __uint_as_float(sa[j]) : -INFINITY);
                        mine = lane == 8 * half + j ? m : mine;
                    }
                }
                if (lane < 16)
                    redb[quad * kNH + hs + lane] = mine;
            }
            // only the four warps of these 16 heads exchange maxima: one 128-thread barrier each
            named_bar(2 + ((warp - 1) >> 2), 128);
            // every warp forms the block maxima of its own 16 heads (lane j and j + 16: head hs + j);
            // the four warps sharing the heads compute the same values, so the running max stays in
            // registers and the rescale decision is per warp
            float mcs_l, alpha_l;
            {
                const int hj = hs + (lane & 15);
                const float mb = fmaxf(fmaxf(redb[hj], redb[kNH + hj]), fmaxf(redb[2 * kNH + hj], redb[3 * kNH + hj]));
                float a = 1.f;
                if (m_run == -INFINITY) {
                    m_run = mb;
                } else if (mb > m_run && (mb - m_run) * c2 > kRescaleLog2) {
                    a = exp2f((m_run - mb) * c2);
                    m_run = mb;
                }
                mcs_l = m_run == -INFINITY ? 0.f : m_run * c2;
                alpha_l = a;
            }
            if (__any_sync(0xffffffffu, alpha_l != 1.f)) {   // a max grew past the threshold: rescale O^T, row sums
#pragma unroll 1
                for (int m = 0; m < 10; ++m) {   // four O^T tiles, then the row sums, 8 columns at a time
                    const uint32_t col = ((m >> 1) < 4 ? kColO + 64 * (m >> 1) : kColL) + hs + 8 * (m & 1);
                    uint32_t x[8];
                    tmem_ld8(lane_base + col, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        x[j] = __float_as_uint(__uint_as_float(x[j]) *
                                               __shfl_sync(0xffffffffu, alpha_l, 8 * (m & 1) + j));
                    tmem_st8(lane_base + col, x);
                }
            }
            // P = 2^(s*c - m*c) -> BF16 P^T row `key`; row sums accumulate per lane in TMEM
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int hb = hs + 8 * half;
                uint32_t sv[8], sb[8], l[8];
                tmem_ld8(lane_base + kColS + hb, sv);
                tmem_ld8(lane_base + kColSb + hb, sb);
                if (b > 0)
                    tmem_ld8(lane_base + kColL + hb, l);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    sv[j] = __float_as_uint(__uint_as_float(sv[j]) + __uint_as_float(sb[j]));
                uint32_t pk[4];
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    const float m0 = __shfl_sync(0xffffffffu, mcs_l, 8 * half + j);
                    const float m1 = __shfl_sync(0xffffffffu, mcs_l, 8 * half + j + 1);
                    const float s0 = __uint_as_float(sv[j]);
                    const float s1 = __uint_as_float(sv[j + 1]);
                    const float p0 = kv ? exp2f(fmaf(s0, c2, -m0)) : 0.f;
                    const float p1 = kv ? exp2f(fmaf(s1, c2, -m1)) : 0.f;
                    l[j] = __float_as_uint((b > 0 ? __uint_as_float(l[j]) : 0.f) + p0);
                    l[j + 1] = __float_as_uint((b > 0 ? __uint_as_float(l[j + 1]) : 0.f) + p1);
                    pk[j >> 1] = pack_bf16x2(p0, p1);
                }
                tmem_st8(lane_base + kColL + hb, l);
                st_shared_v4(sP + sw128(key, hb >> 3), pk[0], pk[1], pk[2], pk[3]);
            }
            if (lane < 8 && b + 2 < nblocks)
                slots[((b + 2) % 3) * kBK + ns] = next_slot;   // read after the next softmax barrier
            tmem_st_wait();
            fence_async_smem();
            tc_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_p);
            // warm L2 for block b + 2 (its register loads are issued in block b + 1), after the hand-off
            // of P: the issuing thread waits on the prefetch
            if (lane < 8 && b + 2 < nblocks && next_slot >= 0)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.kv + (int64_t)(kUnion ? next_slot & kUnionPosMask : next_slot) * kEntryBytes),
                             "r"((uint32_t)kEntryBytes) : "memory");
        }

        if (quad == 0 && lane < 16)
            mrun[hs + lane] = m_run;
        float *rede = red + (nblocks & 1) * 4 * kNH;   // the buffer the last block did not use

        // ---- epilogue: row sums across the 128 lanes, then the normalised output or the staged partial
        {
            uint32_t lr[16];
            tmem_ld16(lane_base + kColL + hs, lr);
            tmem_ld_wait();
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = __uint_as_float(lr[j]);
            // halving exchange: after the step with distance d the lane keeps half of its heads,
            // summed with the partner's; at the end lane l holds head 8 b4 + 4 b3 + 2 b2 + b1
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const bool up = lane & 16;
                const float give = up ? v[k] : v[k + 8];
                const float keep = up ? v[k + 8] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const bool up = lane & 8;
                const float give = up ? v[k] : v[k + 4];
                const float keep = up ? v[k + 4] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const bool up = lane & 4;
                const float give = up ? v[k] : v[k + 2];
                const float keep = up ? v[k + 2] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
            }
            {
                const bool up = lane & 2;
                const float give = up ? v[0] : v[1];
                const float keep = up ? v[1] : v[0];
                v[0] = keep + __shfl_xor_sync(0xffffffffu, give, 2);
            }
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
            const int hsel = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
            if ((lane & 1) == 0)
                rede[quad * kNH + hs + hsel] = v[0];
        }
        named_bar(1, kWorkers);
        if (wid < kNH) {
            const int h = wid;
            const float lsum = (rede[h] + rede[kNH + h]) + (rede[2 * kNH + h] + rede[3 * kNH + h]);
            const float m = mrun[h];
            const float ms = m == -INFINITY ? -INFINITY : m * p.scale;   // natural-log units
            if (p.splits == 1) {
                float M = ms;
                float Z = lsum;
                if (p.sink != nullptr && h < nhv) {
                    const float sk = p.sink[kUnion ? h0 + (h & 31) : h0 + h];
                    M = fmaxf(ms, sk);
                    Z = (ms == -INFINITY ? 0.f : lsum * expf(ms - M)) + expf(sk - M);
                }
                fin[h] = (Z > 0.f && ms != -INFINITY) ? expf(ms - M) / Z : 0.f;
                if (p.lse && h < nhv)
                    p.lse[kUnion ? out_row(h) : (int64_t)t * p.num_heads + h0 + h] = Z > 0.f ? M + logf(Z) : -INFINITY;
            } else {
                alpha[h] = ms;
                fin[h] = ms == -INFINITY ? 0.f : lsum;
            }
        }
        named_bar(1, kWorkers);
        // the row sums and statistics above only read this warp's own TMEM stores: they overlap
        // the last block's P.V products, which the output needs
        mbar_wait(bar_pv + 8, (uint32_t)((nblocks - 1) & 1), flags, p.status);    // tiles 0-1 (warp 0)
        mbar_wait(bar_pv + 24, (uint32_t)((nblocks - 1) & 1), flags, p.status);   // tiles 2-3 (warp 18)
        tc_after();
        if (p.splits == 1) {
            uint32_t x[16];
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
                const int dv = 128 * m + key;
                tmem_ld16(lane_base + kColO + 64 * m + hs, x);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int h = hs + j;
                    if (h < nhv) {
                        if constexpr (kUnion)
                            p.out[out_row(h) * kLatent + dv] = bf16_bits(__uint_as_float(x[j]) * fin[h]);
                        else
                            p.out[((int64_t)t * p.num_heads + h0 + h) * kLatent + dv] =
                                bf16_bits(__uint_as_float(x[j]) * fin[h]);
                    }
                }
            }
        }
    }
    if (p.splits > 1) {
        // the split's partial goes straight from TMEM into the shared memory of each head's owner:
        // recv[split][head - owner's first head][512] in the owner's K tile region
        cluster_sync();   // every split is past its matrix products: partials may land
        if (is_worker) {
            const int S = p.splits;
            const int hp = (kNH + S - 1) / S;
            const int nhe = kUnion ? kNH : min(kNH, p.num_heads - h0);   // the merge reads only the heads that exist
            if (wid < nhe)
                push_stat(smem_u32(gbase), S, split, wid, alpha[wid], fin[wid]);
            const uint32_t recv_s = sK;
            const int r0 = hs / hp;   // this warp's 16 heads belong to owners r0, r0 + 1, r0 + 2 at most
            uint32_t x[16];
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
                if (hs >= nhe)   // nhe is a multiple of 16: whole warps skip
                    break;
                const int dv = 128 * m + key;
                tmem_ld16(lane_base + kColO + 64 * m + hs, x);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int h = hs + j;
                    const int r = r0 + (h >= (r0 + 1) * hp) + (h >= (r0 + 2) * hp);
                    const uint32_t off = (uint32_t)(((split * hp + h - r * hp) * kLatent + dv) * 4);
                    if (r == split)
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(recv_s + off), "f"(__uint_as_float(x[j])) : "memory");
                    else
                        st_cluster_f32(map_to_rank(recv_s + off, (uint32_t)r), __uint_as_float(x[j]));
                }
            }
        }
    }
    tc_before();
    __syncthreads();
    tc_after();
    if (is_mma)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    if (p.splits > 1) {
        cluster_sync();   // every partial has landed
        cluster_merge_local<kUnion>(p.out, p.lse, p.sink, p.num_heads, p.splits, t, h0, split,
                            reinterpret_cast<const float *>(gbase + kQBytes), reinterpret_cast<const float *>(gbase),
                            reinterpret_cast<float *>(gbase + 1024));
    }
}

// Launch order of the (token, head group) units for calls whose per-token lists vary in length
// and whose CTAs span more than one wave: CTAs start in index order as multiprocessors free up,
// so giving the units with the longest lists the first indices lets the short ones fill the
// tail (greedy longest-first scheduling).  The key is the estimated number of 128-key blocks
// of the token's list (its top-k length, at most the positions before the window, plus the
// window); one CTA counting-sorts the units by it, descending.  Units with equal keys may come
// in any order: a unit's result does not depend on which CTA computes it.
constexpr int kOrderThreads = 1024;

__device__ __forceinline__ int order_key(const int32_t *topk_lens, const int32_t *seq_lens, int t, int topk_width,
                                         int window)
{
    const int seq = seq_lens[t];
    int n = topk_lens != nullptr ? topk_lens[t] : topk_width;
    n = n < 0 ? 0 : (n > topk_width ? topk_width : n);
    const int swa = seq > 0 ? min(window, seq) : 0;
    const long long est = (long long)min(n, max(seq - swa, 0)) + swa;
    const long long blocks = (est + kBK - 1) / kBK;
    return (int)(blocks < kOrderThreads - 1 ? blocks : kOrderThreads - 1);
}

// In MTP union calls (ulen not null) the units are (request, 32-head group) and the key is the
// number of 128-key blocks of the request's union list.
__global__ void __launch_bounds__(kOrderThreads) decode_order_kernel(const int32_t *topk_lens, const int32_t *seq_lens,
                                                                     int num_tokens, int topk_width, int window,
                                                                     int groups, int32_t *order, const int32_t *ulen)
{
    auto key_of = [&](int u) -> int {
        if (ulen != nullptr)
            return min(kOrderThreads - 1, (max(ulen[u / groups], 0) + 127) / 128);
        return order_key(topk_lens, seq_lens, u / groups, topk_width, window);
    };
    __shared__ int cnt[kOrderThreads];
    __shared__ int wsum[kOrderThreads / 32];
    const int tid = threadIdx.x;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the lengths may come from the previous kernel
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // the decode waits for this grid itself
    cnt[tid] = 0;
    __syncthreads();
    const int units = num_tokens * groups;
    for (int u = tid; u < units; u += kOrderThreads)
        atomicAdd(&cnt[key_of(u)], 1);
    __syncthreads();
    // start[k] = number of units with a larger key: an inclusive scan of the counts in
    // descending key order (thread i holds key kOrderThreads - 1 - i), minus the own count
    const int k = kOrderThreads - 1 - tid;
    const int c = cnt[k];
    int v = c;
    const int lane = tid & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d)
            v += y;
    }
    if (lane == 31)
        wsum[tid >> 5] = v;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < (tid >> 5); ++w)
        before += wsum[w];
    __syncthreads();
    cnt[k] = before + v - c;
    __syncthreads();
    for (int u = tid; u < units; u += kOrderThreads)
        order[atomicAdd(&cnt[key_of(u)], 1)] = u;
}

// Self-test of the bounded waits: one thread waits, at most `limit` SM cycles, on an mbarrier
// that nothing arrives on; the wait gives up, sets the abort flag and the timeout bit, and the
// kernel ends normally.
__global__ void wait_selftest_kernel(long long limit, unsigned *status)
{
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_flag = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait_one(smem_u32(&bar), 0u, &abort_flag, status, limit);
}

}  // namespace

cudaError_t launch_wait_selftest(long long limit, unsigned *status, cudaStream_t stream)
{
    wait_selftest_kernel<<<1, 32, 0, stream>>>(limit, status);
    return cudaGetLastError();
}

int decode_tc_max_splits() { return kMaxSplits; }
int decode_tc_block_keys() { return kBK; }

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
    if (set_smem_once(reinterpret_cast<const void *>(decode_tc_kernel<false, false>), kSmemBytes, kAttrTc) != cudaSuccess)
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
        if (cudaOccupancyMaxActiveClusters(&clusters, reinterpret_cast<const void *>(decode_tc_kernel<false, false>), &cfg) !=
            cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        n = clusters * splits;
    }
    cache[dev][splits] = n;
    return n;
}

int decode_tc_table_bits(int topk_width)
{
    int bits = 6;
    while (bits < kHashBitsMax && (1 << bits) < 4 * topk_width)
        ++bits;
    return bits;
}

cudaError_t launch_decode_tc(const DecodeParams &p, cudaStream_t stream)
{
    if (p.num_tokens <= 0)
        return cudaSuccess;
    if (p.heads_per_group != (p.ulist != nullptr ? kNH / 2 : kNH) || p.num_heads < 1 || p.chunk <= 0 || p.splits < 1 || p.splits > kMaxSplits || p.topk_width < 0 ||
        p.topk_width > kMaxTopkWidth || p.table_bits < 1 || p.table_bits > kHashBitsMax)
        return cudaErrorInvalidValue;
    // CTAs of more than three blocks load the next block's entries during the dequant
    const bool ride = p.chunk > 3 * kBK;
    const bool uni = p.ulist != nullptr;
    const void *kernel;
    AttrSlot slot;
    if (uni) {
        kernel = ride ? reinterpret_cast<const void *>(decode_tc_kernel<true, true>)
                      : reinterpret_cast<const void *>(decode_tc_kernel<false, true>);
        slot = ride ? kAttrTcUnionLong : kAttrTcUnion;
    } else {
        kernel = ride ? reinterpret_cast<const void *>(decode_tc_kernel<true, false>)
                      : reinterpret_cast<const void *>(decode_tc_kernel<false, false>);
        slot = ride ? kAttrTcLong : kAttrTc;
    }
    cudaError_t e = set_smem_once(kernel, kSmemBytes, slot);
    if (e != cudaSuccess)
        return e;
    if (p.order != nullptr) {   // the launch order, ahead of the decode (which waits for it)
        cudaLaunchConfig_t ocfg = {};
        ocfg.gridDim = dim3(1);
        ocfg.blockDim = dim3(kOrderThreads);
        ocfg.stream = stream;
        cudaLaunchAttribute oattr[1];
        oattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        oattr[0].val.programmaticStreamSerializationAllowed = 1;
        ocfg.attrs = oattr;
        ocfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&ocfg, decode_order_kernel, p.topk_lens, p.seq_lens,
                               p.ulist != nullptr ? p.num_tokens / 2 : p.num_tokens, p.topk_width, p.window, p.groups,
                               p.order, p.ulen);
        if (e != cudaSuccess)
            return e;
    }
    // units: (token, 64-head group), or (request, 32-head group) in union calls
    const long long units = p.ulist != nullptr ? (long long)(p.num_tokens / 2) * p.groups : (long long)p.num_tokens * p.groups;
    const long long grid = units * p.splits;
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
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

}  // namespace dsv4
