/*
 * oracle.c -- plain, slow, fp64 CPU reference for DeepSeek-V4 sparse-MLA decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; it exists so that tests, the smoke check and the benchmark's CPU
 * baseline can check the GPU path against an independent restatement of what
 * the path computes.  It shares no code with the CUDA library.
 *
 * Sources (the vLLM pull-request summaries the method is taken from):
 *  - combine: "[ROCm] [DSv4] [Perf] Support DeepSeek v4 MTP" (vllm #43385),
 *    section "关键源码片段 / rocm.py", the _combine_topk_swa_indices_kernel:
 *    per token, valid top-k entries first (in input order), then the sliding
 *    window [pos - swa_len + 1, pos] ascending, swa_len = min(pos + 1, W),
 *    pos = seq_len - query_len + i; an entry is valid when 0 <= idx < N.
 *    Readings taken here (the pages index two different cache regions, this
 *    path one): entries > pos, entries inside the window and repeats (all but
 *    the first occurrence) are dropped, and the survivors are compacted.
 *  - dequant: "feat: add DeepSeek-V4 XPU attention decode path" (vllm #42953),
 *    section "xpu_sparse_decode_fp8.py", _dequant_gather_slots_kernel:
 *    value = fp8_e4m3 * exp2(ue8m0 - 127); a negative slot contributes zeros;
 *    block_idx = slot // block_size, pos_in_block = slot % block_size; the
 *    BF16 RoPE part is copied as stored.
 *  - logical -> physical: "Enable DeepSeek V4 and GLM-5.1 on SM120"
 *    (vllm #43477), section "flashinfer_mla_sparse_sm120.py",
 *    triton_convert_req_index_to_global_index(req_id_per_token, block_table, ...).
 *  - attention: the same page's forward_mqa: output [T, h, kv_lora_rank=512]
 *    over MQA keys (one KV head, V = the 512-d latent), sinks supported
 *    (flashinfer_sparse.py, supports_sink).  Written here as its plain
 *    definition: s_j = scale * q . k_j over 576 dims; with an optional sink
 *    logit sigma (in the same units as s), Z = sum_j e^{s_j} + e^{sigma},
 *    lse = ln Z, out = sum_j e^{s_j - lse} v_j.
 *  - fused Q per-head RMSNorm + GPT-J RoPE + FP8/UE8M0 KV insert (the step before the path):
 *    "feat: add DeepSeek-V4 XPU attention decode path" (vllm #42953), 实现拆解 4; readings at
 *    oracle_qnorm_rope / oracle_kv_insert.
 *  - top-k selection from indexer scores (what produces topk_idx): "[Model] DeepSeek V4"
 *    (vllm #40860), 实现拆解 2; the selection rule is written out with its readings at
 *    oracle_topk_select.
 *  - merge of split partial results: the log-sum-exp combination, written out
 *    from its definition (not on the pages; needed when one token's keys are
 *    split over several workers).
 *
 * Cache entry layout (656 bytes per token, this library's own layout):
 *   [0,512) E4M3FN latent codes, [512,640) 64 x BF16 rope (little endian),
 *   [640,644) four UE8M0 scale bytes (byte b scales latent dims [128b,128b+128)),
 *   [644,656) padding.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_ENTRY_BYTES 656
#define OR_LATENT 512
#define OR_ROPE 64
#define OR_DIM 576
#define OR_ROPE_OFF 512
#define OR_SCALE_OFF 640
#define OR_SCALE_BLOCK 128

/* OCP FP8 E4M3FN: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0
 * is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there are no infinities. */
double oracle_e4m3_to_double(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* UE8M0: an unsigned 8-bit exponent, value 2^(e - 127); 0xFF is NaN. */
double oracle_ue8m0_to_double(uint8_t e)
{
    if (e == 0xFF)
        return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* BF16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One cache entry -> the 576-d key (512 latent then 64 rope). */
void oracle_dequant_entry(const uint8_t *entry, double *k)
{
    for (int d = 0; d < OR_LATENT; ++d) {
        double scale = oracle_ue8m0_to_double(entry[OR_SCALE_OFF + d / OR_SCALE_BLOCK]);
        k[d] = oracle_e4m3_to_double(entry[d]) * scale;
    }
    for (int i = 0; i < OR_ROPE; ++i) {
        uint16_t h = (uint16_t)entry[OR_ROPE_OFF + 2 * i] | (uint16_t)((uint16_t)entry[OR_ROPE_OFF + 2 * i + 1] << 8);
        k[OR_LATENT + i] = oracle_bf16_to_double(h);
    }
}

/* Compressed-region combine: the page's full variant of the combine ("[ROCm] [DSv4] [Perf]
 * Support DeepSeek v4 MTP", vllm #43385, section 关键源码片段 / rocm.py,
 * _combine_topk_swa_indices_kernel).  Each request b owns a gathered region of M entries:
 * N compressed entries (what top-k indexes), then raw positions from
 * gather_start = seq_len - gather_len on.  Its tokens are [query_start_loc[b], ...[b + 1])
 * (relative to query_start_loc[0]); token i of a request of query_len tokens sits at
 * pos = seq_len - query_len + i and gets
 *   topk_len = min((pos + 1) / C, TOP_K) entries  M*b + v  for its top-k values v in [0, N)
 *                                                 (-1 for any other value, kept in place),
 *   swa_len  = min(pos + 1, W) window entries       M*b + N + (pos - swa_len + 1 - gather_start) + j,
 * length topk_len + swa_len.  No dedup: the two parts index different regions.
 * Readings: a token with pos + 1 <= 0 gets no entries (the page's integer arithmetic would give a
 * negative length); entries past the length are -1 (the page leaves them unwritten); TOP_K must
 * not exceed the top-k row width (so the page's fallback read of entry 0 for offsets past the
 * row never happens).  Returns 0, or 1 for arguments outside those rules. */
int oracle_combine_compressed(const int32_t *topk_idx, int64_t topk_stride, int32_t topk_width,
                              const int32_t *query_start_loc, const int32_t *seq_lens, const int32_t *gather_lens,
                              int32_t num_reqs, int32_t region_stride, int32_t compressed_len, int32_t top_k,
                              int32_t compress_ratio, int32_t window, int32_t *combined, int64_t combined_stride,
                              int32_t combined_width, int32_t *combined_lens)
{
    if (top_k < 0 || top_k > topk_width || compress_ratio < 1 || window < 0 || combined_width < top_k + window)
        return 1;
    const int64_t base = query_start_loc[0];
    for (int32_t b = 0; b < num_reqs; ++b) {
        const int64_t qs = query_start_loc[b] - base;
        const int64_t qe = query_start_loc[b + 1] - base;
        const int64_t start_pos = (int64_t)seq_lens[b] - (qe - qs);
        const int64_t gather_start = (int64_t)seq_lens[b] - gather_lens[b];
        const int64_t region = (int64_t)region_stride * b;
        for (int64_t t = qs; t < qe; ++t) {
            const int64_t pos = start_pos + (t - qs);
            int64_t tk = 0, sw = 0;
            if (pos + 1 > 0) {
                tk = (pos + 1) / compress_ratio;
                if (tk > top_k)
                    tk = top_k;
                sw = pos + 1 < window ? pos + 1 : window;
            }
            int32_t *row = combined + t * combined_stride;
            const int32_t *in = topk_idx + t * topk_stride;
            for (int64_t k = 0; k < tk; ++k) {
                const int32_t v = in[k];
                row[k] = (v >= 0 && v < compressed_len) ? (int32_t)(region + v) : -1;
            }
            for (int64_t j = 0; j < sw; ++j)
                row[tk + j] = (int32_t)(region + compressed_len + (pos - sw + 1 - gather_start) + j);
            for (int64_t k = tk + sw; k < combined_width; ++k)
                row[k] = -1;
            combined_lens[t] = (int32_t)(tk + sw);
        }
    }
    return 0;
}

/* Top-k selection from indexer scores: the step that produces topk_idx ("[Model] DeepSeek V4"
 * (vllm #40860), 实现拆解 2: the MLA wrapper runs the Indexer ahead of the sparse attention).
 * The pages print no selection rule; this is the plain definition, with these readings: row t's
 * candidates are positions [0, n), n = num_cand[t] clamped to [0, width]; the selected set is
 * the min(K, n) candidates that come first in the total order "larger score first, then smaller
 * position", where -0 equals +0 and a NaN score ranks below every number; the output row holds
 * the selected positions in ascending order, then -1; topk_lens[t] = min(K, n).
 * Returns 0, or 1 for K < 1. */
struct topk_item {
    double v;      /* the score (0 for NaN) */
    int nan;       /* 1 for a NaN score */
    int32_t pos;
};

static int topk_before(const void *pa, const void *pb)
{
    const struct topk_item *a = pa, *b = pb;
    if (a->nan != b->nan)
        return a->nan ? 1 : -1;                           /* NaN after every number */
    if (!a->nan && a->v != b->v)
        return a->v > b->v ? -1 : 1;                      /* larger score first */
    return a->pos < b->pos ? -1 : (a->pos > b->pos);      /* then the smaller position */
}

static int ascending_i32(const void *pa, const void *pb)
{
    const int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return a < b ? -1 : (a > b);
}

int oracle_topk_select(const float *scores, int64_t score_stride, int32_t width, const int32_t *num_cand,
                       int32_t num_tokens, int32_t top_k, int32_t *topk_idx, int64_t topk_stride,
                       int32_t *topk_lens)
{
    if (top_k < 1)
        return 1;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t n = num_cand[t];
        if (n < 0)
            n = 0;
        if (n > width)
            n = width;
        struct topk_item *items = malloc(sizeof(struct topk_item) * (size_t)(n > 0 ? n : 1));
        for (int64_t p = 0; p < n; ++p) {
            const float x = scores[t * score_stride + p];
            items[p].nan = isnan(x) ? 1 : 0;
            items[p].v = items[p].nan ? 0.0 : (double)x + 0.0;   /* + 0.0 turns -0 into +0 */
            items[p].pos = (int32_t)p;
        }
        qsort(items, (size_t)n, sizeof(struct topk_item), topk_before);
        const int64_t m = n < top_k ? n : top_k;
        int32_t *row = topk_idx + t * topk_stride;
        for (int64_t k = 0; k < m; ++k)
            row[k] = items[k].pos;
        qsort(row, (size_t)m, sizeof(int32_t), ascending_i32);
        for (int64_t k = m; k < top_k; ++k)
            row[k] = -1;
        topk_lens[t] = (int32_t)m;
        free(items);
    }
    return 0;
}

/* ---- fused Q per-head RMSNorm + GPT-J RoPE + FP8/UE8M0 KV insert ("feat: add DeepSeek-V4 XPU
 * attention decode path" (vllm #42953), 实现拆解 4: xpu_qnorm_rope_kv_fp8_insert, called from
 * forward_mqa as (q, kv, kv_cache, slot_mapping, positions, ...) before the decode).  The page
 * names the steps; the readings taken here:
 *  - each query head (576 dims) is divided by sqrt(mean of its squares + eps), then multiplied
 *    by an optional weight w[576], with no rounding in between;
 *  - GPT-J RoPE rotates the interleaved pairs (512 + 2i, 513 + 2i), i < 32, of the normalised
 *    query and of the key by the angle whose cosine and sine are cos_sin[pos][i] and
 *    cos_sin[pos][32 + i] (a caller-made fp32 table, as rotary caches are);
 *  - the key's latent (512 dims) is quantised as the cache format stores it: per 128 values the
 *    smallest integer e with 448 * 2^e >= amax (0 for amax 0, clamped to [-127, 127]), codes =
 *    E4M3 round-to-nearest-even of x * 2^-e, scale byte e + 127; the rotated rope part is
 *    rounded to BF16; the entry's 12 padding bytes are zero;
 *  - the entry goes to slot slot_mapping[t]; a negative slot writes nothing (a padding token);
 *    a slot past the cache or a position outside the table writes nothing and is counted;
 *    such a token's query is normalised but not rotated.
 * Every result is rounded once, from fp64. */
static uint16_t bf16_from_double(double x)
{
    if (x == 0.0)
        return signbit(x) ? 0x8000u : 0u;
    int k;
    frexp(x, &k);                          /* |x| in [2^(k-1), 2^k) */
    int e = k - 1;
    if (e < -126)
        e = -126;                          /* BF16 subnormals share the quantum 2^-133 */
    const double quantum = ldexp(1.0, e - 7);
    const double r = rint(x / quantum) * quantum;   /* nearest, ties to even */
    const float f = (float)r;              /* exact: at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* E4M3FN code of a finite |y| <= 448, round to nearest, ties to even. */
uint8_t oracle_e4m3_encode(double y)
{
    const uint8_t s = signbit(y) ? 0x80u : 0u;
    const double a = fabs(y);
    if (a < ldexp(1.0, -6))                /* subnormal codes: value = q * 2^-9 (q = 8: 2^-6, code 8) */
        return (uint8_t)(s | (uint8_t)rint(a * 512.0));
    int k;
    const double m = frexp(a, &k);         /* a = m * 2^k, m in [0.5, 1) */
    int q = (int)rint((2.0 * m - 1.0) * 8.0);   /* a = (1 + q/8) * 2^(k-1) */
    int ef = k - 1 + 7;
    if (q == 8) {
        q = 0;
        ++ef;
    }
    return (uint8_t)(s | (uint8_t)(ef << 3) | (uint8_t)q);
}

/* Smallest integer e with 448 * 2^e >= amax (0 for amax 0), clamped to [-127, 127]. */
static int ue8m0_exponent_of(double amax)
{
    if (amax <= 0.0)
        return 0;
    int e = -127;
    while (e < 127 && 448.0 * ldexp(1.0, e) < amax)
        ++e;
    return e;
}

/* Rotates the pair (x, y) by the angle of (c, s). */
static void rope_pair(double *x, double *y, double c, double s)
{
    const double a = *x, b = *y;
    *x = a * c - b * s;
    *y = a * s + b * c;
}

/* Queries: q, q_out BF16 bits [T, H, 576] (token strides in elements).  Returns the number of
 * tokens whose position is outside [0, max_pos). */
int64_t oracle_qnorm_rope(const uint16_t *q, int64_t q_stride, int32_t T, int32_t H, const float *norm_w, double eps,
                          const int64_t *positions, const float *cos_sin, int32_t max_pos, uint16_t *q_out,
                          int64_t q_out_stride)
{
    int64_t bad = 0;
    double x[OR_DIM];
    for (int32_t t = 0; t < T; ++t) {
        const int64_t pos = positions[t];
        const int rot = pos >= 0 && pos < max_pos;
        bad += !rot;
        for (int32_t h = 0; h < H; ++h) {
            const uint16_t *in = q + t * q_stride + (int64_t)h * OR_DIM;
            double ss = 0.0;
            for (int d = 0; d < OR_DIM; ++d) {
                x[d] = oracle_bf16_to_double(in[d]);
                ss += x[d] * x[d];
            }
            const double r = 1.0 / sqrt(ss / OR_DIM + eps);
            for (int d = 0; d < OR_DIM; ++d)
                x[d] = x[d] * r * (norm_w ? (double)norm_w[d] : 1.0);
            if (rot)
                for (int i = 0; i < OR_ROPE / 2; ++i)
                    rope_pair(&x[OR_LATENT + 2 * i], &x[OR_LATENT + 2 * i + 1], (double)cos_sin[pos * 64 + i],
                              (double)cos_sin[pos * 64 + 32 + i]);
            uint16_t *o = q_out + t * q_out_stride + (int64_t)h * OR_DIM;
            for (int d = 0; d < OR_DIM; ++d)
                o[d] = bf16_from_double(x[d]);
        }
    }
    return bad;
}

/* Keys: kv BF16 bits [T, 576] (token stride in elements) into cache entries uint8 [num_slots, 656].
 * Returns the number of tokens with a slot past the cache or a position outside the table. */
int64_t oracle_kv_insert(const uint16_t *kv, int64_t kv_stride, int32_t T, const int64_t *slots,
                         const int64_t *positions, const float *cos_sin, int32_t max_pos, uint8_t *cache,
                         int64_t num_slots)
{
    int64_t bad = 0;
    double x[OR_DIM];
    for (int32_t t = 0; t < T; ++t) {
        const int64_t slot = slots[t], pos = positions[t];
        if (slot < 0)
            continue;
        if (slot >= num_slots || pos < 0 || pos >= max_pos) {
            ++bad;
            continue;
        }
        for (int d = 0; d < OR_DIM; ++d)
            x[d] = oracle_bf16_to_double(kv[t * kv_stride + d]);
        uint8_t *e = cache + slot * OR_ENTRY_BYTES;
        memset(e, 0, OR_ENTRY_BYTES);
        for (int b = 0; b < OR_LATENT / OR_SCALE_BLOCK; ++b) {
            double amax = 0.0;
            for (int d = b * OR_SCALE_BLOCK; d < (b + 1) * OR_SCALE_BLOCK; ++d)
                amax = fabs(x[d]) > amax ? fabs(x[d]) : amax;
            const int ex = ue8m0_exponent_of(amax);
            for (int d = b * OR_SCALE_BLOCK; d < (b + 1) * OR_SCALE_BLOCK; ++d)
                e[d] = oracle_e4m3_encode(ldexp(x[d], -ex));
            e[OR_SCALE_OFF + b] = (uint8_t)(ex + 127);
        }
        for (int i = 0; i < OR_ROPE / 2; ++i)
            rope_pair(&x[OR_LATENT + 2 * i], &x[OR_LATENT + 2 * i + 1], (double)cos_sin[pos * 64 + i],
                      (double)cos_sin[pos * 64 + 32 + i]);
        for (int i = 0; i < OR_ROPE; ++i) {
            const uint16_t h = bf16_from_double(x[OR_LATENT + i]);
            e[OR_ROPE_OFF + 2 * i] = (uint8_t)(h & 0xFF);
            e[OR_ROPE_OFF + 2 * i + 1] = (uint8_t)(h >> 8);
        }
    }
    return bad;
}

/* Combined index list of one token.  Returns its length L; row[0..L) holds
 * the kept top-k entries then the window, row[L..width) is -1. */
int oracle_combine_token(const int32_t *topk_row, int32_t n_topk, int32_t seq_len, int32_t window,
                         int32_t *row, int32_t width)
{
    int32_t pos = seq_len - 1;
    int32_t win_lo = pos - window + 1;
    if (win_lo < 0)
        win_lo = 0;
    int32_t L = 0;
    for (int32_t i = 0; i < n_topk; ++i) {
        int32_t v = topk_row[i];
        if (v < 0 || v > pos)
            continue;                 /* invalid or not causal */
        if (v >= win_lo)
            continue;                 /* already covered by the window */
        int dup = 0;
        for (int32_t j = 0; j < L; ++j) {
            if (row[j] == v) {
                dup = 1;
                break;
            }
        }
        if (!dup)
            row[L++] = v;
    }
    for (int32_t p = win_lo; p <= pos; ++p)
        row[L++] = p;
    for (int32_t j = L; j < width; ++j)
        row[j] = -1;
    return L;
}

/* Batched combine; returns 0, or -1 when a row would not fit in `width`. */
int oracle_combine(const int32_t *topk_idx, int64_t topk_stride, int32_t topk_width, const int32_t *topk_lens,
                   const int32_t *seq_lens, int32_t num_tokens, int32_t window, int32_t *combined,
                   int64_t combined_stride, int32_t combined_width, int32_t *combined_lens)
{
    int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * ((size_t)topk_width + (size_t)(window > 0 ? window : 0) + 1));
    if (!tmp)
        return -1;
    int rc = 0;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int32_t n = topk_lens ? topk_lens[t] : topk_width;
        if (n < 0)
            n = 0;
        if (n > topk_width)
            n = topk_width;
        int32_t L = oracle_combine_token(topk_idx + (int64_t)t * topk_stride, n, seq_lens[t], window, tmp,
                                         topk_width + (window > 0 ? window : 0));
        if (L > combined_width) {
            rc = -1;
            L = combined_width;
        }
        memcpy(combined + (int64_t)t * combined_stride, tmp, sizeof(int32_t) * (size_t)L);
        for (int32_t j = L; j < combined_width; ++j)
            combined[(int64_t)t * combined_stride + j] = -1;
        combined_lens[t] = L;
    }
    free(tmp);
    return rc;
}

/* Attention of one head over an explicit key list keys[L][576] (V = first 512 dims).
 * q is the 576-d query in fp64.  has_sink selects the optional sink logit. */
void oracle_attend(const double *q, const double *keys, int32_t L, double softmax_scale, int has_sink, double sink,
                   double *out, double *lse)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double m = -INFINITY;
    for (int32_t j = 0; j < L; ++j) {
        double acc = 0.0;
        for (int d = 0; d < OR_DIM; ++d)
            acc += q[d] * keys[(int64_t)j * OR_DIM + d];
        s[j] = softmax_scale * acc;
        if (s[j] > m)
            m = s[j];
    }
    if (has_sink && sink > m)
        m = sink;
    for (int d = 0; d < OR_LATENT; ++d)
        out[d] = 0.0;
    if (m == -INFINITY) {           /* no key and no (finite) sink */
        *lse = -INFINITY;
        free(s);
        return;
    }
    double z = 0.0;
    for (int32_t j = 0; j < L; ++j)
        z += exp(s[j] - m);
    if (has_sink)
        z += exp(sink - m);
    double l = m + log(z);
    for (int32_t j = 0; j < L; ++j) {
        double w = exp(s[j] - l);
        for (int d = 0; d < OR_LATENT; ++d)
            out[d] += w * keys[(int64_t)j * OR_DIM + d];
    }
    *lse = l;
    free(s);
}

/* Merge of S partial results over disjoint key sets, each given as
 * (lse_c = ln sum_{j in c} e^{s_j}, out_c normalised within c), plus the
 * optional sink: lse = ln(sum_c e^{lse_c} + e^{sink}), out = sum_c e^{lse_c - lse} out_c. */
void oracle_merge(int32_t S, const double *lse_parts, const double *out_parts, int has_sink, double sink,
                  double *out, double *lse)
{
    double m = -INFINITY;
    for (int32_t c = 0; c < S; ++c)
        if (lse_parts[c] > m)
            m = lse_parts[c];
    if (has_sink && sink > m)
        m = sink;
    for (int d = 0; d < OR_LATENT; ++d)
        out[d] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double z = 0.0;
    for (int32_t c = 0; c < S; ++c)
        z += exp(lse_parts[c] - m);
    if (has_sink)
        z += exp(sink - m);
    double l = m + log(z);
    for (int32_t c = 0; c < S; ++c) {
        double w = exp(lse_parts[c] - l);
        if (w == 0.0)
            continue;
        for (int d = 0; d < OR_LATENT; ++d)
            out[d] += w * out_parts[(int64_t)c * OR_LATENT + d];
    }
    *lse = l;
}

typedef struct {
    const uint16_t *q;
    int64_t q_token_stride;
    const uint8_t *kv_cache;
    int32_t num_blocks, page_block;
    const int32_t *block_table;
    int64_t bt_stride;
    int32_t max_blocks, num_reqs;
    const int32_t *req_idx;
    const int32_t *topk_idx;
    int64_t topk_stride;
    int32_t topk_width;
    const int32_t *topk_lens, *seq_lens;
    int32_t num_tokens, num_heads, window;
    int32_t head_begin, head_end;
    const float *sink;
    double softmax_scale;
    double *out, *lse;
    const int32_t *tokens;
    int32_t n_tokens_todo;
    int32_t worker, n_workers;
    int64_t bad;
} decode_job;

static void *decode_worker(void *arg)
{
    decode_job *jb = (decode_job *)arg;
    int32_t cap = jb->topk_width + (jb->window > 0 ? jb->window : 0) + 1;
    int32_t *list = (int32_t *)malloc(sizeof(int32_t) * (size_t)cap);
    double *keys = (double *)malloc(sizeof(double) * (size_t)cap * OR_DIM);
    double qh[OR_DIM];
    jb->bad = 0;
    for (int32_t w = jb->worker; w < jb->n_tokens_todo; w += jb->n_workers) {
        int32_t t = jb->tokens ? jb->tokens[w] : w;
        int32_t n = jb->topk_lens ? jb->topk_lens[t] : jb->topk_width;
        if (n < 0)
            n = 0;
        if (n > jb->topk_width)
            n = jb->topk_width;
        int32_t L = oracle_combine_token(jb->topk_idx + (int64_t)t * jb->topk_stride, n, jb->seq_lens[t],
                                         jb->window, list, cap);
        int32_t row = jb->req_idx ? jb->req_idx[t] : t;
        int32_t nk = 0;
        for (int32_t j = 0; j < L; ++j) {
            int32_t idx = list[j];
            int32_t blk = idx / jb->page_block;
            int32_t off = idx % jb->page_block;
            if (row < 0 || row >= jb->num_reqs || blk >= jb->max_blocks) {
                jb->bad++;
                continue;
            }
            int32_t phys = jb->block_table[(int64_t)row * jb->bt_stride + blk];
            if (phys < 0 || phys >= jb->num_blocks) {
                jb->bad++;
                continue;
            }
            int64_t slot = (int64_t)phys * jb->page_block + off;
            oracle_dequant_entry(jb->kv_cache + slot * OR_ENTRY_BYTES, keys + (int64_t)nk * OR_DIM);
            nk++;
        }
        int32_t nh = jb->head_end - jb->head_begin;
        for (int32_t h = jb->head_begin; h < jb->head_end; ++h) {
            const uint16_t *qp = jb->q + (int64_t)t * jb->q_token_stride + (int64_t)h * OR_DIM;
            for (int d = 0; d < OR_DIM; ++d)
                qh[d] = oracle_bf16_to_double(qp[d]);
            int64_t r = (int64_t)w * nh + (h - jb->head_begin);
            double *o = jb->out + r * OR_LATENT;
            oracle_attend(qh, keys, nk, jb->softmax_scale, jb->sink != NULL, jb->sink ? (double)jb->sink[h] : 0.0, o,
                          jb->lse + r);
        }
    }
    free(list);
    free(keys);
    return NULL;
}

/* Full decode for a subset of tokens (tokens == NULL: all, in order) and the heads
 * [head_begin, head_end).  out is fp64 [n_todo, head_end - head_begin, 512] and
 * lse fp64 [n_todo, head_end - head_begin], rows in the order of `tokens`.  Keys
 * whose block-table lookup is out of range are skipped and counted; the count is
 * returned. */
int64_t oracle_sparse_mla_decode(const uint16_t *q, int64_t q_token_stride, const uint8_t *kv_cache,
                                 int32_t num_blocks, int32_t page_block, const int32_t *block_table,
                                 int64_t bt_stride, int32_t max_blocks, int32_t num_reqs, const int32_t *req_idx,
                                 const int32_t *topk_idx, int64_t topk_stride, int32_t topk_width,
                                 const int32_t *topk_lens, const int32_t *seq_lens, int32_t num_tokens,
                                 int32_t num_heads, int32_t window, const float *sink, double softmax_scale,
                                 double *out, double *lse, const int32_t *tokens, int32_t n_tokens_todo,
                                 int32_t head_begin, int32_t head_end, int32_t n_threads)
{
    if (n_threads < 1)
        n_threads = 1;
    if (tokens == NULL)
        n_tokens_todo = num_tokens;
    if (n_threads > n_tokens_todo)
        n_threads = n_tokens_todo > 0 ? n_tokens_todo : 1;
    decode_job *jobs = (decode_job *)calloc((size_t)n_threads, sizeof(decode_job));
    pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    for (int32_t i = 0; i < n_threads; ++i) {
        decode_job *jb = &jobs[i];
        jb->q = q;
        jb->q_token_stride = q_token_stride;
        jb->kv_cache = kv_cache;
        jb->num_blocks = num_blocks;
        jb->page_block = page_block;
        jb->block_table = block_table;
        jb->bt_stride = bt_stride;
        jb->max_blocks = max_blocks;
        jb->num_reqs = num_reqs;
        jb->req_idx = req_idx;
        jb->topk_idx = topk_idx;
        jb->topk_stride = topk_stride;
        jb->topk_width = topk_width;
        jb->topk_lens = topk_lens;
        jb->seq_lens = seq_lens;
        jb->num_tokens = num_tokens;
        jb->num_heads = num_heads;
        jb->window = window;
        jb->head_begin = head_begin;
        jb->head_end = head_end;
        jb->sink = sink;
        jb->softmax_scale = softmax_scale;
        jb->out = out;
        jb->lse = lse;
        jb->tokens = tokens;
        jb->n_tokens_todo = n_tokens_todo;
        jb->worker = i;
        jb->n_workers = n_threads;
    }
    for (int32_t i = 1; i < n_threads; ++i)
        pthread_create(&th[i], NULL, decode_worker, &jobs[i]);
    decode_worker(&jobs[0]);
    int64_t bad = jobs[0].bad;
    for (int32_t i = 1; i < n_threads; ++i) {
        pthread_join(th[i], NULL);
        bad += jobs[i].bad;
    }
    free(jobs);
    free(th);
    return bad;
}
