"""Seeded synthetic inputs for DeepSeek-V4 sparse-MLA decode.

This module builds the arrays that one decode step consumes:
  * BF16 queries ``q`` [T, H, 576] (stored as uint16 bit patterns),
  * the paged FP8 KV cache ``kv_cache`` uint8 [num_blocks, page, 656],
  * a shuffled ``block_table`` int32 [R, max_blocks] and ``req_idx`` [T],
  * per-token top-k position lists ``topk_idx`` int32 [T, K] (-1 padded),
    optional ``topk_lens`` [T], causal lengths ``seq_lens`` [T] (= pos + 1),
  * the sliding-window size, optional per-head ``sink`` logits, the softmax scale.

It is shared by the CPU oracle's tests and by the GPU path's tests and
benchmark, so it deliberately holds none of the decode arithmetic: no index
combine, no dequantisation, no attention.  The only numeric work here is
turning random draws into the cache's byte format, i.e. what a KV-cache
insert would write:
  * E4M3 (OCP FP8 E4M3FN: bias 7, max 448, no infinities, NaN = S.1111.111)
    with round-to-nearest-even,
  * one UE8M0 power-of-two scale 2^e per 128 latent values, with e the
    smallest integer such that 448 * 2^e >= amax of the block
    (i.e. 2^ceil(log2(amax/448)); amax = 0 gives e = 0),
  * BF16 with round-to-nearest-even for the RoPE part and for Q.

Cache entry byte layout (656 bytes, 41 x 16 B, token-major inside a page):
  [0, 512)   512 E4M3 latent codes
  [512, 640) 64 BF16 RoPE values, little-endian
  [640, 644) 4 UE8M0 scale bytes (block b covers latent dims [128b, 128b+128))
  [644, 656) zero padding

Seeds: workload n of the five decode workloads uses PCG64 seeded with 1000 + n.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

ENTRY_BYTES = 656
LATENT_DIM = 512
ROPE_DIM = 64
HEAD_DIM = LATENT_DIM + ROPE_DIM
ROPE_OFFSET = 512
SCALE_OFFSET = 640
SCALE_BLOCK = 128
E4M3_MAX = 448.0


# ----------------------------------------------------------------------------
# byte-format encoders (input construction only)
# ----------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float values to BF16 (nearest-even) and return the uint16 bit patterns."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """Encode values with |y| <= 448 as E4M3FN codes, round-to-nearest-even."""
    y = np.asarray(y, dtype=np.float64)
    if np.any(~np.isfinite(y)) or np.any(np.abs(y) > E4M3_MAX):
        raise ValueError("e4m3_encode expects finite |y| <= 448")
    sign = np.signbit(y).astype(np.int32)
    a = np.abs(y)
    # subnormal range (a < 2^-6): value = q * 2^-9, q in 0..8 (q == 8 is the smallest normal, code 8)
    code_sub = np.rint(a * 2.0 ** 9).astype(np.int32)
    m, k = np.frexp(a)                     # a = m * 2^k, m in [0.5, 1)
    q = np.rint((2.0 * m - 1.0) * 8.0).astype(np.int32)   # a = (1 + q/8) * 2^(k-1)
    carry = (q == 8).astype(np.int32)
    code_nrm = ((k.astype(np.int32) - 1 + carry + 7) << 3) | (q * (1 - carry))
    code = np.where(a < 2.0 ** -6, code_sub, code_nrm) | (sign << 7)
    return code.astype(np.uint8)


def ue8m0_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer e with 448 * 2^e >= amax (0 where amax == 0), clamped to [-127, 127]."""
    amax = np.asarray(amax, dtype=np.float64)
    e = np.zeros(amax.shape, dtype=np.int64)
    pos = amax > 0
    if np.any(pos):
        _, k = np.frexp(amax[pos] / E4M3_MAX)
        k = k.astype(np.int64)
        # frexp gives a candidate within one of the answer; settle it with exact comparisons
        k = np.where(E4M3_MAX * np.ldexp(1.0, k - 1) >= amax[pos], k - 1, k)
        k = np.where(E4M3_MAX * np.ldexp(1.0, k) < amax[pos], k + 1, k)
        e[pos] = k
    return np.clip(e, -127, 127)


def quantize_entries(latent: np.ndarray, rope: np.ndarray) -> np.ndarray:
    """Pack float latent [N, 512] and rope [N, 64] into cache entries uint8 [N, 656]."""
    latent = np.asarray(latent, dtype=np.float64)
    n = latent.shape[0]
    blocks = latent.reshape(n, LATENT_DIM // SCALE_BLOCK, SCALE_BLOCK)
    e = ue8m0_exponent(np.abs(blocks).max(axis=2))                  # [N, 4]
    scaled = blocks * np.ldexp(1.0, -e)[:, :, None]                   # exact power-of-two scaling
    codes = e4m3_encode(scaled).reshape(n, LATENT_DIM)
    out = np.zeros((n, ENTRY_BYTES), dtype=np.uint8)
    out[:, :LATENT_DIM] = codes
    out[:, ROPE_OFFSET:SCALE_OFFSET] = bf16_bits(rope).astype('<u2').view(np.uint8).reshape(n, 2 * ROPE_DIM)
    out[:, SCALE_OFFSET:SCALE_OFFSET + 4] = (e + 127).astype(np.uint8)
    return out


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    """One decode step's inputs (host numpy arrays)."""
    name: str
    q: np.ndarray                 # uint16 [T, H, 576] BF16 bits
    kv_cache: np.ndarray          # uint8 [num_blocks, page, 656]
    block_table: np.ndarray       # int32 [R, max_blocks]; -1 beyond a request's pages
    req_idx: Optional[np.ndarray]  # int32 [T] token -> block_table row, None = identity
    topk_idx: np.ndarray          # int32 [T, K], -1 padded
    topk_lens: Optional[np.ndarray]  # int32 [T] or None (= K)
    seq_lens: np.ndarray          # int32 [T], causal visible length (pos + 1)
    window: int
    sink: Optional[np.ndarray]    # float32 [H] or None
    softmax_scale: float
    page: int

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def topk_width(self) -> int:
        return int(self.topk_idx.shape[1])

    @property
    def num_blocks(self) -> int:
        return int(self.kv_cache.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def num_reqs(self) -> int:
        return int(self.block_table.shape[0])


def _distinct_uniform(rng, hi: int, n: int) -> np.ndarray:
    """n distinct integers uniform in [0, hi), in random order."""
    n = min(n, hi)
    if n <= 0:
        return np.zeros(0, dtype=np.int64)
    if n * 4 >= hi:
        return rng.permutation(hi)[:n].astype(np.int64)
    chosen = np.unique(rng.integers(0, hi, size=2 * n + 16))
    while chosen.size < n:
        chosen = np.unique(np.concatenate([chosen, rng.integers(0, hi, size=n)]))
    return rng.permutation(chosen)[:n].astype(np.int64)


def _distinct_biased(rng, hi: int, n: int, recent: int, recent_frac: float) -> np.ndarray:
    """n distinct positions in [0, hi): a recent_frac share weighted onto the last `recent` positions."""
    n = min(n, hi)
    w = np.full(hi, (1.0 - recent_frac) / hi)
    lo = max(0, hi - recent)
    w[lo:] += recent_frac / (hi - lo)
    w /= w.sum()
    return rng.choice(hi, size=n, replace=False, p=w).astype(np.int64)


def make_workload(*, name: str, seed: int, heads: int, req_seq_lens, tokens_per_req: int = 1,
                  topk_width: int, topk_mode: str = "uniform", topk_counts=None, topk_hi_margin: int = 0,
                  window: int, sink: bool, latent_dist: str = "normal", page: int = 64,
                  softmax_scale: Optional[float] = None, pass_topk_lens: bool = False,
                  spare_pages: int = 0, pool_rows: int = 1 << 15) -> Workload:
    """General recipe.

    req_seq_lens: per-request sequence lengths; token i (0-based) of request r sits
      at position seq_r - tokens_per_req + i, so its causal visible length is that + 1.
    topk_mode: 'uniform' (distinct uniform over the visible history, minus
      topk_hi_margin trailing positions), or 'biased' (80 % uniform, 20 % on the last 4096).
    topk_counts: optional per-token number of valid entries (the rest is -1).
    """
    rng = np.random.default_rng(seed)
    req_seq_lens = np.asarray(req_seq_lens, dtype=np.int64)
    R = int(req_seq_lens.size)
    T = R * tokens_per_req
    H = int(heads)
    K = int(topk_width)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(HEAD_DIM)

    # --- paging: each request owns ceil(seq/page) pages, scattered over the pool by a permutation
    pages_per_req = (req_seq_lens + page - 1) // page
    total_pages = int(pages_per_req.sum()) + int(spare_pages)
    max_blocks = int(max(1, pages_per_req.max(initial=1)))
    perm = rng.permutation(total_pages).astype(np.int32)
    block_table = np.full((R, max_blocks), -1, dtype=np.int32)
    off = 0
    for r in range(R):
        n = int(pages_per_req[r])
        block_table[r, :n] = perm[off:off + n]
        off += n

    # --- cache contents: every row holds a real quantised (latent, rope) draw; rows come from a
    # pool of distinct quantised rows so that huge caches stay cheap to build
    total_rows = total_pages * page
    n_pool = int(min(total_rows, pool_rows))
    if latent_dist == "normal":
        latent = rng.standard_normal((n_pool, LATENT_DIM))
    elif latent_dist == "t3":
        latent = rng.standard_t(3.0, size=(n_pool, LATENT_DIM))
    else:
        raise ValueError(latent_dist)
    rope = rng.standard_normal((n_pool, ROPE_DIM))
    pool = quantize_entries(latent, rope)
    if total_rows == n_pool:
        rows = pool[rng.permutation(n_pool)]
    else:
        rows = pool[rng.integers(0, n_pool, size=total_rows)]
    kv_cache = rows.reshape(total_pages, page, ENTRY_BYTES)

    # --- tokens
    req_idx = np.repeat(np.arange(R, dtype=np.int32), tokens_per_req)
    pos = np.concatenate([np.arange(s - tokens_per_req, s) for s in req_seq_lens]).astype(np.int64)
    seq_lens = (pos + 1).astype(np.int32)

    topk_idx = np.full((T, K), -1, dtype=np.int32)
    counts = np.zeros(T, dtype=np.int32)
    for t in range(T):
        hi = int(pos[t] + 1 - topk_hi_margin)
        want = K if topk_counts is None else int(topk_counts[t])
        if topk_mode == "uniform":
            sel = _distinct_uniform(rng, max(hi, 0), want)
        elif topk_mode == "biased":
            sel = _distinct_biased(rng, max(hi, 1), want, recent=4096, recent_frac=0.2)
        else:
            raise ValueError(topk_mode)
        topk_idx[t, :sel.size] = sel
        counts[t] = sel.size

    q = bf16_bits(rng.standard_normal((T, H, HEAD_DIM)))
    sink_arr = rng.standard_normal(H).astype(np.float32) if sink else None
    return Workload(name=name, q=q, kv_cache=kv_cache, block_table=block_table,
                    req_idx=None if tokens_per_req == 1 else req_idx,
                    topk_idx=topk_idx, topk_lens=counts if pass_topk_lens else None,
                    seq_lens=seq_lens, window=int(window), sink=sink_arr,
                    softmax_scale=float(softmax_scale), page=int(page))


WORKLOAD_NAMES = {
    1: "tiny-correctness T=2 h=16 seq=256 topk=64 W=32",
    2: "mid-decode T=32 h=64 seq=8192 topk=512 W=128",
    3: "compute-heavy T=128 h=128 seq=32768 topk=2048 W=128 sink",
    4: "spec-verify 64x2 tokens h=128 seq~U[4096,65536] topk_lens~U[256,2048] W=128 sink",
    5: "long-ragged T=16 h=64 seq~U[1024,131072] topk=2048 W=256 t3-latent sink",
}


def config(n: int) -> Workload:
    """The five decode workloads at full size (seed 1000 + n)."""
    seed = 1000 + n
    name = WORKLOAD_NAMES[n]
    if n == 1:
        return make_workload(name=name, seed=seed, heads=16, req_seq_lens=[256, 256], topk_width=64,
                             topk_hi_margin=32, window=32, sink=False)
    if n == 2:
        return make_workload(name=name, seed=seed, heads=64, req_seq_lens=[8192] * 32, topk_width=512,
                             window=128, sink=False)
    if n == 3:
        return make_workload(name=name, seed=seed, heads=128, req_seq_lens=[32768] * 128, topk_width=2048,
                             topk_mode="biased", window=128, sink=True)
    if n == 4:
        rng = np.random.default_rng(seed + 50_000)
        seqs = rng.integers(4096, 65536, size=64, endpoint=True)
        counts = rng.integers(256, 2048, size=128, endpoint=True)
        return make_workload(name=name, seed=seed, heads=128, req_seq_lens=seqs, tokens_per_req=2,
                             topk_width=2048, topk_counts=counts, window=128, sink=True, pass_topk_lens=True)
    if n == 5:
        rng = np.random.default_rng(seed + 50_000)
        seqs = rng.integers(1024, 131072, size=16, endpoint=True)
        return make_workload(name=name, seed=seed, heads=64, req_seq_lens=seqs, topk_width=2048,
                             window=256, sink=True, latent_dist="t3")
    raise ValueError(n)


def small_config(n: int) -> Workload:
    """Scaled-down versions of the five workloads with the same structure.

    Each spans several 128-key tiles with ragged tails, and all finish in the
    oracle within seconds (seed 2000 + n).
    """
    seed = 2000 + n
    if n == 1:
        return config(1)
    if n == 2:
        return make_workload(name="small-mid", seed=seed, heads=64, req_seq_lens=[1000, 700, 1500, 333, 1200],
                             topk_width=200, window=48, sink=False)
    if n == 3:
        return make_workload(name="small-heavy", seed=seed, heads=128, req_seq_lens=[3000, 5000, 4097],
                             topk_width=300, topk_mode="biased", window=64, sink=True)
    if n == 4:
        rng = np.random.default_rng(seed + 50_000)
        seqs = rng.integers(500, 2000, size=3, endpoint=True)
        counts = rng.integers(40, 300, size=6, endpoint=True)
        return make_workload(name="small-verify", seed=seed, heads=128, req_seq_lens=seqs, tokens_per_req=2,
                             topk_width=300, topk_counts=counts, window=64, sink=True, pass_topk_lens=True)
    if n == 5:
        rng = np.random.default_rng(seed + 50_000)
        seqs = rng.integers(200, 3000, size=4, endpoint=True)
        return make_workload(name="small-long", seed=seed, heads=64, req_seq_lens=seqs, topk_width=400,
                             window=96, sink=True, latent_dist="t3")
    raise ValueError(n)


def with_shared_picks(w: Workload, seed: int, keep: float) -> Workload:
    """Two-token requests whose draft token's top-k row repeats most of its partner's: a fraction
    `keep` of token 2r + 1's entries copied from token 2r's row (an indexer scores neighbouring
    positions alike, so a request's two tokens pick mostly the same keys)."""
    rng = np.random.default_rng(seed)
    topk = w.topk_idx.copy()
    for r in range(w.num_tokens // 2):
        m = rng.random(topk.shape[1]) < keep
        topk[2 * r + 1, m] = topk[2 * r, m]
    return dataclasses.replace(w, name=f"{w.name}, draft picks {int(round(100 * keep))}% shared", topk_idx=topk)


def to_device(w: Workload, device="cuda") -> dict:
    """Copy a workload's arrays into torch tensors on `device` (BF16 q, uint8 cache, int32 indices)."""
    import torch

    def t(a, dtype):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)

    q = torch.from_numpy(np.ascontiguousarray(w.q).view(np.int16)).view(torch.bfloat16).to(device)
    return dict(q=q, kv_cache=t(w.kv_cache, torch.uint8), block_table=t(w.block_table, torch.int32),
                req_idx=t(w.req_idx, torch.int32), topk_idx=t(w.topk_idx, torch.int32),
                topk_lens=t(w.topk_lens, torch.int32), seq_lens=t(w.seq_lens, torch.int32),
                window=int(w.window), sink=t(w.sink, torch.float32), softmax_scale=float(w.softmax_scale))


# ----------------------------------------------------------------------------
# indexer scores (inputs of the top-k selection)
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class TopkWorkload:
    name: str
    scores: np.ndarray       # float32 [T, width]
    num_cand: np.ndarray     # int32 [T]
    top_k: int

    @property
    def num_tokens(self) -> int:
        return int(self.scores.shape[0])

    @property
    def width(self) -> int:
        return int(self.scores.shape[1])


def indexer_scores(rng, num_tokens: int, width: int) -> np.ndarray:
    """float32 [T, width] indexer-like scores: ReLU of N(0, 1) draws rounded to BF16, so about
    half the scores are exactly zero and equal scores are common among the rest."""
    x = np.maximum(rng.standard_normal((num_tokens, width), dtype=np.float32), np.float32(0))
    return (bf16_bits(x).astype(np.uint32) << 16).view(np.float32)


def topk_config(name: str) -> TopkWorkload:
    """Top-k selection workloads shaped like the decode workloads' top-k rows:
      "long-batch"   128 tokens, 32768 candidates each, top-k 2048 (the long-context decode);
      "long-decode"  16 tokens, 1024..131071 candidates (uniform), top-k 2048 (the very long
                     decode: few rows, each split over a cluster of CTAs)."""
    if name == "long-batch":
        rng = np.random.default_rng(2003)
        T, width = 128, 32768
        nc = np.full(T, width, dtype=np.int32)
    elif name == "long-decode":
        rng = np.random.default_rng(2005)
        T, width = 16, 131072
        nc = rng.integers(1024, width, size=T).astype(np.int32)
    else:
        raise ValueError(name)
    return TopkWorkload(name=name, scores=indexer_scores(rng, T, width), num_cand=nc, top_k=2048)
