"""Helpers shared by the GPU parity tests."""
from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import synth

# Tolerances of the decode against the fp64 oracle (BF16 output, fp32 LSE).
# Per output element: |gpu - ref| <= max(MAX_ABS, BF16_ULP_REL * |ref|).  The 2e-2
# absolute bound holds wherever BF16 can meet it; above |ref| = 2.56 a correctly
# rounded BF16 value alone can be half an ulp (2^-8 |ref|) away, so the bound there
# is one BF16 ulp of the reference.  rel-L2 and the LSE bound apply unchanged.
MAX_ABS = 2e-2
BF16_ULP_REL = 2.0 ** -7
REL_L2 = 1e-2
LSE_ABS = 1e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@functools.lru_cache(maxsize=None)
def full_config(n: int) -> synth.Workload:
    return synth.config(n)


@functools.lru_cache(maxsize=None)
def small(n: int) -> synth.Workload:
    return synth.small_config(n)


def compare_decode(out: torch.Tensor, lse: torch.Tensor, ref_out: np.ndarray, ref_lse: np.ndarray, rows=None,
                   what: str = ""):
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o = o[rows]
        l = l[rows]
    assert o.shape == ref_out.shape and l.shape == ref_lse.shape
    assert np.all(np.isfinite(o)), what
    err = np.abs(o - ref_out)
    tol = np.maximum(MAX_ABS, BF16_ULP_REL * np.abs(ref_out))
    ref_norm = np.linalg.norm(ref_out)
    rel = np.linalg.norm(o - ref_out) / ref_norm if ref_norm > 0 else np.linalg.norm(o - ref_out)
    both_inf = np.isneginf(l) & np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l), np.isneginf(ref_lse)), what
    lerr = np.zeros_like(l)
    lerr[~both_inf] = np.abs(l[~both_inf] - ref_lse[~both_inf])
    worst = float((err / tol).max()) if err.size else 0.0
    msg = (f"{what}: max_abs={err.max():.3e} worst err/tol={worst:.3f} rel_l2={rel:.3e} "
           f"lse_abs={lerr.max():.3e}")
    assert np.all(err <= tol), msg
    assert rel <= REL_L2, msg
    assert lerr.max() <= LSE_ABS, msg
    return err.max(), rel, lerr.max()


# ---- workloads with junk in the top-k rows, shared by the decode and combined-list tests

def junk_workload(heads: int) -> synth.Workload:
    """Repeats (also across the fused combine's 2176-entry passes), -1 padding, positions past
    the token, positions inside the window and a topk_lens cut, in 3000-wide top-k rows."""
    rng = np.random.default_rng(41)
    w = synth.make_workload(name="junk", seed=43, heads=heads, req_seq_lens=[5000, 4200, 300, 129, 2600],
                            topk_width=3000, window=64, sink=True)
    topk = w.topk_idx.copy()
    T, K = topk.shape
    for t in range(T):
        pos = int(w.seq_lens[t]) - 1
        row = topk[t]
        m = rng.random(K)
        src = rng.integers(0, K, size=K)
        row[m < 0.2] = row[src[m < 0.2]]                                          # repeats anywhere in the row
        row[(m >= 0.2) & (m < 0.3)] = -1
        row[(m >= 0.3) & (m < 0.35)] = pos + 1 + rng.integers(0, 100, size=int(((m >= 0.3) & (m < 0.35)).sum()))
        row[(m >= 0.35) & (m < 0.4)] = np.maximum(0, pos - rng.integers(0, 64, size=int(((m >= 0.35) & (m < 0.4)).sum())))
        row[2500:2600] = row[100:200]                                             # repeats across passes
    lens = np.array([K, 2900, 1000, 0, 2300], dtype=np.int32)
    return synth.Workload(**{**w.__dict__, "topk_idx": topk, "topk_lens": lens})


def widest_workload(heads: int) -> synth.Workload:
    """The widest top-k rows the library takes (8192 entries) with a 1024-entry window: many
    repeats of a few thousand positions, -1 padding, positions past the token and inside the
    window."""
    rng = np.random.default_rng(47)
    K = 8192
    w = synth.make_workload(name="widest", seed=49, heads=heads, req_seq_lens=[40000, 12000, 9000],
                            topk_width=K, window=1024, sink=True)
    topk = w.topk_idx.copy()
    for t in range(w.num_tokens):
        pos = int(w.seq_lens[t]) - 1
        row = topk[t]
        m = rng.random(K)
        pool = rng.integers(0, pos + 1, size=3000)
        row[m < 0.5] = pool[rng.integers(0, 3000, size=int((m < 0.5).sum()))]   # repeats of 3000 positions
        row[(m >= 0.5) & (m < 0.6)] = -1
        row[(m >= 0.6) & (m < 0.65)] = pos + 1 + rng.integers(0, 50, size=int(((m >= 0.6) & (m < 0.65)).sum()))
        row[(m >= 0.65) & (m < 0.7)] = pos - rng.integers(0, 1024, size=int(((m >= 0.65) & (m < 0.7)).sum()))
    return synth.Workload(**{**w.__dict__, "topk_idx": topk, "topk_lens": None})


def long_window_workload() -> synth.Workload:
    """A 20000-key window: one token whose window dwarfs its top-k (split into many CTAs), one
    whose window covers its whole history (every top-k entry is dropped), one shorter than its
    top-k row."""
    return synth.make_workload(name="long window", seed=61, heads=64, req_seq_lens=[30000, 9000, 70], topk_width=512,
                               window=20000, sink=True)


def edge_workload(heads: int, sink: bool, window: int = 16, seqs=(1, 0, 2, 5, 300, 129, 64, 65), topk_width: int = 40,
                  seed: int = 77) -> synth.Workload:
    """Tokens with an empty history, a single key, keys only in the window, ragged tiles."""
    return synth.make_workload(name="edge", seed=seed, heads=heads, req_seq_lens=list(seqs), topk_width=topk_width,
                               window=window, sink=sink)
