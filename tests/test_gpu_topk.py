"""Top-k selection on the GPU against the oracle: bit-exact rows and lengths.

Covers the hand-worked examples, random tie-heavy rows (signed zeros, infinities, NaN,
counts below zero, past the row and between), rows that are not 16-byte aligned, the
single-CTA path (many rows), the cluster path (few long rows), rows longer than the
shared-memory key cache, all-equal rows (candidate lists overflow), and the two full-size
workloads of ``synth.topk_config``.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins
import synth
import sparse_mla_decode_combine_gb300 as pkg
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu


def run_gpu(scores: np.ndarray, num_cand, top_k: int, stride: int = 0):
    """Runs the selection on a [T, width] score matrix stored with row stride `stride` (>= width)."""
    T, width = scores.shape
    stride = max(stride, width)
    buf = torch.full((T, stride), float("nan"), dtype=torch.float32)
    buf[:, :width] = torch.from_numpy(scores)
    sc = buf.cuda()[:, :width]
    nc = torch.from_numpy(np.asarray(num_cand, dtype=np.int32)).cuda()
    # guard bands around the outputs (and a row stride wider than the row) catch stray writes
    idx_full = torch.full((T + 2, top_k + 16), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    idx = idx_full[1:T + 1, 8:8 + top_k]
    lens_full = torch.full((T + 16,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    lens = lens_full[8:8 + T]
    pkg.check(pkg.dsv4_topk_select(sc, nc, top_k, idx, lens), "topk_select")
    torch.cuda.synchronize()
    xf = idx_full.cpu().numpy()
    assert np.all(xf[0] == 0x5A5A5A5A) and np.all(xf[-1] == 0x5A5A5A5A)
    assert np.all(xf[:, :8] == 0x5A5A5A5A) and np.all(xf[:, 8 + top_k:] == 0x5A5A5A5A)
    lf = lens_full.cpu().numpy()
    assert np.all(lf[:8] == 0x5A5A5A5A) and np.all(lf[8 + T:] == 0x5A5A5A5A)
    return idx.cpu().numpy(), lens.cpu().numpy()


def assert_same(scores, num_cand, top_k, stride=0, what=""):
    want_idx, want_len = oracle.topk_select(scores, num_cand, top_k)
    got_idx, got_len = run_gpu(scores, num_cand, top_k, stride)
    assert np.array_equal(got_len, want_len), what
    bad = np.argwhere(got_idx != want_idx)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first row {bad[0][0]} col {bad[0][1]}: " \
                          f"got {got_idx[bad[0][0], bad[0][1]]} want {want_idx[bad[0][0], bad[0][1]]}"


def test_topk_golden():
    need_gpu()
    for ex in oracle_pins.load_golden_topk():
        sc = np.array([r[1] for r in ex["rows"]], dtype=np.float32)
        idx, ln = run_gpu(sc, [r[0] for r in ex["rows"]], ex["K"])
        for i, (_, _, want, wl) in enumerate(ex["rows"]):
            assert idx[i].tolist() == want, (ex["name"], i, idx[i].tolist(), want)
            assert int(ln[i]) == wl, (ex["name"], i)


@pytest.mark.parametrize("seed", range(6))
def test_topk_random_tie_heavy(seed):
    need_gpu()
    rng = np.random.default_rng(500 + seed)
    pool = np.array([0.0, -0.0, 1.0, -1.0, 2.5, np.inf, -np.inf, np.nan, 7.0, 1e-30, -3e38], dtype=np.float32)
    T = int(rng.integers(1, 40))
    width = int(rng.integers(1, 12000))
    K = int(rng.integers(1, 3000))
    sc = rng.choice(pool, size=(T, width)).astype(np.float32)
    mask = rng.random((T, width)) < 0.3
    sc[mask] = rng.standard_normal(int(mask.sum())).astype(np.float32)
    nc = rng.integers(-2, width + 5, size=T).astype(np.int32)
    nc[0] = width
    assert_same(sc, nc, K, what=f"seed {seed}")


@pytest.mark.parametrize("stride_pad", [0, 1, 3])
def test_topk_unaligned_rows(stride_pad):
    """Row starts that are not 16-byte aligned take the scalar-load path."""
    need_gpu()
    rng = np.random.default_rng(77 + stride_pad)
    T, width, K = 9, 5001, 700
    sc = synth.indexer_scores(rng, T, width)
    nc = rng.integers(0, width + 1, size=T).astype(np.int32)
    assert_same(sc, nc, K, stride=width + stride_pad, what=f"pad {stride_pad}")


@pytest.mark.parametrize("T,width,K", [(2, 40000, 2048), (4, 70000, 1000), (19, 33000, 4096), (1, 131072, 1)])
def test_topk_cluster_rows(T, width, K):
    """Few long rows: each row is split over a thread-block cluster of CTAs."""
    need_gpu()
    rng = np.random.default_rng(T * 1000 + K)
    sc = synth.indexer_scores(rng, T, width)
    nc = rng.integers(width // 2, width + 1, size=T).astype(np.int32)
    assert_same(sc, nc, K, what=f"T={T} width={width} K={K}")


def test_topk_uncached_rows():
    """Many long rows: one CTA a row whose 45000 candidates exceed the shared-memory key cache, so
    every pass reads the scores from global memory."""
    need_gpu()
    rng = np.random.default_rng(91)
    T, width, K = 96, 45000, 2048
    sc = synth.indexer_scores(rng, T, width)
    nc = rng.integers(40000, width + 1, size=T).astype(np.int32)
    nc[0] = width
    assert_same(sc, nc, K, what="uncached rows")


def test_topk_extreme_ties():
    """All-equal rows, rows of NaN, and a single larger value at the end."""
    need_gpu()
    T, width, K = 6, 50000, 2048
    sc = np.zeros((T, width), dtype=np.float32)
    sc[1] = np.nan
    sc[2] = -0.0
    sc[3, -1] = 1.0
    sc[4, ::2] = 3.0
    sc[5] = np.float32(-np.inf)
    sc[5, 12345] = np.nan
    assert_same(sc, [width] * T, K, what="ties")


def test_topk_no_candidates_and_empty():
    need_gpu()
    sc = np.zeros((3, 0), dtype=np.float32)
    idx, ln = run_gpu(sc, [0, 5, -1], 4)
    assert np.all(idx == -1) and np.all(ln == 0)
    # no tokens: nothing is enqueued
    nc = torch.zeros(0, dtype=torch.int32, device="cuda")
    out = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    assert pkg.dsv4_topk_select(torch.zeros((0, 8), device="cuda"), nc, 4, out) == pkg.DSV4_OK


@pytest.mark.parametrize("name", ["long-batch", "long-decode"])
def test_topk_full_size(name):
    """The benchmark's workloads at full size, every row compared."""
    need_gpu()
    w = synth.topk_config(name)
    assert_same(w.scores, w.num_cand, w.top_k, what=name)
