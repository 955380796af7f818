"""GPU parity of dsv4_combine_topk_swa_indices_compressed against the oracle (bit for bit).

The compressed-region combine ("[ROCm] [DSv4] [Perf] Support DeepSeek v4 MTP", rocm.py,
_combine_topk_swa_indices_kernel): hand-worked examples, random batches of multi-token requests
with invalid top-k entries, positions before the start of the history, empty requests, and a
full-size batch; rows no request covers come back as -1 with the bad-index status.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins
import sparse_mla_decode_combine_gb300 as pkg
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu


def run(topk, qsl, seqs, gls, M, N, top_k, C, W, width, num_tokens=None):
    dev = "cuda"
    T = topk.shape[0] if num_tokens is None else num_tokens
    tk = torch.from_numpy(np.ascontiguousarray(topk, dtype=np.int32)).to(dev)
    q = torch.from_numpy(np.asarray(qsl, dtype=np.int32)).to(dev)
    s = torch.from_numpy(np.asarray(seqs, dtype=np.int32)).to(dev)
    g = torch.from_numpy(np.asarray(gls, dtype=np.int32)).to(dev)
    # guard bands around the outputs (and a row stride wider than the row) catch stray writes
    out_full = torch.full((T + 2, width + 16), 0x5A5A5A5A, dtype=torch.int32, device=dev)
    out = out_full[1:T + 1, 8:8 + width]
    lens_full = torch.full((T + 16,), 0x5A5A5A5A, dtype=torch.int32, device=dev)
    lens = lens_full[8:8 + T]
    pkg.check(pkg.dsv4_combine_topk_swa_indices_compressed(tk, q, s, g, M, N, top_k, C, W, out, lens),
              "compressed combine")
    torch.cuda.synchronize()
    of = out_full.cpu().numpy()
    assert np.all(of[0] == 0x5A5A5A5A) and np.all(of[-1] == 0x5A5A5A5A)
    assert np.all(of[:, :8] == 0x5A5A5A5A) and np.all(of[:, 8 + width:] == 0x5A5A5A5A)
    lf = lens_full.cpu().numpy()
    assert np.all(lf[:8] == 0x5A5A5A5A) and np.all(lf[8 + T:] == 0x5A5A5A5A)
    return out.cpu().numpy(), lens.cpu().numpy()


@pytest.mark.parametrize("seed", range(6))
def test_compressed_random_batches(seed):
    need_gpu()
    rng = np.random.default_rng(100 + seed)
    C = [1, 2, 4, 128, 3, 7][seed]
    R = int(rng.integers(1, 40))
    N = int(rng.integers(1, 800))
    top_k = int(rng.integers(0, 300))
    W = int(rng.integers(0, 200))
    M = N + 4000
    qlens = rng.integers(0, 6, size=R)
    seqs = rng.integers(0, 3000, size=R).astype(np.int32)
    gls = np.minimum(seqs, rng.integers(0, 3000, size=R) + W).astype(np.int32)
    T = int(qlens.sum())
    K = top_k + int(rng.integers(0, 3))
    topk = rng.integers(-3, N + 3, size=(T, K)).astype(np.int32)
    qsl = np.concatenate([[11], 11 + np.cumsum(qlens)]).astype(np.int32)
    width = top_k + W + int(rng.integers(0, 40))
    want, wl = oracle.combine_compressed(topk, qsl, seqs, gls, M, N, top_k, C, W, width)
    got, gl = run(topk, qsl, seqs, gls, M, N, top_k, C, W, width)
    assert np.array_equal(got, want)
    assert np.array_equal(gl, wl)
    assert pkg.dsv4_get_device_status() == pkg.DSV4_OK


def test_compressed_full_size_batch():
    """64 requests x 4 tokens, top-k 2048 of a 4x-compressed region, window 128."""
    need_gpu()
    rng = np.random.default_rng(7)
    R, qlen, top_k, C, W = 64, 4, 2048, 4, 128
    seqs = rng.integers(8192, 65536, size=R).astype(np.int32)
    gls = np.full(R, W + qlen, dtype=np.int32)
    N = 65536 // C
    M = N + int(gls.max())
    T = R * qlen
    topk = rng.integers(-1, N, size=(T, top_k)).astype(np.int32)
    qsl = (np.arange(R + 1) * qlen).astype(np.int32)
    width = 2304
    want, wl = oracle.combine_compressed(topk, qsl, seqs, gls, M, N, top_k, C, W, width)
    got, gl = run(topk, qsl, seqs, gls, M, N, top_k, C, W, width)
    assert np.array_equal(got, want) and np.array_equal(gl, wl)


def test_compressed_uncovered_rows_flagged():
    need_gpu()
    pkg.dsv4_get_device_status()   # clear
    topk = np.zeros((5, 4), dtype=np.int32)
    qsl = np.array([0, 2, 3], dtype=np.int32)   # covers rows 0..2 of 5
    got, gl = run(topk, qsl, [10, 10], [10, 10], 64, 8, 4, 1, 2, 8)
    want, wl = oracle.combine_compressed(topk[:3], qsl, [10, 10], [10, 10], 64, 8, 4, 1, 2, 8)
    assert np.array_equal(got[:3], want) and np.array_equal(gl[:3], wl)
    assert np.all(got[3:] == -1) and np.all(gl[3:] == 0)
    assert pkg.dsv4_get_device_status() == pkg.DSV4_ERR_BAD_INDEX
