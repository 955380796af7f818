"""Randomised parity of dsv4_sparse_mla_decode against the fp64 oracle.

Seeded draws over the decode's argument space, each a whole small batch checked on every token
and head within the decode tolerances (gpu_util): head counts 16/32/64/128, page sizes, top-k
widths from 1 to 2048 with repeats, -1 padding and entries past the history, windows from 0 to
past the history, sequence lengths from 0, multi-token requests sharing a block-table row,
per-token top-k lengths (negative and past the width included), sinks, softmax scales, and
batch sizes that give one or many splits per token and, with varying lengths over many units,
the longest-first launch order.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_mla_decode_combine_gb300 as pkg
from gpu_util import compare_decode, need_gpu
from test_gpu_decode import run_decode

pytestmark = pytest.mark.gpu


def draw(seed: int) -> synth.Workload:
    rng = np.random.default_rng(seed)
    heads = int(rng.choice([16, 32, 64, 128]))
    page = int(rng.choice([16, 64, 128]))
    tpr = int(rng.choice([1, 1, 2, 3]))
    many = rng.random() < 0.3   # enough (token, head group) units to span more than one wave
    reqs = int(rng.integers(100, 220) if many else rng.integers(1, 9))
    hist_max = int(rng.choice([64, 600, 5000]))
    seqs = rng.integers(tpr, hist_max + tpr, size=reqs)
    width = int(rng.choice([1, 7, 64, 300, 1000, 2048]))
    window = int(rng.choice([0, 1, 16, 128, 700]))
    counts = None
    pass_lens = rng.random() < 0.5
    if pass_lens:
        counts = rng.integers(0, width + 1, size=reqs * tpr)
    w = synth.make_workload(name=f"random seed {seed}", seed=seed, heads=heads, req_seq_lens=seqs,
                            tokens_per_req=tpr, topk_width=width, topk_counts=counts, window=window,
                            sink=bool(rng.random() < 0.5), page=page, pass_topk_lens=pass_lens,
                            softmax_scale=float(rng.choice([0.02, 1.0 / 24.0, 0.2])),
                            latent_dist=str(rng.choice(["normal", "t3"])), spare_pages=int(rng.integers(0, 4)))
    topk = w.topk_idx.copy()
    T = w.num_tokens
    # repeats, -1 padding and positions at or past the token's own history, in some rows
    for t in range(T):
        if rng.random() < 0.3 and width > 1:
            i = rng.integers(0, width, size=min(width, 8))
            topk[t, i] = topk[t, rng.integers(0, width, size=i.size)]
        if rng.random() < 0.2:
            topk[t, rng.integers(0, width)] = int(w.seq_lens[t]) + int(rng.integers(0, 50))
    lens = w.topk_lens
    if lens is not None and rng.random() < 0.5:
        lens = lens.copy()
        lens[rng.integers(0, T, size=max(1, T // 5))] = -3
        lens[rng.integers(0, T, size=max(1, T // 5))] = width + 9
    seq_lens = w.seq_lens.copy()
    if rng.random() < 0.3:   # some tokens with no history at all
        seq_lens[rng.integers(0, T, size=max(1, T // 6))] = 0
    return dataclasses.replace(w, topk_idx=topk, topk_lens=lens, seq_lens=seq_lens)


@pytest.mark.parametrize("seed", list(range(7000, 7024)))
def test_decode_random_draws(seed):
    need_gpu()
    w = draw(seed)
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK, (w.name, status)
    ref_out, ref_lse, bad = oracle.sparse_mla_decode(w)
    assert bad == 0
    compare_decode(out, lse, ref_out, ref_lse, what=w.name)


@pytest.mark.parametrize("seed", list(range(7100, 7112)))
def test_decode_random_layouts(seed):
    """The same kind of draws with the top-k and block-table rows inside wider buffers (junk in
    the padding, which must not be read), and without the LSE output: the output bit-identical
    to the contiguous call's."""
    need_gpu()
    w = draw(seed)
    rng = np.random.default_rng(seed + 1)
    d = synth.to_device(w, "cuda")
    T, H = w.num_tokens, w.num_heads
    ws = pkg.workspace_for(T, H, w.topk_width, w.window)
    ref = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    pkg.check(pkg.dsv4_sparse_mla_decode(out=ref, lse=ref_lse, workspace=ws, **d), "decode")
    K = w.topk_width
    tk = torch.full((T, K + int(rng.integers(1, 40))), 7, dtype=torch.int32, device="cuda")
    tk[:, :K] = d["topk_idx"]
    bt0 = d["block_table"]
    bt = torch.full((bt0.shape[0], bt0.shape[1] + int(rng.integers(1, 9))), -5, dtype=torch.int32, device="cuda")
    bt[:, :bt0.shape[1]] = bt0
    d2 = dict(d, topk_idx=tk[:, :K], block_table=bt[:, :bt0.shape[1]])
    assert d2["topk_idx"].stride(0) > K and d2["block_table"].stride(0) > bt0.shape[1]
    out = torch.full((T, H, 512), 3.0, dtype=torch.bfloat16, device="cuda")
    pkg.check(pkg.dsv4_sparse_mla_decode(out=out, lse=None, workspace=ws, **d2), "decode, strided rows, no lse")
    torch.cuda.synchronize()
    assert pkg.dsv4_get_device_status() == pkg.DSV4_OK
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), w.name
