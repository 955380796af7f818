"""GPU parity of dsv4_sparse_mla_decode against the fp64 oracle.

Tolerances (gpu_util): BF16 output max |err| <= 2e-2 and rel-L2 <= 1e-2; LSE |err| <= 1e-3.
Small versions of the five workloads run whole; the full-size workloads run in
the same launch configuration the benchmark times, checked on every token.  16 and 32
heads (a 64-head group with zero queries for the missing heads) run the edge cases,
the junk and widest top-k rows, and the long ragged workload at full size.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_mla_decode_combine_gb300 as pkg
from gpu_util import (compare_decode, edge_workload, full_config, junk_workload, long_window_workload, need_gpu,
                      small, widest_workload)

pytestmark = pytest.mark.gpu


def run_decode(w: synth.Workload, guard: bool = True):
    d = synth.to_device(w, "cuda")
    T, H = w.num_tokens, w.num_heads
    pad = 64
    out_full = torch.full((T * H * 512 + 2 * pad,), -7.0, dtype=torch.bfloat16, device="cuda")
    lse_full = torch.full((T * H + 2 * pad,), -7.0, dtype=torch.float32, device="cuda")
    out = out_full[pad:pad + T * H * 512].view(T, H, 512)
    lse = lse_full[pad:pad + T * H].view(T, H)
    ws = pkg.workspace_for(T, H, w.topk_width, w.window)
    ws.fill_(0xA5)   # stale workspace contents must not matter
    pkg.check(pkg.dsv4_sparse_mla_decode(out=out, lse=lse, workspace=ws, **d), "decode")
    torch.cuda.synchronize()
    status = pkg.dsv4_get_device_status()
    if guard:
        of = out_full.float().cpu().numpy()
        lf = lse_full.cpu().numpy()
        assert np.all(of[:pad] == -7.0) and np.all(of[-pad:] == -7.0), "write outside out"
        assert np.all(lf[:pad] == -7.0) and np.all(lf[-pad:] == -7.0), "write outside lse"
    return out, lse, status


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_decode_small_configs(n):
    need_gpu()
    w = small(n)
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    ref_out, ref_lse, bad = oracle.sparse_mla_decode(w)
    assert bad == 0
    compare_decode(out, lse, ref_out, ref_lse, what=w.name)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_decode_full_configs_all_tokens(n):
    """The five workloads at full size, in the launch configuration the benchmark times, every
    token and head against the oracle."""
    need_gpu()
    w = full_config(n)
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    ref_out, ref_lse, _ = oracle.sparse_mla_decode(w)
    compare_decode(out, lse, ref_out, ref_lse, what=w.name)


@pytest.mark.parametrize("heads", [16, 32])
def test_decode_low_heads_full_size(heads):
    """16 or 32 heads (one 64-head group whose missing heads have zero queries) over the long
    ragged workload's rows: 16 tokens, histories of 1024..131072, top-k 2048, window 256,
    Student-t latents, sinks; every token against the oracle, and nothing written past the
    heads that exist."""
    need_gpu()
    w5 = full_config(5)
    w = synth.make_workload(name=f"long-ragged h={heads}", seed=1105, heads=heads, req_seq_lens=list(w5.seq_lens),
                            topk_width=2048, window=256, sink=True, latent_dist="t3")
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    ref_out, ref_lse, _ = oracle.sparse_mla_decode(w)
    compare_decode(out, lse, ref_out, ref_lse, what=w.name)


@pytest.mark.parametrize("heads", [16, 32, 64, 128])
@pytest.mark.parametrize("sink", [False, True])
def test_decode_edge_lengths(heads, sink):
    """Tokens with an empty history, a single key, keys only in the window, ragged tiles."""
    need_gpu()
    w = edge_workload(heads, sink)
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    ref_out, ref_lse, _ = oracle.sparse_mla_decode(w)
    compare_decode(out, lse, ref_out, ref_lse, what=f"edge h={heads} sink={sink}")


@pytest.mark.parametrize("heads", [32, 64, 128])
def test_decode_junk_topk_entries(heads):
    """Repeats (also across the 2176-entry passes of the fused combine), -1 padding, positions
    past the token, positions inside the window and a topk_lens cut, in 3000-wide top-k rows."""
    need_gpu()
    w = junk_workload(heads)
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    ref_out, ref_lse, _ = oracle.sparse_mla_decode(w)
    compare_decode(out, lse, ref_out, ref_lse, what=f"junk top-k h={heads}")


@pytest.mark.parametrize("heads", [32, 64, 128])
def test_decode_max_topk_width(heads):
    """The widest top-k rows the library takes (8192 entries, the fused combine's hash set at its
    2^14-slot cap and half full) with a 1024-entry window."""
    need_gpu()
    w = widest_workload(heads)
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    ref_out, ref_lse, _ = oracle.sparse_mla_decode(w)
    compare_decode(out, lse, ref_out, ref_lse, what=f"widest top-k h={heads}")


def test_decode_window_only_and_topk_only():
    need_gpu()
    w = small(5)
    w0 = synth.Workload(**{**w.__dict__, "topk_lens": np.zeros(w.num_tokens, dtype=np.int32)})
    out, lse, _ = run_decode(w0)
    r = oracle.sparse_mla_decode(w0)
    compare_decode(out, lse, r[0], r[1], what="window only")
    w1 = synth.Workload(**{**w.__dict__, "window": 0})
    out, lse, _ = run_decode(w1)
    r = oracle.sparse_mla_decode(w1)
    compare_decode(out, lse, r[0], r[1], what="top-k only")


def test_decode_long_window():
    """A 20000-key window (the window is a position range, never hashed)."""
    need_gpu()
    w = long_window_workload()
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    ref_out, ref_lse, _ = oracle.sparse_mla_decode(w)
    compare_decode(out, lse, ref_out, ref_lse, what=w.name)


def test_decode_many_tokens_no_split():
    """Enough tokens that every token runs in one worker (no merge)."""
    need_gpu()
    rng = np.random.default_rng(5)
    seqs = rng.integers(100, 600, size=400)
    w = synth.make_workload(name="many", seed=9, heads=32, req_seq_lens=seqs, topk_width=48, window=16, sink=True)
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    rows = np.arange(0, 400, 7)
    r = oracle.sparse_mla_decode(w, tokens=rows)
    compare_decode(out, lse, r[0], r[1], rows=rows, what="many tokens")


@pytest.mark.parametrize("heads,reqs,tpr", [(128, 80, 2), (16, 200, 1), (64, 120, 2)])
def test_decode_longest_first_launch_order(heads, reqs, tpr):
    """Per-token list lengths that vary (topk_lens given, some rows empty) over more CTAs than
    one wave: the call orders the units longest first before the decode.  Every token and head
    against the oracle (a unit skipped or run twice would leave or corrupt rows), and the
    result identical to the same call on a copy of the batch without topk_lens but with the
    rows cut at the same lengths (index order)."""
    need_gpu()
    rng = np.random.default_rng(77 + heads)
    seqs = rng.integers(150, 3000, size=reqs)
    counts = rng.integers(0, 300, size=reqs * tpr)
    counts[::17] = 0
    w = synth.make_workload(name=f"ordered h={heads}", seed=400 + heads, heads=heads, req_seq_lens=seqs,
                            tokens_per_req=tpr, topk_width=300, topk_counts=counts, window=32, sink=True,
                            pass_topk_lens=True)
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    ref_out, ref_lse, _ = oracle.sparse_mla_decode(w)
    compare_decode(out, lse, ref_out, ref_lse, what=w.name)
    # the same lists given without topk_lens (entries past each length are -1): index order
    w2 = dataclasses.replace(w, topk_lens=None)
    out2, lse2, status2 = run_decode(w2)
    assert status2 == pkg.DSV4_OK
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))


def test_decode_launch_order_many_units_and_odd_lengths():
    """The ordering kernel over more units than its 1024 threads, with top-k lengths below 0 and
    above the row width (clamped), empty histories and single keys; every token against the
    oracle, and the no-alloc entry point (whose static scratch holds the order too) bit-identical
    to the workspace call."""
    need_gpu()
    rng = np.random.default_rng(3131)
    T = 1300
    seqs = rng.integers(0, 400, size=T)
    seqs[::11] = 0
    seqs[5::13] = 1
    counts = rng.integers(0, 48, size=T)
    w = synth.make_workload(name="ordered many", seed=3132, heads=16, req_seq_lens=np.maximum(seqs, 1),
                            topk_width=48, topk_counts=counts, window=8, sink=True, pass_topk_lens=True)
    w.seq_lens[seqs == 0] = 0
    lens = counts.astype(np.int32).copy()
    lens[::7] = -5
    lens[3::7] = 60
    w = dataclasses.replace(w, topk_lens=lens)
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    ref_out, ref_lse, _ = oracle.sparse_mla_decode(w)
    compare_decode(out, lse, ref_out, ref_lse, what=w.name)
    d = synth.to_device(w, "cuda")
    out2 = torch.full_like(out, 3.0)
    lse2 = torch.full_like(lse, 3.0)
    pkg.check(pkg.dsv4_sparse_mla_decode_noalloc(out=out2, lse=lse2, **d), "no-alloc decode")
    torch.cuda.synchronize()
    assert pkg.dsv4_get_device_status() == pkg.DSV4_OK
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))


def test_decode_launch_order_with_split_clusters():
    """Varying lengths up to the widest top-k row over more units than multiprocessors, long
    enough that the planner splits every token over a cluster: the ordered units start as whole
    clusters.  Sampled tokens (the longest, the shortest and others) against the oracle, and the
    whole result bit-identical to the same lists in index order."""
    need_gpu()
    rng = np.random.default_rng(5150)
    T = 160
    seqs = rng.integers(9000, 20000, size=T)
    counts = rng.integers(0, 8193, size=T)
    counts[:4] = [0, 1, 8192, 5000]
    w = synth.make_workload(name="ordered clusters", seed=5151, heads=16, req_seq_lens=seqs, topk_width=8192,
                            topk_counts=counts, window=128, sink=True, pass_topk_lens=True)
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    rows = np.unique(np.concatenate([np.arange(4), [int(np.argmax(counts)), int(np.argmin(counts))],
                                     rng.choice(T, size=10, replace=False)]))
    r = oracle.sparse_mla_decode(w, tokens=rows)
    compare_decode(out, lse, r[0], r[1], rows=rows, what=w.name)
    w2 = dataclasses.replace(w, topk_lens=None)
    out2, lse2, status2 = run_decode(w2)
    assert status2 == pkg.DSV4_OK
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))


def test_decode_padded_q_rows_and_repeat_determinism():
    need_gpu()
    w = small(2)
    d = synth.to_device(w, "cuda")
    T, H = w.num_tokens, w.num_heads
    qpad = torch.zeros((T, H * 576 + 64), dtype=torch.bfloat16, device="cuda")
    qpad[:, :H * 576] = d["q"].reshape(T, H * 576)
    d["q"] = qpad[:, :H * 576].view(T, H, 576)
    assert d["q"].stride(0) == H * 576 + 64
    o1, l1 = pkg.sparse_mla_decode(**d)
    o2, l2 = pkg.sparse_mla_decode(**d)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    r = oracle.sparse_mla_decode(w)
    compare_decode(o1, l1, r[0], r[1], what="padded q")


def test_decode_bad_block_table_entry_sets_status():
    need_gpu()
    w = small(4)
    t = 0
    pos = int(w.seq_lens[t]) - 1
    bt = w.block_table.copy()
    row = int(w.req_idx[t])
    bt[row, pos // w.page] = w.num_blocks + 5      # out of range under token 0's window
    wb = synth.Workload(**{**w.__dict__, "block_table": bt})
    pkg.dsv4_get_device_status()                   # clear
    out, lse, status = run_decode(wb)
    assert status == pkg.DSV4_ERR_BAD_INDEX
    assert pkg.dsv4_get_device_status() == pkg.DSV4_OK   # cleared by the read
    r = oracle.sparse_mla_decode(wb)
    assert r[2] > 0
    compare_decode(out, lse, r[0], r[1], what="bad block table entry (keys skipped)")


def test_decode_rejects_bad_arguments():
    need_gpu()
    w = small(2)
    d = synth.to_device(w, "cuda")
    T, H = w.num_tokens, w.num_heads
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    need = pkg.dsv4_sparse_mla_decode_workspace_size(T, H, w.topk_width, w.window)
    small_ws = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    assert pkg.dsv4_sparse_mla_decode(out=out, lse=lse, workspace=small_ws, **d) == pkg.DSV4_ERR_INVALID_ARG
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    assert pkg.dsv4_sparse_mla_decode(out=out, lse=lse, workspace=ws[1:need + 1], **d) == pkg.DSV4_ERR_INVALID_ARG
    assert pkg.dsv4_sparse_mla_decode_workspace_size(T, 48, w.topk_width, w.window) == 0
    d_neg = {**d, "softmax_scale": -abs(w.softmax_scale)}
    assert pkg.dsv4_sparse_mla_decode(out=out, lse=lse, workspace=ws, **d_neg) == pkg.DSV4_ERR_INVALID_ARG


def test_decode_zero_softmax_scale_gives_uniform_weights():
    """scale 0: every key of a token weighs the same (the sink still counts), lse = ln(L [+ e^sink])."""
    need_gpu()
    w = small(5)
    w0 = synth.Workload(**{**w.__dict__, "softmax_scale": 0.0})
    out, lse, status = run_decode(w0)
    assert status == pkg.DSV4_OK
    r = oracle.sparse_mla_decode(w0)
    compare_decode(out, lse, r[0], r[1], what="softmax scale 0")
