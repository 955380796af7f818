"""dsv4_sparse_mla_decode_mtp_union against the fp64 oracle.

The MTP union call runs the two query tokens of a request (tokens 2r and 2r + 1, sharing a
block-table row) in one tile over the union of their combined key lists, each key masked for the
token that does not list it ("[ROCm] [DSv4] [Perf] Support DeepSeek v4 MTP", 风险 1).  Its
result is the per-token decode of dsv4_sparse_mla_decode, so every token is compared with the
oracle's per-token decode within the decode tolerances (gpu_util), and with the plain decode
call on the same inputs.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_mla_decode_combine_gb300 as pkg
from gpu_util import compare_decode, need_gpu, small

pytestmark = pytest.mark.gpu


def run_union(w: synth.Workload):
    d = synth.to_device(w, "cuda")
    T, H = w.num_tokens, w.num_heads
    out = torch.full((T, H, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), 7.0, dtype=torch.float32, device="cuda")
    ws = pkg.workspace_for_mtp_union(T, H, w.topk_width, w.window)
    ws.fill_(0xA5)   # stale workspace contents must not matter
    rc = pkg.dsv4_sparse_mla_decode_mtp_union(out=out, lse=lse, workspace=ws, **d)
    torch.cuda.synchronize()
    return rc, out, lse, pkg.dsv4_get_device_status()


def shared_picks(w: synth.Workload, seed: int, keep: float) -> synth.Workload:
    return synth.with_shared_picks(w, seed, keep)


def mtp_workload(seed: int, heads: int, seqs, width: int, window: int, sink: bool, counts=None,
                 latent="normal") -> synth.Workload:
    return synth.make_workload(name=f"mtp h{heads} K{width} W{window} seed {seed}", seed=seed, heads=heads,
                               req_seq_lens=seqs, tokens_per_req=2, topk_width=width, topk_counts=counts,
                               window=window, sink=sink, pass_topk_lens=counts is not None, latent_dist=latent)


CASES = [
    ("small-verify", lambda: small(4)),
    ("h32", lambda: mtp_workload(3001, 32, [700, 1300, 90, 2200], 200, 64, True)),
    ("h64-shared", lambda: shared_picks(mtp_workload(3002, 64, [3000, 1800, 2500], 512, 128, False), 5, 0.8)),
    ("h128-ragged", lambda: mtp_workload(3003, 128, [4000, 600, 2600, 5100], 600, 96, True,
                                         counts=np.array([600, 31, 0, 600, 250, 599, 7, 300]))),
    ("h64-long-split", lambda: mtp_workload(3004, 64, [9000, 6000], 2048, 256, True, latent="t3")),
    ("h128-window-only", lambda: mtp_workload(3005, 128, [150, 3000], 1, 700, False)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_mtp_union_matches_oracle(name, make):
    need_gpu()
    w = make()
    rc, out, lse, status = run_union(w)
    assert rc == pkg.DSV4_OK, (name, rc)
    assert status == pkg.DSV4_OK, (name, status)
    ref_out, ref_lse, bad = oracle.sparse_mla_decode(w)
    assert bad == 0
    compare_decode(out, lse, ref_out, ref_lse, what=f"mtp union {name}")


def test_mtp_union_matches_the_plain_decode():
    """Same inputs through both calls: within the decode tolerance of each other (the union
    sums each token's keys in another order and another tile)."""
    need_gpu()
    w = shared_picks(mtp_workload(3006, 128, [2048, 4000, 777], 700, 128, True), 9, 0.9)
    rc, out_u, lse_u, status = run_union(w)
    assert rc == pkg.DSV4_OK and status == pkg.DSV4_OK
    d = synth.to_device(w, "cuda")
    T, H = w.num_tokens, w.num_heads
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    pkg.check(pkg.dsv4_sparse_mla_decode(out=out, lse=lse, workspace=pkg.workspace_for(T, H, w.topk_width, w.window),
                                         **d), "decode")
    torch.cuda.synchronize()
    compare_decode(out_u, lse_u, out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                   what="mtp union against the plain decode")


def test_mtp_union_full_spec_verify_workload():
    """The spec-verify workload at full size (64 requests x 2 tokens x 128 heads), every token."""
    need_gpu()
    w = synth.config(4)
    rc, out, lse, status = run_union(w)
    assert rc == pkg.DSV4_OK and status == pkg.DSV4_OK
    ref_out, ref_lse, bad = oracle.sparse_mla_decode(w)
    assert bad == 0
    compare_decode(out, lse, ref_out, ref_lse, what="mtp union, spec-verify workload")


def test_mtp_union_rejects_pairs_on_different_rows():
    """A request whose two tokens name different block-table rows is a data error: recorded in
    the status word; the other requests decode as usual."""
    need_gpu()
    w = small(4)
    req = w.req_idx.copy()
    req[3] = req[2] + 1 if req[2] + 1 < w.block_table.shape[0] else req[2] - 1   # request 1's second token
    w = dataclasses.replace(w, req_idx=req)
    rc, out, lse, status = run_union(w)
    assert rc == pkg.DSV4_OK
    assert status == pkg.DSV4_ERR_BAD_INDEX
    ref_out, ref_lse, bad = oracle.sparse_mla_decode(w)
    keep = [t for t in range(w.num_tokens) if t // 2 != 1]
    compare_decode(out[keep], lse[keep], ref_out[keep], ref_lse[keep], what="mtp union, the other requests")
