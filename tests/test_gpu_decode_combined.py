"""The decode kernel's own combined index lists, bit for bit against the oracle's combine.

dsv4_sparse_mla_decode fuses the top-k / window combine into the decode kernel's prologue
(a shared-memory hash set and ballot ranks, not the standalone combine kernel).
dsv4_sparse_mla_decode_trace runs that same kernel and records, from each CTA, the logical
positions of the keys it decoded at their ranks in the token's list, plus the list length.
Every split of every token writes its own rank range, so the record is the list the
kernel actually used; it must equal oracle.combine's list exactly (and nothing past the
length may be written), and the decode's output must be bit-identical to the plain call's.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_mla_decode_combine_gb300 as pkg
from gpu_util import (edge_workload, full_config, junk_workload, long_window_workload, need_gpu, small,
                      widest_workload)

pytestmark = pytest.mark.gpu

SENTINEL = -12345


def traced_lists(w: synth.Workload):
    d = synth.to_device(w, "cuda")
    T, H, K, W = w.num_tokens, w.num_heads, w.topk_width, w.window
    width = (K + W + 127) // 128 * 128
    comb = torch.full((T, width), SENTINEL, dtype=torch.int32, device="cuda")
    lens = torch.full((T,), SENTINEL, dtype=torch.int32, device="cuda")
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws = pkg.workspace_for(T, H, K, W)
    pkg.check(pkg.dsv4_sparse_mla_decode_trace(out=out, lse=lse, workspace=ws, combined=comb, combined_lens=lens, **d),
              "decode trace")
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    pkg.check(pkg.dsv4_sparse_mla_decode(out=out2, lse=lse2, workspace=ws, **d), "decode")
    torch.cuda.synchronize()
    assert pkg.dsv4_get_device_status() == pkg.DSV4_OK
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), "the traced decode differs from the plain one"
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    return comb.cpu().numpy(), lens.cpu().numpy(), width


def check_lists(w: synth.Workload):
    got, got_lens, width = traced_lists(w)
    ref, ref_lens = oracle.combine(w.topk_idx, w.topk_lens, w.seq_lens, w.window, width)
    assert np.array_equal(got_lens, ref_lens), (w.name, np.flatnonzero(got_lens != ref_lens)[:8])
    for t in range(w.num_tokens):
        L = int(ref_lens[t])
        assert np.array_equal(got[t, :L], ref[t, :L]), (w.name, t, np.flatnonzero(got[t, :L] != ref[t, :L])[:8])
        assert np.all(got[t, L:] == SENTINEL), (w.name, t, "written past the list")


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_decode_kernel_combined_lists_full_configs(n):
    """The five workloads at full size, in the launch configuration (splits, clusters) the
    benchmark times: every token's list."""
    need_gpu()
    check_lists(full_config(n))


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_decode_kernel_combined_lists_small_configs(n):
    need_gpu()
    check_lists(small(n))


@pytest.mark.parametrize("heads", [32, 64, 128])
def test_decode_kernel_combined_lists_junk_rows(heads):
    """Repeats (first occurrence kept, also across the combine's passes), -1 padding, positions
    past the token and inside the window, a topk_lens cut."""
    need_gpu()
    check_lists(junk_workload(heads))


@pytest.mark.parametrize("heads", [64, 128])
def test_decode_kernel_combined_lists_widest_rows(heads):
    """8192-entry rows with thousands of repeats and a 1024-entry window."""
    need_gpu()
    check_lists(widest_workload(heads))


def test_decode_kernel_combined_lists_long_window():
    """A 20000-key window split over many CTAs of a cluster."""
    need_gpu()
    check_lists(long_window_workload())


@pytest.mark.parametrize("heads", [16, 128])
def test_decode_kernel_combined_lists_edges(heads):
    """Empty histories, single keys, window-only tokens."""
    need_gpu()
    check_lists(edge_workload(heads, True))


def test_decode_trace_rejects_a_narrow_record():
    need_gpu()
    w = small(2)
    d = synth.to_device(w, "cuda")
    T, H, K, W = w.num_tokens, w.num_heads, w.topk_width, w.window
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    ws = pkg.workspace_for(T, H, K, W)
    comb = torch.empty((T, K + W - 1), dtype=torch.int32, device="cuda")
    lens = torch.empty((T,), dtype=torch.int32, device="cuda")
    rc = pkg.dsv4_sparse_mla_decode_trace(out=out, lse=None, workspace=ws, combined=comb, combined_lens=lens, **d)
    assert rc == pkg.DSV4_ERR_INVALID_ARG
