"""dsv4_sparse_mla_decode_noalloc against dsv4_sparse_mla_decode (GPU).

The no-alloc entry point is for callers that cannot allocate device memory when they
decode (pipelines whose memory is fixed at set-up, plug-ins whose framework owns all
allocations); it uses the library's static 32 MiB scratch array instead of a caller
workspace.  Two calls in a row must each match the workspace entry point within the
decode tolerance of the other GPU tests, the second call finding the first call's
scratch left in the array.  This file is collected last so that a run stopping at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import synth
import sparse_mla_decode_combine_gb300 as pkg
from gpu_util import compare_decode, need_gpu

pytestmark = pytest.mark.gpu


def _outputs(w):
    T, H = w.num_tokens, w.num_heads
    return (torch.full((T, H, 512), 3.0, dtype=torch.bfloat16, device="cuda"),
            torch.full((T, H), 3.0, dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("n", [1, 2, 5])
def test_noalloc_matches_workspace_entry_point_twice(n):
    need_gpu()
    w = synth.small_config(n)
    d = synth.to_device(w, "cuda")
    ref_out, ref_lse = _outputs(w)
    ws = pkg.workspace_for(w.num_tokens, w.num_heads, w.topk_width, w.window)
    pkg.check(pkg.dsv4_sparse_mla_decode(out=ref_out, lse=ref_lse, workspace=ws, **d), "workspace decode")
    torch.cuda.synchronize()
    r_out = ref_out.double().cpu().numpy()
    r_lse = ref_lse.double().cpu().numpy()
    for _ in range(2):
        out, lse = _outputs(w)
        pkg.check(pkg.dsv4_sparse_mla_decode_noalloc(out=out, lse=lse, **d), "no-alloc decode")
        torch.cuda.synchronize()
        assert pkg.dsv4_get_device_status() == pkg.DSV4_OK
        compare_decode(out, lse, r_out, r_lse, what=f"no-alloc vs workspace ({w.name})")


def test_noalloc_larger_batch_then_smaller():
    """A larger batch leaves more scratch in the shared array than a smaller batch writes; the
    smaller one must not read the leftovers.  Each result is compared with the workspace entry
    point's on the same inputs."""
    need_gpu()
    for n in (5, 3, 1):
        w = synth.small_config(n)
        d = synth.to_device(w, "cuda")
        ref_out, ref_lse = _outputs(w)
        ws = pkg.workspace_for(w.num_tokens, w.num_heads, w.topk_width, w.window)
        pkg.check(pkg.dsv4_sparse_mla_decode(out=ref_out, lse=ref_lse, workspace=ws, **d), "workspace decode")
        out, lse = _outputs(w)
        pkg.check(pkg.dsv4_sparse_mla_decode_noalloc(out=out, lse=lse, **d), "no-alloc decode")
        torch.cuda.synchronize()
        assert pkg.dsv4_get_device_status() == pkg.DSV4_OK
        compare_decode(out, lse, ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                       what=f"no-alloc after a larger batch ({w.name})")


def test_noalloc_rejects_batches_beyond_the_scratch_array():
    need_gpu()
    T, H, K, W = 4096, 128, 2048, 128
    assert pkg.dsv4_sparse_mla_decode_workspace_size(T, H, K, W) > (32 << 20)
    lib = pkg.load_library()
    rc = lib.dsv4_sparse_mla_decode_noalloc(
        8, H * 576, 16, 1, 64, 16, 1, 1, T, None, 16, K, K, None, 16, T, H, W, None, 0.1, 16, None, None)
    assert rc == pkg.DSV4_ERR_UNSUPPORTED
