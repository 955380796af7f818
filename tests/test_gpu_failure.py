"""Failure detection without a GPU fault: a bounded wait on an mbarrier that nothing arrives on
gives up, the host reads DSV4_ERR_TIMEOUT from the device status word (which the read clears),
and the context stays usable for the next decode."""
import pytest
import torch

import oracle
import sparse_mla_decode_combine_gb300 as pkg
from gpu_util import compare_decode, need_gpu, small
from test_gpu_decode import run_decode

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_stays_usable():
    need_gpu()
    pkg.dsv4_get_device_status()   # start from a clear word
    assert pkg.dsv4_selftest_wait_timeout(2_000_000) == pkg.DSV4_OK   # about a millisecond
    torch.cuda.synchronize()
    assert pkg.dsv4_get_device_status() == pkg.DSV4_ERR_TIMEOUT
    assert pkg.dsv4_get_device_status() == pkg.DSV4_OK
    w = small(2)
    out, lse, status = run_decode(w)
    assert status == pkg.DSV4_OK
    ref_out, ref_lse, _ = oracle.sparse_mla_decode(w)
    compare_decode(out, lse, ref_out, ref_lse, what="decode after a timed-out wait")
