"""CPU-only checks of the CUDA library: it builds for sm_103a, loads, exports every
entry point that include/dsv4.h declares, and rejects bad arguments on the host
before touching the GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import sparse_mla_decode_combine_gb300 as pkg
from sparse_mla_decode_combine_gb300 import build as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "dsv4.h")).read()
    return sorted(set(re.findall(r"DSV4_API\s+[\w\s\*]+?\b(dsv4_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    b.build()
    return pkg.load_library()


def test_header_declares_the_abi():
    syms = declared_symbols()
    for name in pkg.EXPORTED:
        assert name in syms
    assert set(syms) == set(pkg.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pkg.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (dsv4_\w+)", out))
    for name in declared_symbols():
        assert name in exported, name
        assert hasattr(lib, name)


def test_library_is_built_for_sm103a(lib):
    out = subprocess.run(["cuobjdump", "--list-elf", pkg.library_path()], capture_output=True, text=True).stdout
    assert "sm_103a" in out


def test_host_side_argument_errors(lib):
    S = None
    # combine: negative token count, oversize top-k, too narrow output
    assert lib.dsv4_combine_topk_swa_indices(None, 0, 0, None, None, -1, 0, None, 0, 0, None, S) == pkg.DSV4_ERR_INVALID_ARG
    assert lib.dsv4_combine_topk_swa_indices(None, 9000, 9000, None, None, 1, 0, None, 0, 9000, None, S) == pkg.DSV4_ERR_UNSUPPORTED
    assert lib.dsv4_combine_topk_swa_indices(None, 4, 4, None, ctypes.c_void_p(16), 1, 8, None, 12, 11, None, S) == pkg.DSV4_ERR_INVALID_ARG
    assert lib.dsv4_combine_topk_swa_indices(None, 4, 4, None, None, 0, 8, None, 12, 12, None, S) == pkg.DSV4_OK
    # compressed combine: top_k above the row width, ratio 0, too narrow output, region overflow, nothing to do
    P = ctypes.c_void_p(16)
    cc = lib.dsv4_combine_topk_swa_indices_compressed
    #        topk, stride, width, qsl, seq, gather, R, T, M,  N,  top_k, C, W, combined, cstride, cwidth, lens, stream
    assert cc(P, 4, 4, P, P, P, 1, 1, 64, 8, 5, 1, 0, P, 8, 8, P, S) == pkg.DSV4_ERR_INVALID_ARG
    assert cc(P, 4, 4, P, P, P, 1, 1, 64, 8, 4, 0, 0, P, 8, 8, P, S) == pkg.DSV4_ERR_INVALID_ARG
    assert cc(P, 4, 4, P, P, P, 1, 1, 64, 8, 4, 1, 8, P, 11, 11, P, S) == pkg.DSV4_ERR_INVALID_ARG
    assert cc(P, 4, 4, P, P, P, 3, 1, 1 << 30, 8, 4, 1, 0, P, 8, 8, P, S) == pkg.DSV4_ERR_INVALID_ARG
    assert cc(P, 9000, 9000, P, P, P, 1, 1, 64, 8, 4, 1, 0, P, 8, 8, P, S) == pkg.DSV4_ERR_UNSUPPORTED
    assert cc(None, 4, 4, None, None, None, 0, 0, 64, 8, 4, 1, 4, None, 8, 8, None, S) == pkg.DSV4_OK
    # top-k selection: K < 1, negative token count, missing pointers, narrow output rows, nothing to do
    tk = lib.dsv4_topk_select
    #        scores, stride, width, num_cand, T, K, idx, istride, lens, stream
    assert tk(P, 16, 16, P, 1, 0, P, 4, None, S) == pkg.DSV4_ERR_INVALID_ARG
    assert tk(P, 16, 16, P, -1, 4, P, 4, None, S) == pkg.DSV4_ERR_INVALID_ARG
    assert tk(None, 16, 16, P, 1, 4, P, 4, None, S) == pkg.DSV4_ERR_INVALID_ARG
    assert tk(P, 16, 16, None, 1, 4, P, 4, None, S) == pkg.DSV4_ERR_INVALID_ARG
    assert tk(P, 16, 16, P, 1, 4, P, 3, None, S) == pkg.DSV4_ERR_INVALID_ARG
    assert tk(P, 8, 16, P, 1, 4, P, 4, None, S) == pkg.DSV4_ERR_INVALID_ARG
    assert tk(None, 0, 0, None, 0, 4, None, 0, None, S) == pkg.DSV4_OK
    # wait self-test: a limit out of range
    assert lib.dsv4_selftest_wait_timeout(0, S) == pkg.DSV4_ERR_INVALID_ARG
    assert lib.dsv4_selftest_wait_timeout((1 << 31) + 1, S) == pkg.DSV4_ERR_INVALID_ARG
    # fused norm/RoPE/insert: heads 0 and 129, NaN eps, odd stride, nothing to do
    ins = lib.dsv4_qnorm_rope_kv_insert
    #         q, qs,   qo, qos,  T, H,  w,    eps,  kv, kvs, pos, slot, cs, maxp, cache, nslots, stream
    good = [P, 1152, P, 1152, 1, 2, None, 1e-6, P, 576, P, P, P, 8, P, 4, S]
    for i, v in ((5, 0), (5, 129), (7, float("nan")), (1, 1153), (9, 577), (13, 0)):
        bad = list(good)
        bad[i] = v
        assert ins(*bad) == pkg.DSV4_ERR_INVALID_ARG, (i, v)
    bad = list(good)
    bad[4] = 0
    assert ins(*bad) == pkg.DSV4_OK
    # decode: unsupported head count, non-finite or negative scale, missing pointers
    args = [None, 576 * 16, None, 1, 64, None, 1, 1, 1, None, None, 0, 0, None, ctypes.c_void_p(16), 1, 16, 8, None,
            1.0, None, None, None, 0, S]
    bad = list(args)
    bad[16] = 48
    assert lib.dsv4_sparse_mla_decode(*bad) == pkg.DSV4_ERR_UNSUPPORTED
    bad = list(args)
    bad[19] = float("nan")
    assert lib.dsv4_sparse_mla_decode(*bad) == pkg.DSV4_ERR_INVALID_ARG
    bad[19] = -0.5   # a negative scale: the running max would be taken on the wrong side
    assert lib.dsv4_sparse_mla_decode(*bad) == pkg.DSV4_ERR_INVALID_ARG
    assert lib.dsv4_sparse_mla_decode(*args) == pkg.DSV4_ERR_INVALID_ARG
    bad = list(args)
    bad[15] = 0
    assert lib.dsv4_sparse_mla_decode(*bad) == pkg.DSV4_OK   # nothing to do
    # MTP union decode: 16 heads, an odd token count, no req_idx; nothing to do
    un = lib.dsv4_sparse_mla_decode_mtp_union
    uargs = list(args)
    uargs[9] = ctypes.c_void_p(16)   # req_idx
    uargs[15] = 2                    # two tokens: one request
    uargs[16] = 32
    bad = list(uargs)
    bad[16] = 16
    assert un(*bad) == pkg.DSV4_ERR_UNSUPPORTED
    bad = list(uargs)
    bad[15] = 3
    assert un(*bad) == pkg.DSV4_ERR_INVALID_ARG
    bad = list(uargs)
    bad[9] = None
    assert un(*bad) == pkg.DSV4_ERR_INVALID_ARG
    bad = list(uargs)
    bad[15] = 0
    assert un(*bad) == pkg.DSV4_OK
    assert lib.dsv4_sparse_mla_decode_mtp_union_workspace_size(3, 64, 64, 8) == 0   # odd token count
