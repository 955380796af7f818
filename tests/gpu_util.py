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
