"""Bit-exact FP8-E4M3 x UE8M0 dequant through the decode, every code at many scales.

A token whose only key is one cache entry, with q = 0, has s = 0 for that key, so
its softmax weight is exactly 1 and out[t][h] = BF16(v) for every head h, where v is
the entry's dequantised latent part.  The dequantised value e4m3 * 2^(e - 127) has at
most four significant bits, so BF16 holds it exactly and the output must equal the
oracle's fp64 value bit for bit ("feat: add DeepSeek-V4 XPU attention decode path",
_dequant_gather_slots_kernel: value = e4m3 * 2^(ue8m0 - 127)).  The one exception is the
sign of zero: the code 0x80 is -0, and 0 + (-0) * 1 accumulates to +0, so both zeros
compare equal.

Each 128-element scale block holds half of the 254 non-NaN codes under one scale
exponent; the exponents run from 20 to 240, so every dequantised value and every
partial result stays a normal fp32 number (scale exponents below 20 would take values
under 2^-116, where the fp32 accumulator itself is subnormal; they are left to the
tolerance tests).  It runs at 64 heads and at 16 heads (a 64-head group whose missing
heads have zero queries).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_mla_decode_combine_gb300 as pkg
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu

SCALE_EXPONENTS = [20, 60, 100, 110, 120, 126, 127, 128, 130, 134, 135, 136, 150, 200, 240]
CODES = [c for c in range(256) if (c & 0x7F) != 0x7F]   # 254 codes, NaN excluded


def exact_workload(heads: int, seed: int) -> synth.Workload:
    rng = np.random.default_rng(seed)
    blocks = []   # (scale exponent, 128 codes)
    for se in SCALE_EXPONENTS:
        for half in range(2):
            codes = CODES[128 * half:128 * half + 128]
            codes = codes + CODES[:128 - len(codes)]
            blocks.append((se, rng.permutation(np.array(codes, dtype=np.uint8))))
    while len(blocks) % 4:
        blocks.append((127, rng.permutation(np.array(CODES[:128], dtype=np.uint8))))
    T = len(blocks) // 4
    page = 64
    kv = np.zeros((1, page, 656), dtype=np.uint8)
    for t in range(T):
        for j in range(4):
            se, codes = blocks[4 * t + j]
            kv[0, t, 128 * j:128 * j + 128] = codes
            kv[0, t, 640 + j] = se
    return synth.Workload(
        name=f"dequant-exact-h{heads}",
        q=np.zeros((T, heads, 576), dtype=np.uint16),
        kv_cache=kv,
        block_table=np.zeros((T, 1), dtype=np.int32),
        req_idx=None,
        topk_idx=np.arange(T, dtype=np.int32).reshape(T, 1),
        topk_lens=None,
        seq_lens=np.full((T,), page, dtype=np.int32),
        window=0,
        sink=None,
        softmax_scale=576 ** -0.5,
        page=page,
    )


def bf16_bits_exact(x: np.ndarray) -> np.ndarray:
    f = x.astype(np.float32)
    assert np.array_equal(f.astype(np.float64), x), "value not exact in fp32"
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in BF16"
    return (u >> 16).astype(np.uint16)


@pytest.mark.parametrize("heads", [16, 64])
@pytest.mark.parametrize("seed", [0, 1])
def test_dequant_bit_exact(heads, seed):
    need_gpu()
    w = exact_workload(heads, seed)
    d = synth.to_device(w, "cuda")
    T = w.num_tokens
    out = torch.full((T, heads, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, heads), 7.0, dtype=torch.float32, device="cuda")
    ws = pkg.workspace_for(T, heads, w.topk_width, w.window)
    pkg.check(pkg.dsv4_sparse_mla_decode(out=out, lse=lse, workspace=ws, **d), "decode")
    torch.cuda.synchronize()
    assert pkg.dsv4_get_device_status() == pkg.DSV4_OK
    got = out.view(torch.int16).cpu().numpy().view(np.uint16).copy()
    got[got == 0x8000] = 0
    for t in range(T):
        want = bf16_bits_exact(oracle.dequant_entry(w.kv_cache[0, t])[:512])
        want[want == 0x8000] = 0
        bad = np.nonzero(got[t] != want[None, :])
        assert bad[0].size == 0, (f"token {t}: {bad[0].size} mismatches, first head {bad[0][0]} dim {bad[1][0]}: "
                                  f"got {got[t][bad[0][0], bad[1][0]]:#06x} want {want[bad[1][0]]:#06x}")
    assert np.all(lse.cpu().numpy() == 0.0)
