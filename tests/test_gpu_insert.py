"""Fused Q RMSNorm + GPT-J RoPE + FP8/UE8M0 KV insert on the GPU against the oracle.

The entries' latent codes, scale bytes and padding must match bit for bit (the quantisation
is exact integer work on exact inputs).  The query's latent values must be within one BF16
step of the oracle's correctly rounded result (the kernel computes in fp32, so a value within
a few fp32 steps of a rounding boundary may round the other way).  A rotated value
(x c - y s, x s + y c) is a difference of fp32 products, whose rounding error is bounded by a
few fp32 steps of the pair's norm, not of the (possibly much smaller) result; so the query's
and the entries' rope values must be within one BF16 step of the value plus 2^-20 times the
pair's norm, which the rotation keeps.  Slots and cache bytes the call must not touch are
compared byte for byte.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_mla_decode_combine_gb300 as pkg
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu


def rope_table(rng, max_pos):
    ang = rng.uniform(0, 2 * np.pi, (max_pos, 32))
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def bf16_close(got_bits, want_bits):
    """Element-wise: equal bits, or adjacent BF16 values of the same sign (signed zeros equal)."""
    g = got_bits.astype(np.int32)
    w = want_bits.astype(np.int32)
    gz = (g & 0x7FFF) == 0
    wz = (w & 0x7FFF) == 0
    same_sign = (g & 0x8000) == (w & 0x8000)
    return (g == w) | (gz & wz) | (same_sign & (np.abs(g - w) <= 1))


def to_f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def rope_close(got_bits, want_bits):
    """Rotated pairs along the last axis (even, odd): one BF16 step of the value plus 2^-20 of the
    pair's norm."""
    g, w = to_f64(got_bits), to_f64(want_bits)
    norm = np.sqrt(w[..., 0::2] ** 2 + w[..., 1::2] ** 2)
    norm = np.repeat(norm, 2, axis=-1)
    return np.abs(g - w) <= np.abs(w) * 2.0 ** -7 + norm * 2.0 ** -20


def run_case(rng, T, H, max_pos=512, num_slots=300, weight=True, in_place=False, bad=True, eps=1e-6):
    q = synth.bf16_bits(rng.standard_normal((T, H, 576)) * rng.uniform(0.01, 30, (T, H, 1)))
    kv = synth.bf16_bits(np.concatenate([rng.standard_normal((T, 512)) * np.ldexp(1.0, rng.integers(-20, 20, (T, 1))),
                                         rng.standard_normal((T, 64))], axis=1))
    pos = rng.integers(0, max_pos, T).astype(np.int64)
    slots = rng.permutation(num_slots)[:T].astype(np.int64) if T <= num_slots else \
        rng.integers(0, num_slots, T).astype(np.int64)
    if bad and T >= 4:
        slots[0] = -1              # padding token: nothing written, nothing flagged
        slots[1] = num_slots + 3   # past the cache: flagged
        pos[2] = max_pos           # outside the table: flagged, query not rotated
    w = rng.uniform(0.5, 1.5, 576).astype(np.float32) if weight else None
    table = rope_table(rng, max_pos)
    cache0 = rng.integers(0, 256, (num_slots, 656)).astype(np.uint8)

    want_q, qbad = oracle.qnorm_rope(q, pos, table, w, eps)
    want_cache, cbad = oracle.kv_insert(kv, slots, pos, table, cache0)

    dev = "cuda"
    q_d = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(dev)
    q_out = q_d if in_place else torch.empty_like(q_d)
    kv_d = torch.from_numpy(kv.view(np.int16)).view(torch.bfloat16).to(dev)
    cache_d = torch.from_numpy(cache0.copy()).to(dev)
    pkg.dsv4_get_device_status()
    rc = pkg.dsv4_qnorm_rope_kv_insert(q_d, q_out, kv_d, torch.from_numpy(pos).to(dev),
                                       torch.from_numpy(slots).to(dev), torch.from_numpy(table).to(dev), cache_d,
                                       torch.from_numpy(w).to(dev) if w is not None else None, eps)
    pkg.check(rc, "qnorm_rope_kv_insert")
    torch.cuda.synchronize()
    status = pkg.dsv4_get_device_status()
    got_q = q_out.view(torch.int16).cpu().numpy().view(np.uint16)
    got_cache = cache_d.cpu().numpy()

    ok = bf16_close(got_q[..., :512], want_q[..., :512])
    assert ok.all(), f"q latent: {(~ok).sum()} values off by more than one BF16 step, first {np.argwhere(~ok)[0]}"
    ok = rope_close(got_q[..., 512:], want_q[..., 512:])
    assert ok.all(), f"q rope: {(~ok).sum()} values off, first {np.argwhere(~ok)[0]}"
    written = np.zeros(num_slots, dtype=bool)
    ok_tok = (slots >= 0) & (slots < num_slots) & (pos >= 0) & (pos < max_pos)
    written[slots[ok_tok]] = True
    assert np.array_equal(got_cache[~written], cache0[~written]), "bytes of slots the call must not write changed"
    gw, ww = got_cache[written], want_cache[written]
    lat_ok = np.array_equal(gw[:, :512], ww[:, :512])
    scale_ok = np.array_equal(gw[:, 640:], ww[:, 640:])
    assert lat_ok and scale_ok, (np.argwhere(gw[:, :512] != ww[:, :512])[:3], np.argwhere(gw[:, 640:] != ww[:, 640:])[:3])
    rope_ok = rope_close(gw[:, 512:640].copy().view("<u2"), ww[:, 512:640].copy().view("<u2"))
    assert rope_ok.all(), np.argwhere(~rope_ok)[:3]
    assert (status == pkg.DSV4_ERR_BAD_INDEX) == (qbad + cbad > 0), (status, qbad, cbad)


@pytest.mark.parametrize("H", [1, 3, 16, 64, 128])
def test_insert_heads(H):
    need_gpu()
    run_case(np.random.default_rng(700 + H), T=37, H=H)


def test_insert_in_place_no_weight():
    need_gpu()
    run_case(np.random.default_rng(801), T=20, H=64, weight=False, in_place=True)


def test_insert_no_bad_tokens_and_small_values():
    """No bad index (status stays OK); eps matters for heads of tiny values."""
    need_gpu()
    run_case(np.random.default_rng(802), T=9, H=32, bad=False, eps=1e-2)


def test_insert_full_size():
    """128 tokens x 128 heads, positions up to 32768, a cache of 65536 slots."""
    need_gpu()
    run_case(np.random.default_rng(803), T=128, H=128, max_pos=32768, num_slots=65536)


def test_insert_then_decode_reads_the_entry():
    """An entry written by the insert decodes, through the oracle's dequant, to the latent within
    half an E4M3 step of the BF16 input at its block's scale."""
    need_gpu()
    rng = np.random.default_rng(804)
    kv = synth.bf16_bits(rng.standard_normal((1, 576)))
    table = np.concatenate([np.ones((1, 32)), np.zeros((1, 32))], axis=1).astype(np.float32)
    cache = torch.zeros((4, 656), dtype=torch.uint8, device="cuda")
    q = torch.zeros((1, 1, 576), dtype=torch.bfloat16, device="cuda")
    pkg.check(pkg.dsv4_qnorm_rope_kv_insert(
        q, torch.empty_like(q), torch.from_numpy(kv.view(np.int16)).view(torch.bfloat16).cuda(),
        torch.zeros(1, dtype=torch.int64, device="cuda"), torch.full((1,), 2, dtype=torch.int64, device="cuda"),
        torch.from_numpy(table).cuda(), cache))
    entry = cache[2].cpu().numpy()
    k = oracle.dequant_entry(entry)
    x = (kv[0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for b in range(4):
        half_step = np.ldexp(1.0, int(entry[640 + b]) - 127) * 16   # the top binade's half step
        assert np.all(np.abs(k[128 * b:128 * b + 128] - x[128 * b:128 * b + 128]) <= half_step)
    assert np.array_equal(k[512:], x[512:])   # identity rotation: rope bytes as given
