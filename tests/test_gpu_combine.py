"""GPU parity of dsv4_combine_topk_swa_indices: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins
import sparse_mla_decode_combine_gb300 as pkg
from gpu_util import full_config, need_gpu, small

pytestmark = pytest.mark.gpu


def run_combine(topk, topk_lens, seq_lens, window, width):
    dev = "cuda"
    tk = torch.from_numpy(np.ascontiguousarray(topk, dtype=np.int32)).to(dev)
    tl = None if topk_lens is None else torch.from_numpy(np.ascontiguousarray(topk_lens, dtype=np.int32)).to(dev)
    sl = torch.from_numpy(np.ascontiguousarray(seq_lens, dtype=np.int32)).to(dev)
    T = tk.shape[0]
    # guard bands around the outputs catch writes past the row or the array
    comb_full = torch.full((T + 2, width + 16), 0x5A5A5A5A, dtype=torch.int32, device=dev)
    comb = comb_full[1:T + 1, 8:8 + width]
    lens_full = torch.full((T + 16,), 0x5A5A5A5A, dtype=torch.int32, device=dev)
    lens = lens_full[8:8 + T]
    pkg.check(pkg.dsv4_combine_topk_swa_indices(tk, tl, sl, window, comb, lens), "combine")
    torch.cuda.synchronize()
    cf = comb_full.cpu().numpy()
    assert np.all(cf[0] == 0x5A5A5A5A) and np.all(cf[-1] == 0x5A5A5A5A)
    assert np.all(cf[:, :8] == 0x5A5A5A5A) and np.all(cf[:, 8 + width:] == 0x5A5A5A5A)
    lf = lens_full.cpu().numpy()
    assert np.all(lf[:8] == 0x5A5A5A5A) and np.all(lf[8 + T:] == 0x5A5A5A5A)
    return comb.cpu().numpy(), lens.cpu().numpy()


def check_against_oracle(topk, topk_lens, seq_lens, window, width):
    got_c, got_l = run_combine(topk, topk_lens, seq_lens, window, width)
    ref_c, ref_l = oracle.combine(topk, topk_lens, seq_lens, window, width)
    assert np.array_equal(got_l, ref_l)
    assert np.array_equal(got_c, ref_c)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_combine_full_configs(n):
    need_gpu()
    w = full_config(n)
    width = (w.topk_width + w.window + 127) // 128 * 128
    check_against_oracle(w.topk_idx, w.topk_lens, w.seq_lens, w.window, width)


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_combine_small_configs(n):
    need_gpu()
    w = small(n)
    check_against_oracle(w.topk_idx, w.topk_lens, w.seq_lens, w.window, w.topk_width + w.window)


def test_combine_golden_examples():
    need_gpu()
    for c in oracle_pins.load_golden():
        tl = None if c["topk_len"] is None else np.array([c["topk_len"]], dtype=np.int32)
        # the C ABI asks for width >= topk_width + window; the examples' rows are the prefix
        width = max(c["width"], len(c["topk"]) + c["window"])
        got_c, got_l = run_combine(np.array([c["topk"]], dtype=np.int32), tl, np.array([c["seq"]], dtype=np.int32),
                                   c["window"], width)
        assert got_c[0, :c["width"]].tolist() == c["row"] and int(got_l[0]) == c["length"], c
        assert np.all(got_c[0, c["width"]:] == -1)


def test_combine_random_edge_cases():
    need_gpu()
    rng = np.random.default_rng(41)
    for _ in range(40):
        T = int(rng.integers(1, 300))
        K = int(rng.integers(0, 40))
        W = int(rng.integers(0, 20))
        tk = rng.integers(-5, 60, size=(T, K)).astype(np.int32)
        if K and rng.random() < 0.5:          # many repeats
            tk = rng.choice(tk.ravel(), size=(T, K)).astype(np.int32)
        seq = rng.integers(-2, 70, size=T).astype(np.int32)
        tl = rng.integers(-3, K + 3, size=T).astype(np.int32) if rng.random() < 0.5 else None
        check_against_oracle(tk, tl, seq, W, K + W + int(rng.integers(0, 5)))


def test_combine_max_width_with_repeats():
    need_gpu()
    rng = np.random.default_rng(43)
    T, K, W = 8, 8192, 300
    seq = rng.integers(1, 50000, size=T).astype(np.int32)
    tk = rng.integers(-1, 60000, size=(T, K)).astype(np.int32)
    tk[:, K // 2:] = tk[:, :K // 2]            # every entry repeated once
    check_against_oracle(tk, None, seq, W, K + W)


def test_combine_strided_rows():
    need_gpu()
    w = small(4)
    T, K = w.topk_idx.shape
    wide = np.full((T, K + 13), 7, dtype=np.int32)
    wide[:, :K] = w.topk_idx
    dev = "cuda"
    tk = torch.from_numpy(wide).to(dev)[:, :K]
    sl = torch.from_numpy(w.seq_lens).to(dev)
    tl = torch.from_numpy(w.topk_lens).to(dev)
    comb, lens = pkg.combine_topk_swa_indices(tk, tl, sl, w.window)
    ref_c, ref_l = oracle.combine(w.topk_idx, w.topk_lens, w.seq_lens, w.window, comb.shape[1])
    assert np.array_equal(comb.cpu().numpy(), ref_c) and np.array_equal(lens.cpu().numpy(), ref_l)
