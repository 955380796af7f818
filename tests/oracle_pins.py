"""Checks that pin the fp64 oracle to facts outside itself.

Every check takes an ``oracle.Oracle`` instance so the same checks run against
the real oracle (tests/test_oracle.py) and against deliberately broken copies
of it (tests/test_oracle_mutants.py), which shows that a plausible mistake in
the oracle fails at least one of them.

What pins what:
  * the cache format: all 256 E4M3 codes against torch.float8_e4m3fn, all
    UE8M0 exponents against math.ldexp, BF16 against torch.bfloat16, and a
    hand-built entry for the byte layout;
  * the combine: hand-worked examples from the pages' rule
    (tests/golden/combine_worked_examples.txt), a brute-force restatement
    (first-occurrence dictionary + window set) on thousands of tiny random
    cases, and its invariants;
  * the attention: dense softmax attention computed with numpy/scipy over
    keys decoded by torch's own FP8/BF16 casts, when the top-k list covers
    the whole history; closed forms (one key, two keys + sink); the LSE
    identity; the sink -> -inf limit; invariance to top-k order, -1 padding,
    junk entries and page permutation;
  * the merge: any partition of a key set merges back to the unsplit result.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
from scipy.special import logsumexp

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "combine_worked_examples.txt")


# ----------------------------------------------------------------------------
# independent decoders (torch casts + math.ldexp), used only to build references
# ----------------------------------------------------------------------------
def torch_e4m3(codes: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    return torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_bf16(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(b).view(torch.bfloat16).to(torch.float64).numpy()


def torch_keys(entries: np.ndarray) -> np.ndarray:
    """[N, 656] cache entries -> [N, 576] fp64 keys via torch casts."""
    e = np.ascontiguousarray(entries, dtype=np.uint8).reshape(-1, 656)
    lat = torch_e4m3(e[:, :512]).reshape(-1, 4, 128)
    sc = np.ldexp(1.0, e[:, 640:644].astype(np.int64) - 127)
    lat = (lat * sc[:, :, None]).reshape(-1, 512)
    rope = torch_bf16(np.ascontiguousarray(e[:, 512:640]).view('<u2'))
    return np.concatenate([lat, rope], axis=1)


def gather_entries(w, t: int, positions) -> np.ndarray:
    row = t if w.req_idx is None else int(w.req_idx[t])
    pos = np.asarray(positions, dtype=np.int64)
    phys = w.block_table[row, pos // w.page]
    return w.kv_cache[phys, pos % w.page]


# ----------------------------------------------------------------------------
# cache format
# ----------------------------------------------------------------------------
def check_e4m3_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch_e4m3(codes)
    got = np.array([orc.e4m3_to_f64(c) for c in codes])
    nan = np.isnan(ref)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    # values fixed by the OCP E4M3 definition
    assert orc.e4m3_to_f64(0x7E) == 448.0
    assert orc.e4m3_to_f64(0x08) == 2.0 ** -6
    assert orc.e4m3_to_f64(0x01) == 2.0 ** -9
    assert orc.e4m3_to_f64(0x38) == 1.0
    assert orc.e4m3_to_f64(0xC0) == -2.0


def check_ue8m0(orc):
    for e in range(255):
        assert orc.ue8m0_to_f64(e) == math.ldexp(1.0, e - 127)
    assert math.isnan(orc.ue8m0_to_f64(255))


def check_bf16(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 16, size=4000).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite patterns
    ref = torch_bf16(bits)
    got = np.array([orc.bf16_to_f64(b) for b in bits])
    assert np.array_equal(got, ref)


def check_entry_layout(orc):
    e = np.zeros(656, dtype=np.uint8)
    e[0] = 0x38      # 1.0, block 0
    e[127] = 0xC0    # -2.0, block 0
    e[128] = 0x38    # 1.0, block 1
    e[300] = 0x3C    # 1.5, block 2
    e[511] = 0x01    # 2^-9, block 3
    e[640:644] = [127, 128, 126, 130]           # scales 1, 2, 0.5, 8
    e[512:514] = [0xC0, 0x3F]                   # rope[0] = bf16 0x3FC0 = 1.5
    e[638:640] = [0x40, 0xC0]                   # rope[63] = bf16 0xC040 = -3.0
    e[644:656] = 0xFF                           # padding is not data
    k = orc.dequant_entry(e)
    expect = np.zeros(576)
    expect[0], expect[127], expect[128], expect[300], expect[511] = 1.0, -2.0, 2.0, 0.75, 2.0 ** -9 * 8
    expect[512], expect[575] = 1.5, -3.0
    assert np.array_equal(k, expect)


def check_quantize_roundtrip(orc):
    """The generator's encoder and the oracle's decoder are mutual inverses on all codes."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = np.array([orc.e4m3_to_f64(c) for c in codes])
    assert np.array_equal(synth.e4m3_encode(vals), codes)
    # whole entries: dequant(quantize(x)) within half an E4M3 step, scale rule as stated
    rng = np.random.default_rng(11)
    lat = rng.standard_t(3.0, size=(64, 512)) * np.exp(rng.uniform(-20, 20, size=(64, 1)))
    rope = rng.standard_normal((64, 64))
    ents = synth.quantize_entries(lat, rope)
    for i in range(64):
        k = orc.dequant_entry(ents[i])
        for b in range(4):
            x = lat[i, 128 * b:128 * b + 128]
            e = int(ents[i, 640 + b]) - 127
            amax = np.abs(x).max()
            assert 448.0 * 2.0 ** e >= amax and 448.0 * 2.0 ** (e - 1) < amax
            err = np.abs(k[128 * b:128 * b + 128] - x)
            bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** (e - 10))
            assert np.all(err <= bound * (1 + 1e-12))


# ----------------------------------------------------------------------------
# combine
# ----------------------------------------------------------------------------
def load_golden():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            seq, win, tl, entries, width, row, ln = [s.strip() for s in line.split(";")]
            cases.append(dict(seq=int(seq), window=int(win), topk_len=None if tl == "none" else int(tl),
                              topk=[int(v) for v in entries.split()], width=int(width),
                              row=[int(v) for v in row.split()], length=int(ln)))
    return cases


def check_combine_golden(orc):
    for c in load_golden():
        tk = np.array([c["topk"]], dtype=np.int32)
        tl = None if c["topk_len"] is None else np.array([c["topk_len"]], dtype=np.int32)
        row, ln = orc.combine(tk, tl, np.array([c["seq"]], dtype=np.int32), c["window"], c["width"])
        assert row[0].tolist() == c["row"], c
        assert int(ln[0]) == c["length"], c


def brute_combine(topk_row, n, seq_len, window):
    """First-occurrence dictionary + window set restatement of the combine."""
    pos = seq_len - 1
    win = set(range(max(0, pos - window + 1), pos + 1)) if pos >= 0 else set()
    first = {}
    for i, v in enumerate(list(topk_row[:n])):
        first.setdefault(int(v), i)
    kept = [v for v, i in sorted(first.items(), key=lambda kv: kv[1]) if 0 <= v <= pos and v not in win]
    return kept + sorted(win)


def check_combine_bruteforce(orc, cases: int = 3000):
    rng = np.random.default_rng(3)
    for _ in range(cases // 100):
        T = 100
        K = int(rng.integers(0, 13))
        W = int(rng.integers(0, 11))
        tk = rng.integers(-3, 31, size=(T, K)).astype(np.int32)
        seq = rng.integers(-1, 26, size=T).astype(np.int32)
        tl = rng.integers(-1, K + 2, size=T).astype(np.int32) if rng.random() < 0.5 else None
        width = K + W + int(rng.integers(0, 4))
        rows, lens = orc.combine(tk, tl, seq, W, width)
        for t in range(T):
            n = K if tl is None else min(max(int(tl[t]), 0), K)
            want = brute_combine(tk[t], n, int(seq[t]), W)
            L = int(lens[t])
            assert L == len(want), (tk[t], n, seq[t], W)
            assert rows[t, :L].tolist() == want
            assert np.all(rows[t, L:] == -1)
            # invariants
            assert len(set(want)) == L
            pos = int(seq[t]) - 1
            assert all(0 <= v <= pos for v in want)
            assert L == len({int(v) for v in tk[t, :n] if 0 <= v < max(0, pos - W + 1)}) + max(0, min(pos + 1, W))


def check_combine_config1_lengths(orc):
    w = synth.config(1)
    _, lens = orc.combine(w.topk_idx, w.topk_lens, w.seq_lens, w.window, 128)
    assert np.all(lens == 96)


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------
def full_history_workload(seed=5, sink=True, heads=4, tokens_per_req=1):
    """Small workload whose top-k lists name every position before the window."""
    w = synth.make_workload(name="full-history", seed=seed, heads=heads, req_seq_lens=[41, 70, 100, 3],
                            tokens_per_req=tokens_per_req, topk_width=8, window=8, sink=sink)
    rng = np.random.default_rng(seed)
    T = w.num_tokens
    K = int(w.seq_lens.max())
    tk = np.full((T, K + 5), -1, dtype=np.int32)
    for t in range(T):
        pos = int(w.seq_lens[t]) - 1
        hist = rng.permutation(max(0, pos - w.window + 1))
        tk[t, :hist.size] = hist
    w.topk_idx = tk
    return w


def dense_reference(w, t: int, h: int):
    pos = int(w.seq_lens[t]) - 1
    keys = torch_keys(gather_entries(w, t, np.arange(pos + 1)))
    qh = torch_bf16(w.q[t, h])
    s = w.softmax_scale * (keys @ qh)
    allv = s if w.sink is None else np.concatenate([s, [float(w.sink[h])]])
    lse = logsumexp(allv) if allv.size else -np.inf
    out = np.exp(s - lse) @ keys[:, :512] if s.size else np.zeros(512)
    return out, lse


def check_dense_equivalence(orc):
    for sink, tpr in ((True, 1), (False, 1), (True, 2)):
        w = full_history_workload(sink=sink, tokens_per_req=tpr)
        out, lse, bad = orc.sparse_mla_decode(w, n_threads=2)
        assert bad == 0
        for t in range(w.num_tokens):
            for h in range(w.num_heads):
                o_ref, l_ref = dense_reference(w, t, h)
                assert abs(lse[t, h] - l_ref) <= 1e-12 * max(1.0, abs(l_ref)), (t, h, lse[t, h], l_ref)
                assert np.max(np.abs(out[t, h] - o_ref)) <= 1e-12


def check_order_padding_invariance(orc):
    w = synth.small_config(2)
    base_out, base_lse, _ = orc.sparse_mla_decode(w, tokens=[0, 1, 2], n_threads=2)
    rng = np.random.default_rng(9)
    tk = w.topk_idx
    junk = np.zeros((tk.shape[0], tk.shape[1] + 40), dtype=np.int32)
    for t in range(tk.shape[0]):
        pos = int(w.seq_lens[t]) - 1
        extra = np.concatenate([np.full(10, -1), rng.integers(pos + 1, pos + 1000, size=10),  # invalid / not causal
                                rng.integers(max(0, pos - w.window + 1), pos + 1, size=10),  # inside the window
                                rng.choice(tk[t][tk[t] >= 0], size=10)])  # repeats
        junk[t] = rng.permutation(np.concatenate([tk[t], extra]))
    w2 = synth.Workload(**{**w.__dict__, "topk_idx": junk})
    out, lse, _ = orc.sparse_mla_decode(w2, tokens=[0, 1, 2], n_threads=2)
    assert np.max(np.abs(out - base_out)) <= 1e-12
    assert np.max(np.abs(lse - base_lse)) <= 1e-12


def check_page_permutation(orc):
    w = synth.small_config(5)
    out0, lse0, _ = orc.sparse_mla_decode(w, n_threads=2)
    rng = np.random.default_rng(13)
    perm = rng.permutation(w.num_blocks).astype(np.int32)
    cache = np.empty_like(w.kv_cache)
    cache[perm] = w.kv_cache
    bt = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    w2 = synth.Workload(**{**w.__dict__, "kv_cache": cache, "block_table": bt})
    out1, lse1, _ = orc.sparse_mla_decode(w2, n_threads=2)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def check_closed_forms(orc):
    rng = np.random.default_rng(17)
    # one key, no sink: the output is that key's latent exactly and lse is its logit
    q = rng.standard_normal(576)
    k = rng.standard_normal(576)
    out, lse = orc.attend(q, k[None, :], 0.25)
    assert np.array_equal(out, k[:512])
    assert abs(lse - 0.25 * float(q @ k)) <= 1e-12 * max(1.0, abs(lse))
    # two keys along one axis plus a sink: out = (e^a v1 + e^b v2) / (e^a + e^b + e^c)
    q = np.zeros(576)
    q[3] = 1.0
    k1 = rng.standard_normal(576)
    k2 = rng.standard_normal(576)
    k1[3], k2[3] = 2.0, -1.0
    c = 0.7
    out, lse = orc.attend(q, np.stack([k1, k2]), 0.5, sink=c)
    a, b = 1.0, -0.5
    z = math.exp(a) + math.exp(b) + math.exp(c)
    assert abs(lse - math.log(z)) <= 1e-14
    assert np.max(np.abs(out - (math.exp(a) * k1[:512] + math.exp(b) * k2[:512]) / z)) <= 1e-14
    # no keys: out 0 and lse -inf, or lse = sink
    out, lse = orc.attend(q, np.zeros((0, 576)), 0.5)
    assert lse == -math.inf and not out.any()
    out, lse = orc.attend(q, np.zeros((0, 576)), 0.5, sink=1.25)
    assert lse == 1.25 and not out.any()
    # identical keys: out = v, lse = s + ln L
    out, lse = orc.attend(q, np.stack([k1] * 7), 0.5)
    assert np.max(np.abs(out - k1[:512])) <= 1e-14
    assert abs(lse - (1.0 + math.log(7))) <= 1e-14


def check_lse_identity_and_sink_limit(orc):
    rng = np.random.default_rng(19)
    q = rng.standard_normal(576)
    keys = rng.standard_normal((50, 576)) * 2
    s = 0.1 * keys @ q
    for sink in (None, 3.0, -2.0):
        out, lse = orc.attend(q, keys, 0.1, sink)
        total = np.exp(s - lse).sum() + (0.0 if sink is None else math.exp(sink - lse))
        assert abs(total - 1.0) <= 1e-13
        # the output is a convex combination of the values (weights sum to <= 1 with a sink)
        w = np.exp(s - lse)
        assert np.max(np.abs(out - w @ keys[:, :512])) <= 1e-12
    o1, l1 = orc.attend(q, keys, 0.1, None)
    o2, l2 = orc.attend(q, keys, 0.1, -1e300)
    assert np.array_equal(o1, o2) and l1 == l2


def check_merge_partition(orc):
    rng = np.random.default_rng(23)
    q = rng.standard_normal(576)
    keys = rng.standard_normal((37, 576)) * 1.5
    for sink in (None, 0.3):
        whole_o, whole_l = orc.attend(q, keys, 0.2, sink)
        for S in (1, 2, 4, 6):
            lab = rng.integers(0, S, size=37)
            lses, outs = [], []
            for c in range(S):
                o, l = orc.attend(q, keys[lab == c], 0.2, None)
                lses.append(l)
                outs.append(o)
            mo, ml = orc.merge(lses, np.stack(outs), sink)
            assert abs(ml - whole_l) <= 1e-12 * max(1.0, abs(whole_l))
            assert np.max(np.abs(mo - whole_o)) <= 1e-12


def check_empty_and_bad_index(orc):
    w = synth.small_config(4)
    w2 = synth.Workload(**{**w.__dict__, "seq_lens": w.seq_lens.copy()})
    w2.seq_lens[1] = 0
    out, lse, bad = orc.sparse_mla_decode(w2, tokens=[1], n_threads=1)
    assert bad == 0 and not out.any()
    assert np.array_equal(lse[0], w.sink.astype(np.float64))   # only the sink remains
    # a block-table hole under token 0's window: those keys are skipped and counted
    t = 0
    pos = int(w.seq_lens[t]) - 1
    bt = w.block_table.copy()
    row = 0 if w.req_idx is None else int(w.req_idx[t])
    bt[row, pos // w.page] = -1
    w3 = synth.Workload(**{**w.__dict__, "block_table": bt})
    _, _, bad = orc.sparse_mla_decode(w3, tokens=[t], n_threads=1)
    assert bad > 0


def check_topk_lens_truncation(orc):
    """Entries past topk_lens are never read, whatever they hold."""
    w = synth.small_config(3)
    rng = np.random.default_rng(29)
    lens = rng.integers(0, w.topk_width + 1, size=w.num_tokens).astype(np.int32)
    cut = w.topk_idx.copy()
    for t in range(w.num_tokens):
        cut[t, lens[t]:] = -1
    a = orc.sparse_mla_decode(synth.Workload(**{**w.__dict__, "topk_lens": lens}), n_threads=2)
    b = orc.sparse_mla_decode(synth.Workload(**{**w.__dict__, "topk_idx": cut, "topk_lens": None}), n_threads=2)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    c = orc.sparse_mla_decode(w, n_threads=2)
    assert not np.array_equal(a[1], c[1])


# ----------------------------------------------------------------------------
# compressed-region combine
# ----------------------------------------------------------------------------
GOLDEN_COMPRESSED = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                                 "combine_compressed_worked_examples.txt")
GOLDEN_TOPK = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "topk_select_worked_examples.txt")


def load_golden_compressed():
    examples, cur = [], None
    with open(GOLDEN_COMPRESSED) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "example":
                cur = dict(name=rest, requests=[], tokens=[])
            elif key == "params":
                cur["M"], cur["N"], cur["top_k"], cur["C"], cur["W"], cur["width"] = [int(v) for v in rest.split()]
            elif key == "request":
                cur["requests"].append([int(v) for v in rest.split()])
            elif key == "token":
                topk, row, ln = [p.strip() for p in rest.split("|")]
                cur["tokens"].append(([int(v) for v in topk.split()], [int(v) for v in row.split()], int(ln)))
            elif key == "end":
                examples.append(cur)
    return examples


def check_combine_compressed_golden(orc):
    for ex in load_golden_compressed():
        qlens = [r[0] for r in ex["requests"]]
        qsl = np.array([100] + list(100 + np.cumsum(qlens)), dtype=np.int32)
        width = max(len(t[0]) for t in ex["tokens"])
        topk = np.array([t[0] + [-1] * (width - len(t[0])) for t in ex["tokens"]], dtype=np.int32)
        row, ln = orc.combine_compressed(topk, qsl, [r[1] for r in ex["requests"]], [r[2] for r in ex["requests"]],
                                         ex["M"], ex["N"], ex["top_k"], ex["C"], ex["W"], ex["width"])
        for i, (_, want, wl) in enumerate(ex["tokens"]):
            assert row[i].tolist() == want, (ex["name"], i, row[i].tolist(), want)
            assert int(ln[i]) == wl, (ex["name"], i)


def check_combine_compressed_invariants(orc):
    """Random batches: lengths follow min((pos+1)//C, TOP_K) + min(pos+1, W); the window part is a
    run of consecutive entries ending at the token's own position in its request's region; top-k
    entries keep their order and map into [M*b, M*b + N) or to -1; the rest is -1."""
    rng = np.random.default_rng(31)
    for _ in range(60):
        R = int(rng.integers(1, 6))
        qlens = rng.integers(0, 4, size=R)
        seqs = rng.integers(0, 300, size=R)
        gl = np.minimum(seqs, rng.integers(0, 300, size=R) + 20)
        M, N, top_k, C, W = 1000, int(rng.integers(1, 200)), int(rng.integers(0, 40)), int(rng.integers(1, 9)), int(rng.integers(0, 30))
        T = int(qlens.sum())
        K = top_k + int(rng.integers(0, 5))
        topk = rng.integers(-3, N + 3, size=(max(T, 1), K)).astype(np.int32)[:T]
        qsl = np.concatenate([[7], 7 + np.cumsum(qlens)]).astype(np.int32)
        width = top_k + W + int(rng.integers(0, 4))
        row, ln = orc.combine_compressed(topk.reshape(T, K), qsl, seqs, gl, M, N, top_k, C, W, width)
        t = 0
        for b in range(R):
            for i in range(int(qlens[b])):
                pos = int(seqs[b]) - int(qlens[b]) + i
                tk = min((pos + 1) // C, top_k) if pos + 1 > 0 else 0
                sw = min(pos + 1, W) if pos + 1 > 0 else 0
                assert int(ln[t]) == tk + sw
                for k in range(tk):
                    v = int(topk[t, k])
                    assert row[t, k] == (M * b + v if 0 <= v < N else -1)
                win = row[t, tk:tk + sw]
                if sw:
                    assert np.all(np.diff(win) == 1)
                    assert int(win[-1]) == M * b + N + pos - (int(seqs[b]) - int(gl[b]))
                assert np.all(row[t, tk + sw:] == -1)
                t += 1


def load_golden_topk():
    examples, cur = [], None
    with open(GOLDEN_TOPK) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "example":
                cur = dict(name=rest, rows=[])
            elif key == "params":
                cur["K"], cur["width"] = [int(v) for v in rest.split()]
            elif key == "row":
                nc, sc, want, ln = [p.strip() for p in rest.split("|")]
                cur["rows"].append((int(nc), [float(v) for v in sc.split()], [int(v) for v in want.split()], int(ln)))
            elif key == "end":
                examples.append(cur)
    return examples


def check_topk_golden(orc):
    for ex in load_golden_topk():
        sc = np.array([r[1] for r in ex["rows"]], dtype=np.float32)
        assert sc.shape[1] == ex["width"], ex["name"]
        idx, ln = orc.topk_select(sc, [r[0] for r in ex["rows"]], ex["K"])
        for i, (_, _, want, wl) in enumerate(ex["rows"]):
            assert idx[i].tolist() == want, (ex["name"], i, idx[i].tolist(), want)
            assert int(ln[i]) == wl, (ex["name"], i)


def check_topk_distinct_vs_argpartition(orc):
    """Distinct scores: the selected set is numpy's argpartition of the candidates."""
    rng = np.random.default_rng(41)
    for _ in range(40):
        width = int(rng.integers(1, 400))
        T = int(rng.integers(1, 5))
        K = int(rng.integers(1, 300))
        sc = np.stack([rng.permutation(width).astype(np.float32) * np.float32(rng.choice([-1.5, 0.25, 3.0]))
                       + np.float32(rng.normal()) for _ in range(T)])
        nc = rng.integers(-3, width + 5, size=T).astype(np.int32)
        idx, ln = orc.topk_select(sc, nc, K)
        for t in range(T):
            n = int(min(max(nc[t], 0), width))
            m = min(K, n)
            want = np.sort(np.argpartition(-sc[t, :n].astype(np.float64), m - 1)[:m]) if m > 0 else np.zeros(0, int)
            assert idx[t, :m].tolist() == want.tolist()
            assert np.all(idx[t, m:] == -1) and int(ln[t]) == m


def check_topk_invariants(orc):
    """Tie-heavy rows with signed zeros, infinities and NaN: the row is ascending and -1 padded,
    its length is min(K, n), and no candidate left out precedes a selected one in the order
    (score, with -0 == +0 and NaN lowest; then position)."""
    rng = np.random.default_rng(43)
    pool = np.array([0.0, -0.0, 1.0, -1.0, 2.5, np.inf, -np.inf, np.nan, 7.0], dtype=np.float32)
    for _ in range(60):
        width = int(rng.integers(1, 120))
        T = int(rng.integers(1, 4))
        K = int(rng.integers(1, 60))
        sc = rng.choice(pool, size=(T, width)).astype(np.float32)
        nc = rng.integers(0, width + 3, size=T).astype(np.int32)
        idx, ln = orc.topk_select(sc, nc, K)
        for t in range(T):
            n = int(min(nc[t], width))
            m = min(K, n)
            sel = idx[t, :m].tolist()
            assert int(ln[t]) == m and np.all(idx[t, m:] == -1)
            assert sel == sorted(set(sel)) and all(0 <= p < n for p in sel)

            def rank(p):   # smaller = earlier in the order
                x = float(sc[t, p])
                return (1, 0.0, p) if np.isnan(x) else (0, -x, p)
            if 0 < m < n:
                worst_in = max(rank(p) for p in sel)
                best_out = min(rank(p) for p in range(n) if p not in set(sel))
                assert worst_in < best_out, (t, worst_in, best_out)


# ----------------------------------------------------------------------------
# fused Q RMSNorm + GPT-J RoPE + FP8/UE8M0 KV insert
# ----------------------------------------------------------------------------
def _bf16(x):
    return synth.bf16_bits(np.asarray(x, dtype=np.float32))


def _from_bf16(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _rope_table(angles):
    """fp32 [P, 64]: cos then sin of angles [P, 32]."""
    a = np.asarray(angles, dtype=np.float64)
    return np.concatenate([np.cos(a), np.sin(a)], axis=1).astype(np.float32)


def check_e4m3_encode(orc):
    """The oracle's E4M3 encoder equals torch's float8_e4m3fn cast (round to nearest even) on every
    code value, every midpoint between neighbouring codes and random values of every binade."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    pos = np.unique(vals[vals >= 0])
    mids = (pos[1:] + pos[:-1]) / 2
    rng = np.random.default_rng(51)
    rand = np.ldexp(rng.uniform(1, 2, 3000), rng.integers(-12, 9, 3000))
    ys = np.concatenate([vals, mids, -mids, rand[rand <= 448], -rand[rand <= 448]])
    want = torch.from_numpy(ys).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(y) for y in ys], dtype=np.uint8)
    same = (got == want) | ((got & 0x7F) == 0) & ((want & 0x7F) == 0)   # signed zeros
    assert np.all(same), (ys[~same][:5], got[~same][:5], want[~same][:5])


def check_kv_insert_latent(orc):
    """The latent codes and scale bytes equal the generator's independent encoder; with the
    identity rotation the rope bytes are the input BF16 bits; the padding is zero; the decoded
    latent is within half an E4M3 step of the input."""
    rng = np.random.default_rng(53)
    T = 40
    lat = rng.standard_normal((T, 512)) * np.ldexp(1.0, rng.integers(-30, 30, (T, 1)))
    lat[0] = 0.0
    lat[1, :128] = 448.0
    rope = rng.standard_normal((T, 64))
    kv = np.concatenate([_bf16(lat), _bf16(rope)], axis=1)
    cache = np.full((T + 3, 656), 0xAB, dtype=np.uint8)
    slots = np.arange(T, dtype=np.int64) + 2
    out, bad = orc.kv_insert(kv, slots, np.zeros(T, np.int64), _rope_table(np.zeros((1, 32))), cache)
    assert bad == 0
    want = synth.quantize_entries(_from_bf16(kv[:, :512]), _from_bf16(kv[:, 512:]))
    assert np.array_equal(out[2:T + 2], want)
    assert np.all(out[:2] == 0xAB) and np.all(out[T + 2:] == 0xAB)
    for t in range(T):
        k = orc.dequant_entry(out[2 + t])[:512]
        x = _from_bf16(kv[t, :512])
        step = np.ldexp(1.0, int(out[2 + t, 640 + 0]) - 127)   # block 0's scale
        assert np.all(np.abs(k[:128] - x[:128]) <= step * 32 + 1e-300)   # within half a step of 2^(e-127) * 64


def check_rope_closed_forms(orc):
    """GPT-J pairs: a rotation by 90 degrees maps (x, y) to (-y, x) exactly; a vector with one
    nonzero rope dim 512 + 2i keeps its energy in dims 512 + 2i and 513 + 2i; pair norms are kept."""
    rng = np.random.default_rng(57)
    T = 6
    lat = rng.standard_normal((T, 512))
    rope = rng.standard_normal((T, 64))
    kv = np.concatenate([_bf16(lat), _bf16(rope)], axis=1)
    table = _rope_table(np.stack([np.full(32, np.pi / 2), rng.uniform(0, 6.3, 32)]))
    table[0, :32] = 0.0   # exact cos 0
    table[0, 32:] = 1.0   # exact sin 1
    cache = np.zeros((T, 656), dtype=np.uint8)
    out, _ = orc.kv_insert(kv, np.arange(T), np.zeros(T, np.int64), table, cache)
    r = _from_bf16(out[:, 512:640].copy().view("<u2"))
    x = _from_bf16(kv[:, 512:])
    assert np.array_equal(r[:, 0::2], -x[:, 1::2]) and np.array_equal(r[:, 1::2], x[:, 0::2])
    one = np.zeros((1, 576), dtype=np.uint16)
    one[0, 512 + 6] = _bf16([1.0])[0]
    out1, _ = orc.kv_insert(one, [0], [1], table, np.zeros((1, 656), np.uint8))
    r1 = _from_bf16(out1[0, 512:640].copy().view("<u2"))
    nz = set(np.nonzero(r1)[0].tolist())
    assert nz <= {6, 7} and 6 in nz, nz
    out2, _ = orc.kv_insert(kv, np.arange(T), np.ones(T, np.int64), table, cache)
    r2 = _from_bf16(out2[:, 512:640].copy().view("<u2"))
    n_in = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
    n_out = r2[:, 0::2] ** 2 + r2[:, 1::2] ** 2
    assert np.allclose(n_in, n_out, rtol=2 ** -6, atol=1e-6)


def check_qnorm_closed_forms(orc):
    """A constant head c gives sign(c) / sqrt(1 + eps / c^2) in every dim (also at c = 2^-10, where
    eps matters); the output's mean square is ms / (ms + eps); a weight of 2 doubles the output
    exactly; a head whose only nonzero dims are rope dims is divided by sqrt(sum / 576) (the mean
    runs over all 576 dims); zero stays zero."""
    eps = 1e-6
    ident = _rope_table(np.zeros((1, 32)))
    qs = np.zeros((1, 1, 576), dtype=np.uint16)
    qs[0, 0] = _bf16(np.full(576, 2.0 ** -10))
    ys = _from_bf16(orc.qnorm_rope(qs, [0], ident, None, eps)[0])
    want_s = 2.0 ** -10 / np.sqrt(2.0 ** -20 + eps)
    assert np.all(np.abs(ys - want_s) <= want_s * 2 ** -8), (ys[0, 0, 0], want_s)
    q = np.zeros((1, 4, 576), dtype=np.uint16)
    q[0, 0] = _bf16(np.full(576, -3.0))
    q[0, 1] = _bf16(np.random.default_rng(59).standard_normal(576))
    q[0, 2, 512:] = _bf16(np.full(64, 2.0))
    out, bad = orc.qnorm_rope(q, [0], ident, None, eps)
    assert bad == 0
    y = _from_bf16(out)
    assert np.all(y[0, 0] == _from_bf16(_bf16([-1.0 / np.sqrt(1 + eps / 9.0)]))[0])
    x1 = _from_bf16(q[0, 1])
    ms = np.mean(x1 ** 2)
    assert abs(np.mean(y[0, 1] ** 2) - ms / (ms + eps)) < 2 ** -7
    want2 = 2.0 / np.sqrt(64 * 4.0 / 576 + eps)
    assert np.all(y[0, 2, :512] == 0) and np.all(np.abs(y[0, 2, 512:] - want2) <= want2 * 2 ** -8)
    assert np.all(y[0, 3] == 0)
    out_w, _ = orc.qnorm_rope(q, [0], ident, np.full(576, 2.0, np.float32), eps)
    assert np.array_equal(_from_bf16(out_w), 2 * y)


def check_insert_slots_and_positions(orc):
    """A negative slot writes nothing and is not counted; a slot past the cache or a position
    outside the table writes nothing and is counted; such a query is normalised, not rotated."""
    rng = np.random.default_rng(61)
    kv = _bf16(rng.standard_normal((4, 576)))
    table = _rope_table(rng.uniform(0, 6, (3, 32)))
    cache = np.full((5, 656), 7, dtype=np.uint8)
    out, bad = orc.kv_insert(kv, [-1, 5, 2, 1], [0, 1, 3, 2], table, cache)
    assert bad == 2
    assert np.all(out[[0, 2, 3, 4]] == 7) and not np.all(out[1] == 7)
    q = _bf16(rng.standard_normal((2, 1, 576))).reshape(2, 1, 576)
    qo, qbad = orc.qnorm_rope(q, [-4, 2], table)
    assert qbad == 1
    qi, _ = orc.qnorm_rope(q, [0, 2], _rope_table(np.zeros((3, 32))))
    assert np.array_equal(qo[0], qi[0]) and not np.array_equal(qo[1], qi[1])


ALL_CHECKS = [check_e4m3_codes, check_ue8m0, check_bf16, check_entry_layout, check_quantize_roundtrip,
              check_combine_golden, check_combine_bruteforce, check_combine_config1_lengths,
              check_dense_equivalence, check_order_padding_invariance, check_page_permutation, check_closed_forms,
              check_lse_identity_and_sink_limit, check_merge_partition, check_empty_and_bad_index,
              check_topk_lens_truncation, check_combine_compressed_golden, check_combine_compressed_invariants,
              check_topk_golden, check_topk_distinct_vs_argpartition, check_topk_invariants,
              check_e4m3_encode, check_kv_insert_latent, check_rope_closed_forms, check_qnorm_closed_forms,
              check_insert_slots_and_positions]
