"""fp64 CPU oracle for DeepSeek-V4 sparse-MLA decode (ctypes binding to oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module.  It shares no code with
the CUDA library; it is compiled from ``oracle.c`` with the host C compiler.

Each function restates one step of the path (oracle.c names the page and
section each follows):
  * ``e4m3_to_f64`` / ``ue8m0_to_f64`` / ``bf16_to_f64`` / ``dequant_entry`` - the cache format,
  * ``combine`` - top-k + sliding-window index combine with dedup and compaction,
  * ``combine_compressed`` - the compressed-region variant of the combine,
  * ``topk_select`` - top-k selection from indexer scores (what produces the top-k rows),
  * ``qnorm_rope`` / ``kv_insert`` - the fused Q RMSNorm + GPT-J RoPE and FP8 KV-cache insert,
  * ``attend`` - sink-softmax MQA attention of one head over explicit keys,
  * ``merge`` - log-sum-exp merge of partial results over disjoint key sets,
  * ``sparse_mla_decode`` - the whole decode for all (or a subset of) tokens.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_default = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source into a shared library (plain C, no fast-math, no FMA contraction)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB)
    return _LIB


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """The oracle functions bound to one compiled library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_e4m3_to_double.restype = f64
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_ue8m0_to_double.restype = f64
        lib.oracle_ue8m0_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_bf16_to_double.restype = f64
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_dequant_entry.restype = None
        lib.oracle_dequant_entry.argtypes = [P, P]
        lib.oracle_combine.restype = ctypes.c_int
        lib.oracle_combine.argtypes = [P, i64, i32, P, P, i32, i32, P, i64, i32, P]
        lib.oracle_combine_compressed.restype = ctypes.c_int
        lib.oracle_combine_compressed.argtypes = [P, i64, i32, P, P, P, i32, i32, i32, i32, i32, i32, P, i64, i32, P]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [f64]
        lib.oracle_qnorm_rope.restype = i64
        lib.oracle_qnorm_rope.argtypes = [P, i64, i32, i32, P, f64, P, P, i32, P, i64]
        lib.oracle_kv_insert.restype = i64
        lib.oracle_kv_insert.argtypes = [P, i64, i32, P, P, P, i32, P, i64]
        lib.oracle_topk_select.restype = ctypes.c_int
        lib.oracle_topk_select.argtypes = [P, i64, i32, P, i32, i32, P, i64, P]
        lib.oracle_attend.restype = None
        lib.oracle_attend.argtypes = [P, P, i32, f64, ctypes.c_int, f64, P, P]
        lib.oracle_merge.restype = None
        lib.oracle_merge.argtypes = [i32, P, P, ctypes.c_int, f64, P, P]
        lib.oracle_sparse_mla_decode.restype = i64
        lib.oracle_sparse_mla_decode.argtypes = [P, i64, P, i32, i32, P, i64, i32, i32, P, P, i64, i32, P, P,
                                                 i32, i32, i32, P, f64, P, P, P, i32, i32, i32, i32]
        self.lib = lib

    def e4m3_to_f64(self, code: int) -> float:
        return self.lib.oracle_e4m3_to_double(int(code))

    def ue8m0_to_f64(self, e: int) -> float:
        return self.lib.oracle_ue8m0_to_double(int(e))

    def bf16_to_f64(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(int(bits))

    def dequant_entry(self, entry: np.ndarray) -> np.ndarray:
        """656-byte cache entry -> fp64 key [576] (latent 512, then rope 64)."""
        e = _c(entry, np.uint8)
        assert e.size == 656
        k = np.zeros(576, dtype=np.float64)
        self.lib.oracle_dequant_entry(_ptr(e), _ptr(k))
        return k

    def combine(self, topk_idx, topk_lens, seq_lens, window: int, combined_width: int):
        """Returns (combined int32 [T, width], combined_lens int32 [T])."""
        tk = _c(topk_idx, np.int32)
        T, K = tk.shape
        out = np.empty((T, combined_width), dtype=np.int32)
        lens = np.empty(T, dtype=np.int32)
        rc = self.lib.oracle_combine(_ptr(tk), K, K, _ptr(_c(topk_lens, np.int32)), _ptr(_c(seq_lens, np.int32)), T,
                                     int(window), _ptr(out), combined_width, combined_width, _ptr(lens))
        if rc != 0:
            raise ValueError("combined_width too small")
        return out, lens

    def combine_compressed(self, topk_idx, query_start_loc, seq_lens, gather_lens, region_stride: int,
                           compressed_len: int, top_k: int, compress_ratio: int, window: int, combined_width: int):
        """Compressed-region combine -> (combined int32 [T, width], combined_lens int32 [T])."""
        tk = _c(topk_idx, np.int32)
        T, K = tk.shape
        qsl = _c(query_start_loc, np.int32)
        R = qsl.size - 1
        out = np.empty((T, combined_width), dtype=np.int32)
        lens = np.empty(T, dtype=np.int32)
        rc = self.lib.oracle_combine_compressed(_ptr(tk), K, K, _ptr(qsl), _ptr(_c(seq_lens, np.int32)),
                                                _ptr(_c(gather_lens, np.int32)), R, int(region_stride),
                                                int(compressed_len), int(top_k), int(compress_ratio), int(window),
                                                _ptr(out), combined_width, combined_width, _ptr(lens))
        if rc != 0:
            raise ValueError("arguments outside the compressed combine's rules")
        return out, lens

    def e4m3_encode(self, y: float) -> int:
        """E4M3FN code of a finite |y| <= 448, round to nearest even."""
        return int(self.lib.oracle_e4m3_encode(float(y)))

    def qnorm_rope(self, q_bits, positions, cos_sin, norm_w=None, eps: float = 1e-6):
        """q_bits uint16 BF16 [T, H, 576] -> (normalised, rotated q bits uint16 [T, H, 576], bad count)."""
        q = _c(q_bits, np.uint16)
        T, H, _ = q.shape
        cs = _c(cos_sin, np.float32)
        w = None if norm_w is None else _c(norm_w, np.float32)
        out = np.empty_like(q)
        bad = self.lib.oracle_qnorm_rope(_ptr(q), H * 576, T, H, None if w is None else _ptr(w), float(eps),
                                         _ptr(_c(positions, np.int64)), _ptr(cs), cs.shape[0], _ptr(out), H * 576)
        return out, int(bad)

    def kv_insert(self, kv_bits, slots, positions, cos_sin, cache):
        """kv_bits uint16 BF16 [T, 576] into a copy of cache uint8 [S, 656] -> (cache, bad count)."""
        kv = _c(kv_bits, np.uint16)
        cs = _c(cos_sin, np.float32)
        c = np.array(cache, dtype=np.uint8, copy=True, order="C")
        bad = self.lib.oracle_kv_insert(_ptr(kv), 576, kv.shape[0], _ptr(_c(slots, np.int64)),
                                        _ptr(_c(positions, np.int64)), _ptr(cs), cs.shape[0], _ptr(c),
                                        c.reshape(-1, 656).shape[0])
        return c, int(bad)

    def topk_select(self, scores, num_cand, top_k: int):
        """Top-k selection -> (topk_idx int32 [T, K] ascending then -1, topk_lens int32 [T])."""
        sc = _c(scores, np.float32)
        T, width = sc.shape
        out = np.empty((T, top_k), dtype=np.int32)
        lens = np.empty(T, dtype=np.int32)
        rc = self.lib.oracle_topk_select(_ptr(sc), width, width, _ptr(_c(num_cand, np.int32)), T, int(top_k),
                                         _ptr(out), top_k, _ptr(lens))
        if rc != 0:
            raise ValueError("top_k must be at least 1")
        return out, lens

    def attend(self, q, keys, softmax_scale: float, sink: Optional[float] = None):
        """One head: q fp64 [576], keys fp64 [L, 576] -> (out fp64 [512], lse float)."""
        qq = _c(q, np.float64)
        kk = _c(keys, np.float64).reshape(-1, 576)
        out = np.zeros(512, dtype=np.float64)
        lse = np.zeros(1, dtype=np.float64)
        self.lib.oracle_attend(_ptr(qq), _ptr(kk), kk.shape[0], float(softmax_scale), int(sink is not None),
                               0.0 if sink is None else float(sink), _ptr(out), _ptr(lse))
        return out, float(lse[0])

    def merge(self, lse_parts: Sequence[float], out_parts, sink: Optional[float] = None):
        lp = _c(lse_parts, np.float64)
        op = _c(out_parts, np.float64).reshape(-1, 512)
        out = np.zeros(512, dtype=np.float64)
        lse = np.zeros(1, dtype=np.float64)
        self.lib.oracle_merge(lp.size, _ptr(lp), _ptr(op), int(sink is not None),
                              0.0 if sink is None else float(sink), _ptr(out), _ptr(lse))
        return out, float(lse[0])

    def sparse_mla_decode(self, w, tokens: Optional[Sequence[int]] = None, n_threads: Optional[int] = None,
                          heads: Optional[tuple] = None):
        """Decode for workload `w` (a synth.Workload or anything with the same fields).

        Returns (out fp64 [n, nh, 512], lse fp64 [n, nh], bad_key_count); rows follow
        `tokens` (default: all tokens in order), heads the range `heads` = (begin, end)
        (default: all heads).
        """
        q = _c(w.q, np.uint16)
        T, H, D = q.shape
        assert D == 576
        cache = np.ascontiguousarray(w.kv_cache)
        assert cache.dtype == np.uint8
        bt = _c(w.block_table, np.int32)
        tk = _c(w.topk_idx, np.int32)
        tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n = T if tok is None else tok.size
        h0, h1 = (0, H) if heads is None else (int(heads[0]), int(heads[1]))
        assert 0 <= h0 <= h1 <= H
        out = np.zeros((n, h1 - h0, 512), dtype=np.float64)
        lse = np.zeros((n, h1 - h0), dtype=np.float64)
        if n_threads is None:
            n_threads = os.cpu_count() or 1
        bad = self.lib.oracle_sparse_mla_decode(
            _ptr(q), H * 576, _ptr(cache), cache.shape[0], cache.shape[1], _ptr(bt), bt.shape[1], bt.shape[1],
            bt.shape[0], _ptr(_c(w.req_idx, np.int32)), _ptr(tk), tk.shape[1], tk.shape[1],
            _ptr(_c(w.topk_lens, np.int32)), _ptr(_c(w.seq_lens, np.int32)), T, H, int(w.window),
            _ptr(_c(w.sink, np.float32)), float(w.softmax_scale), _ptr(out), _ptr(lse), _ptr(tok), n, h0, h1,
            int(n_threads))
        return out, lse, int(bad)


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def e4m3_to_f64(code):
    return default().e4m3_to_f64(code)


def ue8m0_to_f64(e):
    return default().ue8m0_to_f64(e)


def bf16_to_f64(bits):
    return default().bf16_to_f64(bits)


def dequant_entry(entry):
    return default().dequant_entry(entry)


def combine(topk_idx, topk_lens, seq_lens, window, combined_width):
    return default().combine(topk_idx, topk_lens, seq_lens, window, combined_width)


def combine_compressed(topk_idx, query_start_loc, seq_lens, gather_lens, region_stride, compressed_len, top_k,
                       compress_ratio, window, combined_width):
    return default().combine_compressed(topk_idx, query_start_loc, seq_lens, gather_lens, region_stride,
                                        compressed_len, top_k, compress_ratio, window, combined_width)


def e4m3_encode(y):
    return default().e4m3_encode(y)


def qnorm_rope(q_bits, positions, cos_sin, norm_w=None, eps=1e-6):
    return default().qnorm_rope(q_bits, positions, cos_sin, norm_w, eps)


def kv_insert(kv_bits, slots, positions, cos_sin, cache):
    return default().kv_insert(kv_bits, slots, positions, cos_sin, cache)


def topk_select(scores, num_cand, top_k):
    return default().topk_select(scores, num_cand, top_k)


def attend(q, keys, softmax_scale, sink=None):
    return default().attend(q, keys, softmax_scale, sink)


def merge(lse_parts, out_parts, sink=None):
    return default().merge(lse_parts, out_parts, sink)


def sparse_mla_decode(w, tokens=None, n_threads=None, heads=None):
    return default().sparse_mla_decode(w, tokens, n_threads, heads)
