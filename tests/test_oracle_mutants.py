"""Plants plausible mistakes in copies of the oracle (CPU only) and checks that
the pins of tests/oracle_pins.py catch every one of them.

Each mutant is oracle.c with one textual change, compiled into a temporary
library; the real oracle.c is never modified.
"""
import os

import pytest

import oracle
import oracle_pins

# (name, original text, replacement) -- each original must occur in oracle.c; a tuple
# pair applies several replacements to one mutant
MUTANTS = [
    ("rope dropped from the logit", "for (int d = 0; d < OR_DIM; ++d)\n            acc +=",
     "for (int d = 0; d < OR_LATENT; ++d)\n            acc +="),
    ("value read from the wrong dims", "out[d] += w * keys[(int64_t)j * OR_DIM + d];",
     "out[d] += w * keys[(int64_t)j * OR_DIM + d + 64];"),
    ("sink scaled like a logit", "jb->sink ? (double)jb->sink[h] : 0.0", "jb->sink ? (double)jb->sink[h] * jb->softmax_scale : 0.0"),
    ("sink left out of the normaliser", "    if (has_sink)\n        z += exp(sink - m);\n    double l = m + log(z);\n    for (int32_t j",
     "    double l = m + log(z);\n    for (int32_t j"),
    ("window one too long", "int32_t win_lo = pos - window + 1;", "int32_t win_lo = pos - window;"),
    ("window not excluded from top-k", "if (v >= win_lo)\n            continue;", "if (v > pos + 1)\n            continue;"),
    ("no dedup of repeats", "if (row[j] == v) {", "if (0) {"),
    ("non-causal entries kept", ("if (v < 0 || v > pos)", "if (v >= win_lo)\n            continue;"),
     ("if (v < 0)", "if (v >= win_lo && v <= pos)\n            continue;")),
    ("position = seq_len", "int32_t pos = seq_len - 1;", "int32_t pos = seq_len;"),
    ("scale bias off by one", "return ldexp(1.0, (int)e - 127);", "return ldexp(1.0, (int)e - 128);"),
    ("scale block of 64", "entry[OR_SCALE_OFF + d / OR_SCALE_BLOCK]", "entry[OR_SCALE_OFF + (d / 64) % 4]"),
    ("e4m3 bias 8", "v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("e4m3 subnormal scale", "v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    ("rope byte order", "(uint16_t)entry[OR_ROPE_OFF + 2 * i] | (uint16_t)((uint16_t)entry[OR_ROPE_OFF + 2 * i + 1] << 8)",
     "(uint16_t)entry[OR_ROPE_OFF + 2 * i + 1] | (uint16_t)((uint16_t)entry[OR_ROPE_OFF + 2 * i] << 8)"),
    ("in-page offset shifted", "int32_t off = idx % jb->page_block;", "int32_t off = (idx + 1) % jb->page_block;"),
    ("request row ignored", "int32_t row = jb->req_idx ? jb->req_idx[t] : t;", "int32_t row = t;"),
    ("topk_lens ignored", "int32_t n = jb->topk_lens ? jb->topk_lens[t] : jb->topk_width;", "int32_t n = jb->topk_width;"),
    ("merge weights against the max", "double w = exp(lse_parts[c] - l);", "double w = exp(lse_parts[c] - m);"),
    ("lse without the log", "double l = m + log(z);\n    for (int32_t j", "double l = m + z;\n    for (int32_t j"),
    ("softmax scale dropped", "s[j] = softmax_scale * acc;", "s[j] = acc;"),
    ("compressed: position off by one", "const int64_t pos = start_pos + (t - qs);", "const int64_t pos = start_pos + (t - qs) + 1;"),
    ("compressed: ratio applied to pos", "tk = (pos + 1) / compress_ratio;", "tk = pos / compress_ratio;"),
    ("compressed: region offset dropped", "row[k] = (v >= 0 && v < compressed_len) ? (int32_t)(region + v) : -1;",
     "row[k] = (v >= 0 && v < compressed_len) ? (int32_t)v : -1;"),
    ("compressed: gather start ignored", "(pos - sw + 1 - gather_start) + j);", "(pos - sw + 1) + j);"),
    ("compressed: window before the compressed part", "(int32_t)(region + compressed_len + (pos - sw + 1 - gather_start) + j)",
     "(int32_t)(region + (pos - sw + 1 - gather_start) + j)"),
    ("compressed: invalid top-k compacted", "row[k] = (v >= 0 && v < compressed_len) ? (int32_t)(region + v) : -1;",
     "row[k] = (v >= 0 && v <= compressed_len) ? (int32_t)(region + v) : -1;"),
    ("top-k: ties to the larger position", "return a->pos < b->pos ? -1 : (a->pos > b->pos);      /* then the smaller position */",
     "return a->pos > b->pos ? -1 : (a->pos < b->pos);"),
    ("top-k: NaN ranked first", "return a->nan ? 1 : -1;                           /* NaN after every number */",
     "return a->nan ? -1 : 1;"),
    ("top-k: smaller scores first", "return a->v > b->v ? -1 : 1;                      /* larger score first */",
     "return a->v < b->v ? -1 : 1;"),
    ("top-k: one candidate too many", "int64_t n = num_cand[t];", "int64_t n = num_cand[t] + 1;"),
    ("top-k: selection order kept", "qsort(row, (size_t)m, sizeof(int32_t), ascending_i32);", ""),
    ("top-k: -0 below +0", "items[p].v = items[p].nan ? 0.0 : (double)x + 0.0;",
     "items[p].v = items[p].nan ? 0.0 : (signbit(x) && x == 0.0f ? -1e-300 : (double)x);"),
    ("top-k: length not capped by K", "topk_lens[t] = (int32_t)m;", "topk_lens[t] = (int32_t)n;"),
    ("q norm: mean over the latent only", "const double r = 1.0 / sqrt(ss / OR_DIM + eps);",
     "const double r = 1.0 / sqrt(ss / OR_LATENT + eps);"),
    ("q norm: eps outside the root", "const double r = 1.0 / sqrt(ss / OR_DIM + eps);",
     "const double r = 1.0 / (sqrt(ss / OR_DIM) + eps);"),
    ("q norm: weight ignored", "x[d] = x[d] * r * (norm_w ? (double)norm_w[d] : 1.0);", "x[d] = x[d] * r;"),
    ("rope: sine sign flipped", "*x = a * c - b * s;", "*x = a * c + b * s;"),
    ("rope: NeoX pairs in the key", ("rope_pair(&x[OR_LATENT + 2 * i], &x[OR_LATENT + 2 * i + 1], (double)cos_sin[pos * 64 + i],\n                      (double)cos_sin[pos * 64 + 32 + i]);\n        for (int i = 0; i < OR_ROPE; ++i)",),
     ("rope_pair(&x[OR_LATENT + i], &x[OR_LATENT + i + 32], (double)cos_sin[pos * 64 + i],\n                      (double)cos_sin[pos * 64 + 32 + i]);\n        for (int i = 0; i < OR_ROPE; ++i)",)),
    ("insert: scale byte off by one", "e[OR_SCALE_OFF + b] = (uint8_t)(ex + 127);", "e[OR_SCALE_OFF + b] = (uint8_t)(ex + 128);"),
    ("insert: codes rounded toward zero", "int q = (int)rint((2.0 * m - 1.0) * 8.0);", "int q = (int)floor((2.0 * m - 1.0) * 8.0);"),
    ("insert: scale exponent one high", "while (e < 127 && 448.0 * ldexp(1.0, e) < amax)", "while (e < 127 && 448.0 * ldexp(1.0, e) <= amax)"),
    ("insert: negative slot counted as bad", "if (slot < 0)\n            continue;\n        if (slot >= num_slots",
     "if (slot < 0) {\n            ++bad;\n            continue;\n        }\n        if (slot >= num_slots"),
]


@pytest.mark.parametrize("name,orig,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, orig, repl, tmp_path):
    mutated = open(oracle.SOURCE).read()
    origs, repls = (orig, repl) if isinstance(orig, tuple) else ((orig,), (repl,))
    for o, r in zip(origs, repls):
        assert mutated.count(o) >= 1, f"mutation site not found: {name}"
        mutated = mutated.replace(o, r, 1)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.compile_source(str(path), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError):
            caught.append(check.__name__)
    assert caught, f"no pin caught the mutant '{name}'"
