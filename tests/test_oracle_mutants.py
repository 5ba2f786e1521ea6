"""Planted mistakes in copies of the oracle must be caught by the pins.

Each mutant is the oracle's C source with one plausible mistake (a dropped
term, a wrong index, a wrong causal offset, a transposed operand ...),
compiled to a temporary library.  The test passes only if at least one pin
of ``oracle_pins`` fails on it, which shows the pins constrain every part of
the oracle's arithmetic.  Runs on the CPU only.
"""

import os

import pytest

import oracle
from tests import oracle_pins

MUTANTS = {
    "no_scale": ("w[t] = scale * dot;", "w[t] = dot;"),
    "gqa_modulo": ("hd, h / group, scale, w, o);", "hd, h % hkv, scale, w, o);"),
    "gqa_modulo_prefill": ("n_keys, bs, hkv, hd, h / group,", "n_keys, bs, hkv, hd, h % hkv,"),
    "causal_off_by_one": ("const int64_t n_keys = (L - n) + j + 1;", "const int64_t n_keys = (L - n) + j;"),
    "top_left_causal": ("const int64_t n_keys = (L - n) + j + 1;", "const int64_t n_keys = j + 1;"),
    "no_causal_mask": ("const int64_t n_keys = (L - n) + j + 1;", "const int64_t n_keys = L;"),
    "v_from_k_cache": ("out[d] += p * widen_bf16(v_cache[base + d]);", "out[d] += p * widen_bf16(k_cache[base + d]);"),
    "slot_wrong_offset": ("return (int64_t)table[p / bs] * bs + p % bs;", "return (int64_t)table[p / bs] * bs + p / bs;"),
    "slot_ignores_table": ("return (int64_t)table[p / bs] * bs + p % bs;", "return p;"),
    "no_normalisation": ("const double p = w[t] / denom;", "const double p = w[t];"),
    "max_not_subtracted_wrong": ("w[t] = exp(w[t] - m);", "w[t] = exp(w[t] + m);"),
    "decode_drops_new_token": ("L, bs, hkv,\n                 hd, h / group, scale, w, o);",
                               "L - 1, bs, hkv,\n                 hd, h / group, scale, w, o);"),
    "pad_rows_not_zero": ("if (L == 0 || !w) {\n        for (int64_t d = 0; d < hd; ++d) o[d] = 0.0;",
                          "if (L == 0 || !w) {\n        for (int64_t d = 0; d < hd; ++d) o[d] = 1.0;"),
    "write_no_skip": ("    if (s == -1) continue;\n    for (int64_t e", "    if (s == -1) s = 0;\n    for (int64_t e"),
    "write_v_from_k": ("v_cache[s * row_elems + e] = v[i * v_token_stride + e];",
                       "v_cache[s * row_elems + e] = k[i * k_token_stride + e];"),
    "write_ignores_stride": ("k_cache[s * row_elems + e] = k[i * k_token_stride + e];",
                             "k_cache[s * row_elems + e] = k[i * row_elems + e];"),
    "philox_nine_rounds": ("for (int r = 0; r < 10; ++r) {", "for (int r = 0; r < 9; ++r) {"),
    "philox_wrong_weyl": ("k[0] += 0x9E3779B9u;", "k[0] += 0x9E3779B8u;"),
    "sampler_no_temperature": ("p[i] = exp((double)l[i] / T - m);", "p[i] = exp((double)l[i] - m);"),
    "sampler_times_noise": ("const double q = (p[i] / sum) / E;", "const double q = (p[i] / sum) * E;"),
    "dot_wrong_index": ("widen_bf16(qrow[d]) * widen_bf16(k_cache[base + d]);",
                        "widen_bf16(qrow[d]) * widen_bf16(k_cache[base + (d + 1) % hd]);"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation anchor for {name} not unique in the oracle source"
    src = tmp_path / f"{name}.c"
    src.write_text(source.replace(old, new))
    lib = oracle.compile_source(str(src), str(tmp_path / f"lib{name}.so"))
    orc = oracle.Oracle(lib)
    orc.set_num_threads(min(4, os.cpu_count() or 1))
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, oracle.OracleError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
