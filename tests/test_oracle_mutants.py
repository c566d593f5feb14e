"""Each planted mistake in a copy of the oracle must make at least one pin fail.

The mistakes are the plausible ones: a wrong row or head index, a dropped scale, a
softmax without the max subtraction or with the wrong sign, P multiplied into K instead
of V, the last token dropped, a combine that forgets the piece weights, an append or pack
that writes the wrong place, and a wrong bf16 upcast. The copies are compiled on the CPU
into a temporary folder; the real oracle is untouched.
"""
import os

import pytest

import pins
from oracle import oracle as orc

SRC = os.path.join(os.path.dirname(orc.__file__), "oracle.c")

# (name, [(old, new, occurrence index or None for all)])
MUTANTS = [
    ("gqa_strided_grouping",
     [("const int h = hk * group + j;", "const int h = j * H_kv + hk;", None)]),
    ("wrong_row_in_block",
     [("(size_t)(t % block_size);\n    for (int d = 0; d < D; ++d) {\n      Kc",
       "(size_t)((t + 1) % block_size);\n    for (int d = 0; d < D; ++d) {\n      Kc", None)]),
    ("scale_dropped", [("s[t] = sc * dot;", "s[t] = dot;", None)]),
    ("no_max_subtraction",
     [("den += exp(s[t] - mx);", "den += exp(s[t]);", None),
      ("const double p = exp(s[t] - mx) / den;", "const double p = exp(s[t]) / den;", None)]),
    ("softmax_sign_flipped",
     [("den += exp(s[t] - mx);", "den += exp(mx - s[t]);", None),
      ("const double p = exp(s[t] - mx) / den;", "const double p = exp(mx - s[t]) / den;", None)]),
    ("pv_reads_k", [("o[d] += p * Vc[(size_t)t * D + d];", "o[d] += p * Kc[(size_t)t * D + d];",
                     None)]),
    ("last_token_dropped",
     [("const int L = context_lens[b];",
       "const int L = context_lens[b] > 1 ? context_lens[b] - 1 : context_lens[b];", None)]),
    ("query_head_uses_kv_head_index",
     [("const size_t qoff = ((size_t)b * H + h) * (size_t)D;\n      double mx",
       "const size_t qoff = ((size_t)b * H + hk) * (size_t)D;\n      double mx", None)]),
    ("append_wrong_offset",
     [("(size_t)block * (size_t)block_size + (size_t)offset)",
       "(size_t)block * (size_t)block_size + (size_t)((offset + 1) % block_size))", None)]),
    ("pack_swaps_k_and_v",
     [("memcpy(dst, (const char*)k_cache + src, row_bytes);",
       "memcpy(dst, (const char*)v_cache + src, row_bytes);", None),
      ("memcpy(dst + row_bytes, (const char*)v_cache + src, row_bytes);",
       "memcpy(dst + row_bytes, (const char*)k_cache + src, row_bytes);", None)]),
    ("bf16_upcast_shift", [("((uint32_t)h) << 16", "((uint32_t)h) << 15", None)]),
    ("unpack_swaps_k_and_v",
     [("    memcpy((char*)k_cache + dst, src, row_bytes);\n    memcpy((char*)v_cache + dst, src + row_bytes, row_bytes);",
       "    memcpy((char*)k_cache + dst, src + row_bytes, row_bytes);\n    memcpy((char*)v_cache + dst, src, row_bytes);",
       None)]),
    ("unpack_wrong_row",
     [("((size_t)block * (size_t)block_size + (size_t)(t % block_size)) * row_bytes;\n    const char* src",
       "((size_t)block * (size_t)block_size + (size_t)((t + 1) % block_size)) * row_bytes;\n    const char* src",
       None)]),
    ("combine_forgets_weights", [("Lsum += l[j] * exp(m[j] - M);", "Lsum += l[j];", None)]),
    ("e4m3_wrong_bias", [("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)", None)]),
    ("e4m3_wrong_subnormal", [("ldexp(m / 8.0, -6)", "ldexp(m / 8.0, -7)", None)]),
    ("e2m1_wrong_bias", [("ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)", None)]),
    ("nvfp4_nibbles_swapped",
     [("(d & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 15)",
       "(d & 1) ? (unsigned)(byte & 15) : (unsigned)(byte >> 4)", None)]),
    ("f16_wrong_exponent_bias",
     [("mag = ldexp((double)(1024 + m), e - 25);", "mag = ldexp((double)(1024 + m), e - 24);",
       None)]),
    ("f16_subnormal_scale",
     [("mag = ldexp((double)m, -24);", "mag = ldexp((double)m, -25);", None)]),
    ("f16_sign_dropped", [("  return sign ? -mag : mag;\n}\n\ndouble oracle_decode_f16",
                           "  return mag;\n}\n\ndouble oracle_decode_f16", None)]),
    ("nvfp4_wrong_block_index",
     [("srow * (size_t)(D / 16) + (size_t)(d / 16)", "srow * (size_t)(D / 16) + (size_t)(d / 32)",
       None)]),
    ("nvfp4_scales_read_token_major",
     [("const size_t srow = (block * (size_t)H_kv + (size_t)hk) * (size_t)block_size + offset;",
       "const size_t srow = (block * (size_t)block_size + offset) * (size_t)H_kv + (size_t)hk;",
       None)]),
    ("block_scale_rows_token_major",
     [("return ((size_t)block * (size_t)H_kv + (size_t)h) * (size_t)block_size + (size_t)offset;",
       "return ((size_t)block * (size_t)block_size + (size_t)offset) * (size_t)H_kv + (size_t)h;",
       None)]),
    ("block_scale_pack_swaps_k_and_v",
     [("memcpy(dst, (const char*)k_scales + src, (size_t)row_bytes);",
       "memcpy(dst, (const char*)v_scales + src, (size_t)row_bytes);", None)]),
    ("nvfp4_block_scale_dropped",
     [("return orc_e2m1(code) * orc_e4m3(sc);", "(void)sc; return orc_e2m1(code);", None)]),
    ("kv_scale_dropped",
     [("off, block_size, hk, d, H_kv, D, kv_dtype) * k_scale;",
       "off, block_size, hk, d, H_kv, D, kv_dtype);", None)]),
]


def _mutate(text, edits):
    for old, new, occ in edits:
        n = text.count(old)
        assert n >= 1, f"mutation anchor not found: {old!r}"
        if occ is None:
            text = text.replace(old, new)
        else:
            parts = text.split(old)
            text = old.join(parts[: occ + 1]) + new + old.join(parts[occ + 1:])
    return text


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, edits):
    src = open(SRC).read()
    mutated = _mutate(src, edits)
    assert mutated != src
    msrc = tmp_path / f"oracle_{name}.c"
    msrc.write_text(mutated)
    lib_path = orc.build(force=True, src=str(msrc), out=str(tmp_path / f"lib_{name}.so"))
    lib = orc.load(lib_path)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches the mutant {name}"
