"""The oracle's pins catch plausible mistakes.

Each case copies oracle/sift_oracle.c, plants one mistake by a text substitution,
builds the copy with gcc in a temporary directory and runs the unchanged pins of
tests/test_oracle_pins.py and tests/test_oracle_ragged_pins.py against it
(SIFT_ORACLE_LIB points the oracle at the copy).  Every mutant must make at least
one pin fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "sift_oracle.c")

# (name, text to replace, replacement) -- each a mistake someone could plausibly make
MUTANTS = [
    ("la_transposed",
     "return la_bit(s, p, g, layer, h, (int)((t - d0) / B), (int)((u - d0) / B));",
     "return la_bit(s, p, g, layer, h, (int)((u - d0) / B), (int)((t - d0) / B));"),
    ("ca_inside_own_doc",
     "return la_bit(s, p, g, layer, h, (int)((t - d0) / B), (int)((u - d0) / B));",
     "return ca_bit(s, p, g, layer, h, (int)((u - d0) / B));"),
    ("no_diagonal", "if ((t - d0) / B == (u - d0) / B) return 1;", "if (0) return 1;"),
    ("suffix_not_dense", "if (g < 0) return 1;\n    int64_t B", "if (g < 0) return 0;\n    int64_t B"),
    ("msb_first_bits", "uint64_t word = s->la_words[base + (int64_t)i * W + j / 64];\n    return (int)((word >> (j % 64)) & 1u);",
     "uint64_t word = s->la_words[base + (int64_t)i * W + j / 64];\n    return (int)((word >> (63 - j % 64)) & 1u);"),
    ("block_order_head_major", "int64_t base = s->la_off[g] + ((int64_t)layer * s->num_kv_heads + h) * T * W;",
     "int64_t base = s->la_off[g] + ((int64_t)h * 2 + layer) * T * W;"),
    ("decode_own_ca", "for (int gp = doc_cu[p]; gp < g; ++gp) {", "for (int gp = doc_cu[p]; gp <= g; ++gp) {"),
    ("decode_suffix_short", "for (int64_t j = cu_seqlens[p] / tile; j <= i; ++j) EMIT(j);",
     "for (int64_t j = cu_seqlens[p] / tile; j < i; ++j) EMIT(j);"),
    ("decode_drops_ca_prefix", "int64_t t0 = doc_begin(&s, p, g) / tile;\n                    int il = (int)(i - t0);",
     "int64_t t0 = doc_begin(&s, p, g) / tile;\n                    int il = (int)(i - t0) - 0 * (n = 0);"),
    ("causal_excludes_self", "if (p < 0 || u < s->cu_seqlens[p] || u > t) return 0;",
     "if (p < 0 || u < s->cu_seqlens[p] || u >= t) return 0;"),
    ("scale_dropped", "sc[u - u0] = scale * acc;", "sc[u - u0] = acc;"),
    ("lse_without_log", "out_lse[r] = m + log(l);", "out_lse[r] = m + l;"),
    ("no_normalisation", "for (int c = 0; c < d; ++c) o[c] /= l;", "for (int c = 0; c < d; ++c) o[c] /= 1.0;"),
    ("wrong_kv_head_for_v", "const uint16_t *vr = v + (u * num_kv_heads + h) * d;",
     "const uint16_t *vr = v + (u * num_kv_heads + (qh % num_kv_heads)) * d;"),
    ("prompt_boundary_ignored", "if (p < 0 || u < s->cu_seqlens[p] || u > t) return 0;",
     "if (p < 0 || u < 0 || u > t) return 0;"),
    # documents of any length and a page size of its own
    ("ca_page_is_tile", "return ca_bit(s, p, gu, layer, h, (int)((u - d0u) / s->page));",
     "return ca_bit(s, p, gu, layer, h, (int)((u - d0u) / s->tile));"),
    ("tiles_rounded_down", "return (int)((n + s->tile - 1) / s->tile);",
     "return (int)(n / s->tile);"),
    ("pages_rounded_down", "return (int)((n + s->page - 1) / s->page);",
     "return (int)(n / s->page);"),
    ("ragged_mask_first_page_only",
     "if (ca_bit(&s, p, gp, l, h, (int)((y - ds + (int64_t)k * pin) / page)))",
     "if (ca_bit(&s, p, gp, l, h, (int)((y - ds) / page)))"),
    ("ragged_full_length_tiles", "int64_t len = de - y < tile ? de - y : tile;",
     "int64_t len = tile;"),
    ("gather_takes_partial_pages", "for (int j = 0; (int64_t)(j + 1) * page <= de - ds; ++j)",
     "for (int j = 0; (int64_t)j * page < de - ds; ++j)"),
    ("gather_groups_always_full", "EMIT(rel + k0, (uint32_t)(in_group * page) | 1u << 9 | full << 16);",
     "EMIT(rel + k0, (uint32_t)(nbits * page) | 1u << 9 | full << 16);"),
    ("ragged_diagonal_not_causal",
     "EMIT(x, (uint32_t)(end - x < tile ? end - x : tile) | 1u << 8 | full << 16);",
     "EMIT(x, (uint32_t)(end - x < tile ? end - x : tile) | full << 16);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation site of {name} not found"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new, 1))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(mutant), "-o",
                    str(lib), "-lm"], check=True)
    env = dict(os.environ, SIFT_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_ragged_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
