"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU, never
in the GPU path), builds it, points the oracle wrapper at it through
KIVI_ORACLE_LIB, and runs the oracle pin tests in a subprocess: at least one pin
must fail. The unmodified source must pass the same tests.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "kivi_oracle.c")
PINS = ["tests/test_oracle_codec.py", "tests/test_oracle_cache.py", "tests/test_oracle_multi.py"]

MUTANTS = {
    # packing: bits of a byte filled from the top instead of the bottom
    "bit_order": ("int shift = (d % per_byte) * bits;", "int shift = (per_byte - 1 - d % per_byte) * bits;"),
    # rounding: half away from zero instead of half to even
    "round_half_away": ("float r = rintf(t);", "float r = roundf(t);"),
    # scale: divide by 2^bits instead of 2^bits - 1
    "scale_divisor": ("float s32 = range / (float)qmax;", "float s32 = range / (float)(qmax + 1);"),
    # dequantization drops the key zero point
    "dropped_zero": ("+ (double)orc_f16_to_f32(s->k_zero[mk]);", "+ 0.0;"),
    # GQA: query head mapped to kv head hq mod Hkv instead of hq / g
    "gqa_mapping": ("int h = hq / g;", "int h = hq % H;"),
    # softmax scale not applied
    "missing_scale": ("score[p] = scale * acc;", "score[p] = acc;"),
    # flush one token early
    "flush_early": ("if (p + 1 - n_packed == R + G) {", "if (p + 1 - n_packed == R + G - 1) {"),
    # residual ring indexed modulo R instead of R + G
    "ring_modulus": ("const int ring = R + G;\n    int64_t L = *kv_len;", "const int ring = R;\n    int64_t L = *kv_len;"),
    # flushed values coded at the key width
    "value_width": ("const int kq = (1 << kb) - 1, vq = (1 << vb) - 1, ring = R + G;",
                    "const int kq = (1 << kb) - 1, vq = (1 << kb) - 1, ring = R + G;"),
    # dequantized keys read at the value width
    "key_read_width": ("k[d] = (double)get_code(kr, d, kb)", "k[d] = (double)get_code(kr, d, vb)"),
    # multi-query: a query does not see its own token
    "causal_excludes_self": ("attend_prefix(cfg, s, L, L - n_query + 1 + i,", "attend_prefix(cfg, s, L, L - n_query + i,"),
    # multi-query: no causal mask
    "no_causal_mask": ("attend_prefix(cfg, s, L, L - n_query + 1 + i,", "attend_prefix(cfg, s, L, L + 0 * i,"),
    # value metadata indexed with 32-channel groups whatever G is
    "value_group_fixed": ("int64_t mv = ((int64_t)h * cap + p) * (D / G) + d / G;",
                          "int64_t mv = ((int64_t)h * cap + p) * (D / G) + d / 32 % (D / G);"),
}


def _run_pins(lib_path):
    env = dict(os.environ, KIVI_ORACLE_LIB=lib_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                       cwd=os.path.dirname(HERE), env=env, capture_output=True, text=True, timeout=600)
    return r.returncode


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path, oracle_lib):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = tmp_path / f"oracle_{name}.c"
    mutant.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutant), str(tmp_path / f"liboracle_{name}.so"))
    assert _run_pins(lib) != 0, f"no pin failed for the planted mistake '{name}'"


def test_unmodified_oracle_passes_the_same_pins(tmp_path, oracle_lib):
    lib = oracle.compile_source(SRC, str(tmp_path / "liboracle_clean.so"))
    assert _run_pins(lib) == 0
