"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of oracle/splitkv_oracle.c (on the CPU),
builds it, and runs the pin suites (tests/test_oracle_pins.py and
tests/test_oracle_append_pins.py) against that build; the suite must fail.  A mutant that survived would mean a part of the
oracle is not pinned by anything but itself."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "splitkv_oracle.c")

MUTANTS = [
    ("half_bias", "ldexp((double)(1024 + m), e - 25)", "ldexp((double)(1024 + m), e - 24)"),
    ("half_subnormal", "ldexp((double)m, -24)", "ldexp((double)m, -25)"),
    ("q8_scale_dropped", "out[32 * b + i] = d * (double)(int8_t)blk[2 + i];",
     "out[32 * b + i] = (double)(int8_t)blk[2 + i];"),
    ("q8_unsigned", "d * (double)(int8_t)blk[2 + i]", "d * (double)(uint8_t)blk[2 + i]"),
    ("q4_nibbles_swapped", "out[32 * b + j] = d * (double)(lo - 8);", "out[32 * b + j] = d * (double)(hi - 8);"),
    ("q4_no_offset", "out[32 * b + j + 16] = d * (double)(hi - 8);", "out[32 * b + j + 16] = d * (double)(hi);"),
    ("gqa_modulo", "const int k = h / G;", "const int k = h % Hk;"),
    ("segment_offset", "return src->base + row * src->row_bytes + (int64_t)head * seg;",
     "return src->base + row * src->row_bytes;"),
    ("paged_order", "return src->base + ((blk * Hk + head) * src->page_rows + in_blk) * seg;",
     "return src->base + ((head * Hk + blk) * src->page_rows + in_blk) * seg;"),
    ("softmax_sign", "const double w = exp(sc[j] - M);", "const double w = exp(M - sc[j]);"),
    ("scale_dropped", "double sj = scale * dot;", "double sj = dot;"),
    ("mask_sign", "sj += orc_half_to_double(mask[st * n_keys + j]);",
     "sj -= orc_half_to_double(mask[st * n_keys + j]);"),
    ("causal_off_by_one", "key_pos0 + j > (int64_t)q_pos[st]", "key_pos0 + j >= (int64_t)q_pos[st]"),
    ("padding_clamped_to_row0", "const int64_t row = kv_rows ? (int64_t)kv_rows[list * n_keys + j] : j;",
     "const int64_t row = kv_rows ? (kv_rows[list * n_keys + j] < 0 ? 0 : (int64_t)kv_rows[list * n_keys + j]) : j;"),
    ("lse_without_max", "out_lse[r] = M + log(Z);", "out_lse[r] = log(Z);"),
    ("not_normalised", "for (int d = 0; d < D; ++d) o[d] = acc[d] / Z;", "for (int d = 0; d < D; ++d) o[d] = acc[d];"),
    ("combine_unweighted", "const double w = exp(l - M);", "const double w = 1.0;"),
    ("combine_lse", "lse[r] = M + log(W);", "lse[r] = log(W);"),
    ("half_ties_away", "double f = nearbyint(ldexp(a, 10 - e));", "double f = floor(ldexp(a, 10 - e) + 0.5);"),
    ("half_truncates", "double f = nearbyint(ldexp(a, 10 - e));", "double f = floor(ldexp(a, 10 - e));"),
    ("half_subnormal_rounding", "const double f = nearbyint(ldexp(a, 24));", "const double f = floor(ldexp(a, 24));"),
    ("q8_scale_128", "const float qmax = type == ORC_Q8_0 ? 127.0f : 7.0f;",
     "const float qmax = type == ORC_Q8_0 ? 128.0f : 7.0f;"),
    ("q4_scale_8", "const float qmax = type == ORC_Q8_0 ? 127.0f : 7.0f;",
     "const float qmax = type == ORC_Q8_0 ? 127.0f : 8.0f;"),
    ("codes_truncated", "code[i] = d > 0.0f ? (int)rintf(x[i] / d) : 0;", "code[i] = d > 0.0f ? (int)(x[i] / d) : 0;"),
    ("q4_append_nibbles", "blk[2 + j] = (uint8_t)(lo | (hi << 4));", "blk[2 + j] = (uint8_t)(hi | (lo << 4));"),
    ("append_input_transposed", "encode_segment(type, x + (i * Hk + k) * D, D, row + k * seg);",
     "encode_segment(type, x + (k * n + i) * D, D, row + k * seg);"),
    ("append_region_split", "uint8_t *row = p < n_rows0 ? (uint8_t *)dst0 + p * row_bytes",
     "uint8_t *row = p < n_rows0 - 1 ? (uint8_t *)dst0 + p * row_bytes"),
    ("paged_append_order", "uint16_t *dst = host + (((blk * Hk + k) * block_rows) + in_blk) * D;",
     "uint16_t *dst = host + (((k * n_blocks + blk) * block_rows) + in_blk) * D;"),
]

PIN_FILES = ["test_oracle_pins.py", "test_oracle_append_pins.py"]


def _build(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} no longer in the oracle"
    mut = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mut)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(c), "-o", str(so), "-lm"],
                   check=True, capture_output=True)
    return so


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    so = _build(tmp_path, name, old, new)
    env = dict(os.environ, SPLITKV_ORACLE_LIB=str(so), OMP_NUM_THREADS="2")
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          *[os.path.join(ROOT, "tests", f) for f in PIN_FILES]],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode != 0, f"mutant {name} survived the oracle pins:\n{res.stdout[-2000:]}"
