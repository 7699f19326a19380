"""Writes the small text fixtures in tests/golden/ from closed forms.

Nothing here runs the oracle or the CUDA library: every expected value is
worked out with exact rational arithmetic (fractions.Fraction) from the
definitions the fixtures cite.  Run ``python tests/golden/make_golden.py`` to
regenerate; the files are committed.
"""
from __future__ import annotations

import os
import struct
from fractions import Fraction

HERE = os.path.dirname(os.path.abspath(__file__))


def f16_bits_exact(x: Fraction) -> int:
    """fp16 bit pattern of a value that fp16 represents exactly (checked)."""
    bits = struct.unpack("<H", struct.pack("<e", float(x)))[0]
    back = Fraction(struct.unpack("<e", struct.pack("<H", bits))[0])
    assert back == x, (x, back)
    return bits


def write_q8_0():
    # One q8_0 block: fp16 scale d = 0.5 (0x3800), 32 int8 codes.
    d = Fraction(1, 2)
    codes = [-127, -64, -1, 0, 1, 2, 63, 127] + [i - 12 for i in range(24)]
    raw = struct.pack("<H", f16_bits_exact(d)) + struct.pack("<32b", *codes)
    vals = [d * c for c in codes]
    with open(os.path.join(HERE, "q8_0_block.txt"), "w") as f:
        f.write("# one q8_0 block (34 bytes): fp16 scale, then 32 int8 codes; value_i = d * q_i\n")
        f.write("# source: Rolling KV patch (opencoti 0070) q8_0 block of 32 values; ggml block layout reading\n")
        f.write("bytes " + raw.hex() + "\n")
        f.write("values " + " ".join(str(v) for v in vals) + "\n")


def write_q4_0():
    # One q4_0 block: fp16 scale d = 0.25 (0x3400); byte j holds value j in its
    # low nibble and value j+16 in its high nibble; value = d * (u - 8).
    d = Fraction(1, 4)
    u = [(3 * i + 1) % 16 for i in range(16)] + [(7 * i + 2) % 16 for i in range(16)]
    qs = bytes((u[j] & 0xF) | ((u[j + 16] & 0xF) << 4) for j in range(16))
    raw = struct.pack("<H", f16_bits_exact(d)) + qs
    vals = [d * (x - 8) for x in u]
    with open(os.path.join(HERE, "q4_0_block.txt"), "w") as f:
        f.write("# one q4_0 block (18 bytes): fp16 scale, 16 bytes of nibbles; value = d * (u - 8)\n")
        f.write("# byte j: low nibble -> value j, high nibble -> value j+16 (ggml block layout reading)\n")
        f.write("bytes " + raw.hex() + "\n")
        f.write("values " + " ".join(str(v) for v in vals) + "\n")


def write_attention_pow2():
    # q = e_0, k_j[0] = j and scale = ln 2, so s_j = j ln 2 and the softmax
    # weights are 2^j / sum_i 2^i: O and lse follow exactly.
    V = [[1, 2, 3, 4], [0, -1, 5, 2], [3, 3, 3, 3], [-2, 1, 0, 8]]
    K = [[j, 7, -3, 5] for j in range(4)]
    w = [Fraction(2) ** j for j in range(4)]
    Z = sum(w)
    O = [sum(w[j] * V[j][d] for j in range(4)) / Z for d in range(4)]
    with open(os.path.join(HERE, "attention_pow2.txt"), "w") as f:
        f.write("# softmax attention with scores j*ln2 (q=e_0, k_j[0]=j, scale=ln 2): weights 2^j/15\n")
        f.write("# source: definition of the per-tile output and its log-sum-exp (Rolling KV patch,\n")
        f.write("# streaming_lse_kernel and the tile combine); lse = ln(sum_j 2^j) = ln 15\n")
        f.write("q 1 0 0 0\n")
        for j in range(4):
            f.write("k " + " ".join(str(x) for x in K[j]) + "\n")
        for j in range(4):
            f.write("v " + " ".join(str(x) for x in V[j]) + "\n")
        f.write("o " + " ".join(str(x) for x in O) + "\n")
        f.write("lse_exp " + str(Z) + "\n")


if __name__ == "__main__":
    write_q8_0()
    write_q4_0()
    write_attention_pow2()
