"""Pins of the oracle's append and quantise-on-append functions.

* fp32 -> binary16 rounding against numpy's own float16 conversion: every
  binary16 value, every midpoint between neighbours (ties to even) and its two
  fp32 neighbours, and random fp32 patterns across and beyond the range;
* q8_0 / q4_0 blocks built from an exact scale and exact codes, whose bytes
  follow from the block layout alone, and which decode (through the separately
  pinned dequantiser) back to the input;
* the nearest-code property of every code of random blocks (several value
  distributions), the scale against numpy's fp32 division and float16 cast,
  and the largest code at the block's largest magnitude;
* write routing: which region and row each position lands in, the head
  segment inside a row, untouched padding, skipped and out-of-range positions;
* the paged host-copy layout against numpy indexing of [block][Hk][rows][D].
"""
import numpy as np
import pytest

import oracle

F16, Q8_0, Q4_0 = oracle.F16, oracle.Q8_0, oracle.Q4_0


def _to_half_bits(x):
    return oracle.quantize(F16, np.asarray(x, np.float32)).view(np.uint16)


def _numpy_half_bits(x):
    with np.errstate(over="ignore"):
        return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def test_half_rounding_every_value_and_midpoint():
    bits = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16)
    finite = np.isfinite(vals)
    exact = vals[finite].astype(np.float32)
    assert np.array_equal(_to_half_bits(exact), _numpy_half_bits(exact))
    # midpoints between consecutive non-negative halves (exact in fp32), and
    # the fp32 values right next to them
    pos = np.sort(vals[finite & (bits < 0x8000)].astype(np.float64))
    mid = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.all(mid.astype(np.float64) == (pos[:-1] + pos[1:]) / 2)
    near = np.concatenate([mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(np.inf))])
    for s in (1.0, -1.0):
        v = (s * near).astype(np.float32)
        assert np.array_equal(_to_half_bits(v), _numpy_half_bits(v))
    # the halfway point to 2^16 and beyond overflow to infinity
    big = np.array([65519.996, 65520.0, 65536.0, 1e30, -65520.0], np.float32)
    assert np.array_equal(_to_half_bits(big), _numpy_half_bits(big))


def test_half_rounding_random_patterns():
    rng = np.random.Generator(np.random.PCG64(2024))
    raw = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # steer half of them into the binary16 range and below it
    exp = rng.integers(127 - 30, 127 + 17, size=raw.size).astype(np.uint32)
    steer = (raw & np.uint32(0x807FFFFF)) | (exp << np.uint32(23))
    x = np.where(np.arange(raw.size) % 2 == 0, steer, raw).view(np.float32)
    x = x[np.isfinite(x)]
    assert np.array_equal(_to_half_bits(x), _numpy_half_bits(x))


def _q8_bytes(scale_bits, codes):
    return np.concatenate([np.array([scale_bits & 0xFF, scale_bits >> 8], np.uint8),
                           np.asarray(codes, np.int8).view(np.uint8)])


def test_q8_exact_block_bytes_and_round_trip():
    codes = np.array([127, -127, 0, 1, -1, 2, -2, 64, -64, 100, -100, 3, 5, 7, 11, 13,
                      17, -19, 23, -29, 31, -37, 41, -43, 47, -53, 59, -61, 67, -71, 73, -79], np.int32)
    d = 0.5                                   # binary16 0x3800
    x = (d * codes).astype(np.float32)
    got = oracle.quantize(Q8_0, x)
    assert np.array_equal(got, _q8_bytes(0x3800, codes))
    assert np.array_equal(oracle.dequant(Q8_0, got, 32), x.astype(np.float64))
    # sign flip of the whole block flips every code, keeps the scale
    got_neg = oracle.quantize(Q8_0, -x)
    assert np.array_equal(got_neg, _q8_bytes(0x3800, -codes))


def test_q4_exact_block_bytes_and_round_trip():
    u = np.array([15, 1, 8, 9, 7, 10, 6, 11, 5, 12, 4, 13, 3, 14, 2, 8,
                  1, 15, 2, 14, 3, 13, 4, 12, 5, 11, 6, 10, 7, 9, 8, 15], np.int32)
    d = 0.25                                  # binary16 0x3400
    x = (d * (u - 8)).astype(np.float32)
    got = oracle.quantize(Q4_0, x)
    want = np.concatenate([[0x00, 0x34], [u[j] | (u[j + 16] << 4) for j in range(16)]]).astype(np.uint8)
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.dequant(Q4_0, got, 32), x.astype(np.float64))


def test_zero_block():
    z = np.zeros(32, np.float32)
    assert np.array_equal(oracle.quantize(Q8_0, z), np.zeros(34, np.uint8))
    assert np.array_equal(oracle.quantize(Q4_0, z), np.array([0, 0] + [0x88] * 16, np.uint8))


def _blocks(rng, n):
    return [rng.standard_normal((n, 32)), rng.uniform(-1e-3, 1e-3, (n, 32)),
            rng.standard_t(2, (n, 32)) * 50, rng.standard_normal((n, 32)) * np.exp(rng.uniform(-20, 8, (n, 1))),
            np.round(rng.standard_normal((n, 32)) * 8) / 4]


@pytest.mark.parametrize("type_", [Q8_0, Q4_0])
def test_nearest_code_property(type_):
    rng = np.random.Generator(np.random.PCG64(77 + type_))
    qmax, blk = (127, 34) if type_ == Q8_0 else (7, 18)
    for x in _blocks(rng, 400):
        x = x.astype(np.float32)
        raw = oracle.quantize(type_, x.ravel()).reshape(-1, blk)
        d_bits = raw[:, 0].astype(np.uint16) | (raw[:, 1].astype(np.uint16) << 8)
        amax = np.abs(x).max(axis=1)
        want_d = (amax / np.float32(qmax)).astype(np.float32).astype(np.float16)
        assert np.array_equal(d_bits, want_d.view(np.uint16))
        d = want_d.astype(np.float64)[:, None]
        if type_ == Q8_0:
            q = raw[:, 2:].view(np.int8).astype(np.int64)
        else:
            lo, hi = raw[:, 2:] & 0xF, raw[:, 2:] >> 4
            q = np.concatenate([lo, hi], axis=1).astype(np.int64) - 8
        xd = x.astype(np.float64)
        live = d[:, 0] > 0
        assert np.all(q[~live] == 0)
        qlo = -qmax if type_ == Q8_0 else -8            # q4_0 codes u - 8 span [-8, 7]
        assert np.all(q <= qmax) and np.all(q >= qlo)
        xl, dl, ql = xd[live], d[live], q[live]
        ratio = xl / dl
        # beyond the end codes' half-intervals the code is the clamped end
        tol = 2.0 ** -20 * qmax
        hi_out, lo_out = ratio > qmax + 0.5 + tol, ratio < qlo - 0.5 - tol
        out = hi_out | lo_out
        assert np.all(ql[hi_out] == qmax) and np.all(ql[lo_out] == qlo)
        # everywhere else the code is a nearest one: no integer is strictly
        # closer, up to the fp32 rounding of x / d (an ulp of the quotient)
        err = np.abs(xl - dl * ql)
        slack = dl * (np.abs(ql) + 1) * 2.0 ** -22
        assert np.all((err <= dl / 2 + slack) | out)
        # with a normal fp16 scale (relative error <= 2^-11) the largest
        # magnitude takes the extreme code
        normal = live & (d[:, 0] >= 2.0 ** -14)
        idx = np.abs(x).argmax(axis=1)
        top = np.abs(q[np.arange(len(q)), idx])
        assert np.all(top[normal] == qmax)


def test_routing_two_regions():
    rng = np.random.Generator(np.random.PCG64(5))
    Hk, D, n0, n1 = 2, 64, 5, 7
    for type_ in (F16, Q8_0, Q4_0):
        seg = oracle.segment_bytes(type_, D)
        row_bytes = Hk * seg + 6                       # 6 padding bytes per row
        r0 = np.full(n0 * row_bytes, 0xAB, np.uint8)
        r1 = np.full(n1 * row_bytes, 0xCD, np.uint8)
        pos = np.array([0, 4, 5, 11, -1, 12, 3, 900], np.int32)
        x = (np.round(rng.standard_normal((pos.size, Hk, D)) * 4) / 8).astype(np.float32)
        bad = oracle.kv_append(type_, x, pos, r0, n0, r1, n1, row_bytes)
        assert bad == 2
        rows0 = r0.reshape(n0, row_bytes)
        rows1 = r1.reshape(n1, row_bytes)
        written = {0: (rows0, 0), 4: (rows0, 4), 5: (rows1, 0), 11: (rows1, 6), 3: (rows0, 3)}
        for i, p in enumerate(pos):
            if p not in written:
                continue
            rows, r = written[p]
            for k in range(Hk):
                segment = rows[r, k * seg:(k + 1) * seg]
                assert np.array_equal(segment, oracle.quantize(type_, x[i, k]))
                if type_ == F16:                       # values on a 1/8 grid are exact in fp16
                    assert np.array_equal(oracle.dequant(type_, segment, D), x[i, k].astype(np.float64))
            assert np.all(rows[r, Hk * seg:] == rows[r, -1]) and rows[r, -1] in (0xAB, 0xCD)
        for r in (1, 2):
            assert np.all(rows0[r] == 0xAB)
        for r in (1, 2, 3, 4, 5):
            assert np.all(rows1[r] == 0xCD)


def test_paged_host_layout():
    rng = np.random.Generator(np.random.PCG64(6))
    Hk, D, br, nb = 3, 64, 8, 4
    host = np.zeros((nb, Hk, br, D), np.uint16)
    pos = np.array([0, 7, 8, 17, 31, -3, 32, 40], np.int32)
    x = rng.standard_normal((pos.size, Hk, D)).astype(np.float32)
    bad = oracle.paged_append(x, pos, host, block_rows=br, n_blocks=nb)
    assert bad == 2
    want = np.zeros_like(host)
    for i, p in enumerate(pos):
        if 0 <= p < nb * br:
            want[p // br, :, p % br, :] = _numpy_half_bits(x[i])
    assert np.array_equal(host, want)
