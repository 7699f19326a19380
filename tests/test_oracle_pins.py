"""Pins of the fp64 oracle against what the definitions fix on their own.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, the wrong nibble or head segment)
fails at least one of them:

* binary16 decoding against numpy's own float16 conversion, all 65536 patterns;
* q8_0 / q4_0 blocks against hand-worked fixtures (tests/golden/);
* softmax attention with scores j*ln2, where the weights are exactly 2^j / sum
  (exact rational expected values), with every subset of 8 keys masked;
* q = 0 gives the mean of the visible values and lse = ln(count), which pins
  the GQA head mapping, padding, causal visibility and masks;
* structural identities: window+tail = one region, identity row list = dense,
  -1 padding is a no-op, paged layout = cell-major layout, quantised storage of
  exactly representable values = fp16 storage, a constant mask shifts lse only;
* split + log-sum-exp combine = unsplit for 1..33 parts and tile sizes 256,
  512, 768, 1024; a -inf part is a no-op; the combine is order-invariant.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from split_kv_flash_attn_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *rest = line.split()
            out.setdefault(key, []).append(rest)
    return out


# ------------------------------------------------------------------ decoding

def test_half_decode_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle_mod.half_to_double(bits)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_half_decode_landmarks(oracle_mod):
    vals = oracle_mod.half_to_double([0x3C00, 0xC000, 0x0001, 0x7BFF, 0x7C00, 0x8000, 0x0400])
    assert list(vals[:4]) == [1.0, -2.0, 2.0 ** -24, 65504.0]
    assert vals[4] == math.inf and vals[5] == 0.0 and math.copysign(1, vals[5]) < 0
    assert vals[6] == 2.0 ** -14


@pytest.mark.parametrize("name,type_", [("q8_0_block.txt", oracle.Q8_0), ("q4_0_block.txt", oracle.Q4_0)])
def test_quant_block_golden(oracle_mod, name, type_):
    fx = _read_fixture(name)
    raw = np.frombuffer(bytes.fromhex(fx["bytes"][0][0]), dtype=np.uint8)
    want = [float(Fraction(x)) for x in fx["values"][0]]
    got = oracle_mod.dequant(type_, raw, 32)
    assert list(got) == want


def test_quant_extremes(oracle_mod):
    # q8: codes +-127 at the largest and smallest drawn scales; q4: u=0 -> -8d, u=15 -> +7d
    for d in (np.float16(0.005), np.float16(0.02)):
        blk = np.zeros(34, np.uint8)
        blk[0:2] = np.array([d], np.float16).view(np.uint8)
        blk[2] = np.uint8(127)
        blk[3] = np.int8(-127).view(np.uint8)
        got = oracle_mod.dequant(oracle.Q8_0, blk, 32)
        assert got[0] == 127 * float(d) and got[1] == -127 * float(d) and got[2] == 0.0
        b4 = np.zeros(18, np.uint8)
        b4[0:2] = np.array([d], np.float16).view(np.uint8)
        b4[2] = 0xF0  # value 0: u=0, value 16: u=15
        got4 = oracle_mod.dequant(oracle.Q4_0, b4, 32)
        assert got4[0] == -8 * float(d) and got4[16] == 7 * float(d) and got4[1] == -8 * float(d)


def test_quant_segment_offsets(oracle_mod):
    assert oracle_mod.segment_bytes(oracle.F16, 128) == 256
    assert oracle_mod.segment_bytes(oracle.Q8_0, 128) == 136
    assert oracle_mod.segment_bytes(oracle.Q4_0, 128) == 72


# ------------------------------------------------------------------ attention

def _f16_rows(arr):
    a = np.ascontiguousarray(np.asarray(arr, dtype=np.float16))
    return a.view(np.uint8).reshape(a.shape[0], -1)


def test_attention_golden_pow2(oracle_mod):
    fx = _read_fixture("attention_pow2.txt")
    q = np.array([[[[float(x) for x in fx["q"][0]]]]], np.float16)
    K = _f16_rows([[float(x) for x in r] for r in fx["k"]])
    V = _f16_rows([[float(x) for x in r] for r in fx["v"]])
    o, lse = oracle_mod.attention(q, D=4, H=1, Hk=1, scale=math.log(2), k0=K, v0=V, n_rows0=4,
                                  k_row_bytes0=8, v_row_bytes0=8, n_keys=4)
    want = [float(Fraction(x)) for x in fx["o"][0]]
    assert np.allclose(o.ravel(), want, rtol=1e-13, atol=1e-13)
    assert abs(lse.ravel()[0] - math.log(float(Fraction(fx["lse_exp"][0][0])))) < 1e-13


def _pow2_case(n, D=16, H=2, Hk=1, seed=0):
    rng = np.random.default_rng(seed)
    q = np.zeros((1, 1, H, D), np.float16)
    q[..., 0] = 1.0
    K = rng.standard_normal((n, Hk, D)).astype(np.float16)
    K[:, :, 0] = np.arange(n)[:, None]
    V = rng.integers(-8, 9, size=(n, Hk, D)).astype(np.float16)
    return q, K, V


def test_attention_pow2_all_masks(oracle_mod):
    n, D = 8, 16
    q, K, V = _pow2_case(n, D)
    Kr, Vr = _f16_rows(K.reshape(n, -1)), _f16_rows(V.reshape(n, -1))
    for bits in range(1 << n):
        mask = np.array([0.0 if (bits >> j) & 1 else -np.inf for j in range(n)], np.float16)
        o, lse = oracle_mod.attention(q, D=D, H=2, Hk=1, scale=math.log(2), k0=Kr, v0=Vr, n_rows0=n,
                                      k_row_bytes0=2 * D, v_row_bytes0=2 * D, n_keys=n,
                                      mask=mask.reshape(1, 1, n))
        vis = [j for j in range(n) if (bits >> j) & 1]
        if not vis:
            assert np.all(o == 0.0) and np.all(lse == -np.inf)
            continue
        Z = sum(Fraction(2) ** j for j in vis)
        for d in range(D):
            want = float(sum(Fraction(2) ** j * Fraction(float(V[j, 0, d])) for j in vis) / Z)
            assert abs(o[0, 0, 0, d] - want) <= 1e-12 * max(1.0, abs(want))
            assert o[0, 0, 1, d] == o[0, 0, 0, d]
        assert abs(lse[0, 0, 0] - math.log(float(Z))) < 1e-12


def test_one_visible_row_returns_that_row(oracle_mod):
    n, D = 32, 64
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 4, D)).astype(np.float16)
    K = rng.standard_normal((n, D)).astype(np.float16)
    V = rng.standard_normal((n, D)).astype(np.float16)
    rows = np.full((1, n), -1, np.int32)
    rows[0, 0] = 17
    o, lse = oracle_mod.attention(q, D=D, H=4, Hk=1, scale=0.125, k0=_f16_rows(K), v0=_f16_rows(V),
                                  n_rows0=n, k_row_bytes0=2 * D, v_row_bytes0=2 * D,
                                  n_keys=n, kv_rows=rows)
    for h in range(4):
        assert np.array_equal(o[0, 0, h], V[17].astype(np.float64))
    # two visible copies of the same key: lse rises by exactly ln 2
    rows[0, 1] = 17
    o2, lse2 = oracle_mod.attention(q, D=D, H=4, Hk=1, scale=0.125, k0=_f16_rows(K), v0=_f16_rows(V),
                                    n_rows0=n, k_row_bytes0=2 * D, v_row_bytes0=2 * D,
                                    n_keys=n, kv_rows=rows)
    assert np.allclose(lse2 - lse, math.log(2), atol=1e-14)
    assert np.allclose(o2, o, atol=1e-15)


def test_identical_keys_mean_of_values(oracle_mod):
    n, D = 12, 32
    rng = np.random.default_rng(4)
    q = np.zeros((1, 1, 1, D), np.float16)
    q[0, 0, 0, 0] = 2.0
    K = np.tile(rng.standard_normal((1, D)).astype(np.float16), (n, 1))
    K[:, 0] = 0.75
    V = rng.integers(-20, 21, size=(n, D)).astype(np.float16)
    o, lse = oracle_mod.attention(q, D=D, H=1, Hk=1, scale=0.5, k0=_f16_rows(K), v0=_f16_rows(V),
                                  n_rows0=n, k_row_bytes0=2 * D, v_row_bytes0=2 * D, n_keys=n)
    # score = 0.5 * 2 * 0.75 = 0.75 for every key
    want = [float(sum(Fraction(float(x)) for x in V[:, d]) / n) for d in range(D)]
    assert np.allclose(o[0, 0, 0], want, rtol=1e-14, atol=1e-14)
    assert abs(lse[0, 0, 0] - (0.75 + math.log(n))) < 1e-13


def test_zero_query_gqa_mapping_and_padding(oracle_mod):
    # q = 0: every visible key has weight 1/count; KV head k = h // G
    S, H, Hk, D, n = 2, 8, 2, 32, 24
    rng = np.random.default_rng(5)
    q = np.zeros((S, 1, H, D), np.float16)
    K = rng.standard_normal((n, Hk, D)).astype(np.float16)
    V = rng.integers(-50, 51, size=(n, Hk, D)).astype(np.float16)
    rows = np.stack([np.r_[np.arange(0, 10), -np.ones(6, int), np.arange(15, 23)],
                     np.r_[np.arange(3, 7), -np.ones(20, int)]]).astype(np.int32)
    o, lse = oracle_mod.attention(q, D=D, H=H, Hk=Hk, scale=0.3, k0=_f16_rows(K.reshape(n, -1)),
                                  v0=_f16_rows(V.reshape(n, -1)), n_rows0=n,
                                  k_row_bytes0=2 * Hk * D, v_row_bytes0=2 * Hk * D,
                                  n_keys=rows.shape[1], kv_rows=rows)
    for s in range(S):
        vis = [r for r in rows[s] if r >= 0]
        for h in range(H):
            kh = h // (H // Hk)
            want = [float(sum(Fraction(float(V[r, kh, d])) for r in vis) / len(vis)) for d in range(D)]
            assert np.allclose(o[s, 0, h], want, rtol=1e-14, atol=1e-13)
            assert abs(lse[s, 0, h] - math.log(len(vis))) < 1e-13


def test_zero_query_causal_visibility(oracle_mod):
    nq, H, D, n = 5, 2, 16, 20
    rng = np.random.default_rng(6)
    q = np.zeros((1, nq, H, D), np.float16)
    K = rng.standard_normal((n, D)).astype(np.float16)
    V = rng.integers(-9, 10, size=(n, D)).astype(np.float16)
    q_pos = np.array([[0, 3, 7, 19, 25]], np.int32)
    o, lse = oracle_mod.attention(q, D=D, H=H, Hk=1, scale=1.0, k0=_f16_rows(K), v0=_f16_rows(V),
                                  n_rows0=n, k_row_bytes0=2 * D, v_row_bytes0=2 * D, n_keys=n,
                                  q_pos=q_pos, key_pos0=2)
    for t in range(nq):
        vis = [j for j in range(n) if 2 + j <= q_pos[0, t]]
        if not vis:
            assert np.all(o[0, t] == 0) and np.all(lse[0, t] == -np.inf)
            continue
        want = [float(sum(Fraction(float(V[j, d])) for j in vis) / len(vis)) for d in range(D)]
        assert np.allclose(o[0, t, 0], want, rtol=1e-14, atol=1e-13)
        assert abs(lse[0, t, 1] - math.log(len(vis))) < 1e-13


def test_all_masked_and_all_padding(oracle_mod):
    D, n = 16, 8
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 1, 2, D)).astype(np.float16)
    K = _f16_rows(rng.standard_normal((n, D)))
    V = _f16_rows(rng.standard_normal((n, D)))
    o, lse = oracle_mod.attention(q, D=D, H=2, Hk=1, scale=0.25, k0=K, v0=V, n_rows0=n,
                                  k_row_bytes0=2 * D, v_row_bytes0=2 * D, n_keys=n,
                                  kv_rows=np.full((1, n), -1, np.int32))
    assert np.all(o == 0) and np.all(lse == -np.inf)
    o, lse = oracle_mod.attention(q, D=D, H=2, Hk=1, scale=0.25, k0=K, v0=V, n_rows0=n,
                                  k_row_bytes0=2 * D, v_row_bytes0=2 * D, n_keys=n,
                                  mask=np.full((1, 1, n), -np.inf, np.float16))
    assert np.all(o == 0) and np.all(lse == -np.inf)
    o, lse = oracle_mod.attention(q, D=D, H=2, Hk=1, scale=0.25, k0=K, v0=V, n_rows0=n,
                                  k_row_bytes0=2 * D, v_row_bytes0=2 * D, n_keys=0)
    assert np.all(o == 0) and np.all(lse == -np.inf)


def _rand_case(seed, n=300, H=8, Hk=2, D=64, nq=1, S=1):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((S, nq, H, D)).astype(np.float16)
    K = _f16_rows(rng.standard_normal((n, Hk * D)))
    V = _f16_rows(rng.standard_normal((n, Hk * D)))
    return q, K, V, dict(D=D, H=H, Hk=Hk, scale=1 / math.sqrt(D))


def test_constant_mask_shifts_lse_only(oracle_mod):
    q, K, V, kw = _rand_case(8)
    n = K.shape[0]
    rb = K.shape[1]
    base = oracle_mod.attention(q, **kw, k0=K, v0=V, n_rows0=n, k_row_bytes0=rb, v_row_bytes0=rb, n_keys=n)
    sh = oracle_mod.attention(q, **kw, k0=K, v0=V, n_rows0=n, k_row_bytes0=rb, v_row_bytes0=rb, n_keys=n,
                              mask=np.full((1, 1, n), -1.5, np.float16))
    assert np.allclose(sh[0], base[0], atol=1e-13)
    assert np.allclose(sh[1], base[1] - 1.5, atol=1e-12)


def test_window_tail_equals_one_region(oracle_mod):
    q, K, V, kw = _rand_case(9, n=300)
    rb = K.shape[1]
    whole = oracle_mod.attention(q, **kw, k0=K, v0=V, n_rows0=300, k_row_bytes0=rb, v_row_bytes0=rb, n_keys=300)
    for wc in (0, 1, 128, 299, 300):
        split = oracle_mod.attention(q, **kw, k0=K[:wc], v0=V[:wc], n_rows0=wc, k_row_bytes0=rb,
                                     v_row_bytes0=rb, k1=K[wc:], v1=V[wc:], n_rows1=300 - wc,
                                     k_row_bytes1=rb, v_row_bytes1=rb, n_keys=300)
        assert np.array_equal(split[0], whole[0]) and np.array_equal(split[1], whole[1])


def test_identity_rows_and_padding_are_noops(oracle_mod):
    q, K, V, kw = _rand_case(10, n=256)
    rb = K.shape[1]
    dense = oracle_mod.attention(q, **kw, k0=K, v0=V, n_rows0=256, k_row_bytes0=rb, v_row_bytes0=rb, n_keys=256)
    ident = np.arange(256, dtype=np.int32).reshape(1, -1)
    g = oracle_mod.attention(q, **kw, k0=K, v0=V, n_rows0=256, k_row_bytes0=rb, v_row_bytes0=rb,
                             n_keys=256, kv_rows=ident)
    assert np.array_equal(g[0], dense[0]) and np.array_equal(g[1], dense[1])
    padded = np.concatenate([ident, -np.ones((1, 256), np.int32)], axis=1)
    p = oracle_mod.attention(q, **kw, k0=K, v0=V, n_rows0=256, k_row_bytes0=rb, v_row_bytes0=rb,
                             n_keys=512, kv_rows=padded)
    assert np.array_equal(p[0], dense[0]) and np.array_equal(p[1], dense[1])
    # padding interleaved anywhere, and a permuted key order: same result up to rounding
    rng = np.random.default_rng(11)
    perm = rng.permutation(512)
    pr = oracle_mod.attention(q, **kw, k0=K, v0=V, n_rows0=256, k_row_bytes0=rb, v_row_bytes0=rb,
                              n_keys=512, kv_rows=padded[:, perm])
    assert np.allclose(pr[0], dense[0], atol=1e-13) and np.allclose(pr[1], dense[1], atol=1e-13)


def test_paged_layout_equals_cell_major(oracle_mod):
    Hk, D, br, nb = 2, 32, 8, 6
    rng = np.random.default_rng(12)
    Kp = rng.standard_normal((nb, Hk, br, D)).astype(np.float16)
    Vp = rng.standard_normal((nb, Hk, br, D)).astype(np.float16)
    Kc = Kp.transpose(0, 2, 1, 3).reshape(nb * br, Hk * D)
    Vc = Vp.transpose(0, 2, 1, 3).reshape(nb * br, Hk * D)
    q = rng.standard_normal((2, 1, 4, D)).astype(np.float16)
    rows = np.stack([rng.permutation(nb * br)[:20] for _ in range(2 * Hk)]).reshape(2, Hk, 20).astype(np.int32)
    kw = dict(D=D, H=4, Hk=Hk, scale=0.2, n_keys=20, kv_rows=rows, rows_per_head=True)
    a = oracle_mod.attention(q, **kw, k0=_f16_rows(Kc), v0=_f16_rows(Vc), n_rows0=nb * br,
                             k_row_bytes0=2 * Hk * D, v_row_bytes0=2 * Hk * D)
    b = oracle_mod.attention(q, **kw, k0=Kp, v0=Vp, n_rows0=nb * br, layout=oracle.PAGED, page_rows=br)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_quant_storage_equals_f16_storage(oracle_mod):
    # scale 1.0 and small integer codes are exact in fp16: both storages hold
    # the same values, so attention must agree bit for bit (checks segment
    # offsets of every head and the nibble order inside attention).
    n, Hk, D = 40, 3, 64
    rng = np.random.default_rng(13)
    codes8 = rng.integers(-127, 128, size=(n, Hk * D // 32, 32), dtype=np.int8)
    u4 = rng.integers(0, 16, size=(n, Hk * D // 32, 32), dtype=np.uint8)
    one = np.array([1.0], np.float16).view(np.uint8)
    K8 = np.empty((n, Hk * D // 32, 34), np.uint8)
    K8[..., 0:2] = one
    K8[..., 2:] = codes8.view(np.uint8)
    V4 = np.empty((n, Hk * D // 32, 18), np.uint8)
    V4[..., 0:2] = one
    V4[..., 2:] = u4[..., :16] | (u4[..., 16:] << 4)
    Kf = codes8.reshape(n, Hk * D).astype(np.float16)
    Vf = (u4.astype(np.int16) - 8).reshape(n, Hk * D).astype(np.float16)
    q = (rng.standard_normal((1, 2, 6, D)) * 0.05).astype(np.float16)
    kw = dict(D=D, H=6, Hk=Hk, scale=1 / 8, n_keys=n)
    a = oracle_mod.attention(q, **kw, k_type=oracle.Q8_0, v_type=oracle.Q4_0,
                             k0=K8.reshape(n, -1), v0=V4.reshape(n, -1), n_rows0=n,
                             k_row_bytes0=K8.shape[1] * 34, v_row_bytes0=V4.shape[1] * 18)
    b = oracle_mod.attention(q, **kw, k0=_f16_rows(Kf), v0=_f16_rows(Vf), n_rows0=n,
                             k_row_bytes0=2 * Hk * D, v_row_bytes0=2 * Hk * D)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------------------------ combine

def _split_parts(oracle_mod, q, K, V, kw, n, bounds):
    rb = K.shape[1]
    os_, ls_ = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        rows = np.full((1, n), -1, np.int32)
        rows[0, a:b] = np.arange(a, b)
        o, l = oracle_mod.attention(q, **kw, k0=K, v0=V, n_rows0=n, k_row_bytes0=rb, v_row_bytes0=rb,
                                    n_keys=n, kv_rows=rows)
        os_.append(o.reshape(-1, kw["D"]))
        ls_.append(l.reshape(-1))
    return np.stack(os_), np.stack(ls_)


@pytest.mark.parametrize("tile", [256, 512, 768, 1024])
def test_split_combine_equals_unsplit_tiles(oracle_mod, tile):
    n = 2600
    q, K, V, kw = _rand_case(14, n=n, H=4, Hk=1, D=32, nq=2)
    rb = K.shape[1]
    whole_o, whole_l = oracle_mod.attention(q, **kw, k0=K, v0=V, n_rows0=n, k_row_bytes0=rb,
                                            v_row_bytes0=rb, n_keys=n)
    bounds = list(range(0, n, tile)) + [n]
    po, pl = _split_parts(oracle_mod, q, K, V, kw, n, bounds)
    o, l = oracle_mod.combine(po, pl)
    assert np.allclose(o, whole_o.reshape(-1, 32), atol=1e-13)
    assert np.allclose(l, whole_l.reshape(-1), atol=1e-12)


@pytest.mark.parametrize("k", [1, 2, 3, 5, 8, 17, 33])
def test_split_combine_any_k(oracle_mod, k):
    n = 700
    q, K, V, kw = _rand_case(15 + k, n=n, H=2, Hk=1, D=16)
    rb = K.shape[1]
    whole_o, whole_l = oracle_mod.attention(q, **kw, k0=K, v0=V, n_rows0=n, k_row_bytes0=rb,
                                            v_row_bytes0=rb, n_keys=n)
    rng = np.random.default_rng(k)
    cuts = sorted(rng.choice(np.arange(1, n), size=k - 1, replace=False).tolist())
    po, pl = _split_parts(oracle_mod, q, K, V, kw, n, [0] + cuts + [n])
    o, l = oracle_mod.combine(po, pl)
    assert np.allclose(o, whole_o.reshape(-1, 16), atol=1e-13)
    assert np.allclose(l, whole_l.reshape(-1), atol=1e-12)
    perm = rng.permutation(k)
    o2, l2 = oracle_mod.combine(po[perm], pl[perm])
    assert np.allclose(o2, o, atol=1e-14) and np.allclose(l2, l, atol=1e-14)


def test_combine_neg_inf_part_and_single_part(oracle_mod):
    rng = np.random.default_rng(20)
    o1 = rng.standard_normal((1, 5, 8))
    l1 = rng.standard_normal((1, 5))
    o, l = oracle_mod.combine(o1, l1)
    assert np.array_equal(o, o1[0]) and np.allclose(l, l1[0], atol=1e-15)
    junk = np.full((1, 5, 8), np.nan)
    o2, l2 = oracle_mod.combine(np.concatenate([o1, junk]), np.concatenate([l1, np.full((1, 5), -np.inf)]))
    assert np.array_equal(o2, o) and np.array_equal(l2, l)
    o3, l3 = oracle_mod.combine(junk, np.full((1, 5), -np.inf))
    assert np.all(o3 == 0) and np.all(l3 == -np.inf)
    # two parts with lse a and b: weights e^a/(e^a+e^b) -- pick a-b = ln 3
    oa, ob = rng.standard_normal((2, 1, 1, 4))
    o4, l4 = oracle_mod.combine(np.stack([oa, ob]).reshape(2, 1, 4), np.array([[math.log(3)], [0.0]]))
    assert np.allclose(o4[0], 0.75 * oa.ravel() + 0.25 * ob.ravel(), atol=1e-15)
    assert abs(l4[0] - math.log(4)) < 1e-15


# ------------------------------------------------------------------ workloads

def test_workload_generators_shapes():
    w = wl.tiny_decode()
    assert w.q.shape == (1, 1, 4, 64) and w.k.shape == (128, 128) and w.k_tail.shape == (128, 128)
    u = wl.unified_decode(n_cache=4096, S=4, rows_per_seq=700, H=8, Hk=2, D=64)
    assert u.kv_rows.shape == (4, 768)
    assert np.all(u.kv_rows[:, 700:] == -1)
    flat = u.kv_rows[u.kv_rows >= 0]
    assert len(np.unique(flat)) == flat.size  # disjoint lists
    assert all(np.all(np.diff(r[r >= 0]) > 0) for r in u.kv_rows)
    l = wl.long_context_decode(n_kv=512, wc=256, tile_rows=128, H=10, Hk=2, D=64)
    assert l.k.shape == (256, 2 * 2 * 34) and l.v_tail.shape == (256, 2 * 2 * 18)
    b = wl.block_sparse_decode(n_kv=64 * 64, S=2, H=8, Hk=2, D=32, n_sel=8, cache_pages=16)
    assert b.kv_rows.shape == (2, 2, 8 * 64)
