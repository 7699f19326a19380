"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bit-exact: q8_0/q4_0 decoding and the row gather.  Attention and the combine:
max|dO| <= 2e-3*max|V|, |dlse| <= 1e-4, empty rows exactly (0, -inf).
Sizes span several 64-key tiles, several CTA splits and ragged tails."""
import math

import numpy as np
import pytest

import oracle
from split_kv_flash_attn_gb300 import workloads as wl
from tests.gpu_util import check_attention, dev, pinned, vmax_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import split_kv_flash_attn_gb300 as skv_mod
    return skv_mod


@pytest.fixture(scope="module")
def h(skv):
    return skv.Handle(0)


def _sync():
    import torch
    torch.cuda.synchronize()


# ------------------------------------------------------------ dequant / gather

@pytest.mark.parametrize("type_", [wl.Q8_0, wl.Q4_0])
def test_dequant_bit_exact(skv, h, oracle_mod, type_):
    rng = wl.generator(3, salt=11)
    rows = wl.cache_rows(rng, type_, 4099, 2, 128)          # ragged row count
    raw = rows.reshape(-1).copy()
    blk = 34 if type_ == wl.Q8_0 else 18
    # edge blocks: extreme codes at the smallest and largest drawn scales
    for i, d in enumerate((0.005, 0.02)):
        b = raw[i * blk:(i + 1) * blk]
        b[0:2] = np.array([d], np.float16).view(np.uint8)
        b[2:] = 0x7F if type_ == wl.Q8_0 else 0xF0
        if type_ == wl.Q8_0:
            b[3] = np.int8(-127).view(np.uint8)
    n_vals = raw.size // blk * 32
    fn = skv.kv_dequant_q8_0 if type_ == wl.Q8_0 else skv.kv_dequant_q4_0
    got = fn(h, dev(raw), n_vals).cpu().numpy()
    want = oracle_mod.dequant(type_, raw, n_vals).astype(np.float32)
    assert np.array_equal(got.view(np.int32), want.view(np.int32))


@pytest.mark.parametrize("row_bytes", [256, 68, 34, 2048])
def test_gather_bit_exact(skv, h, row_bytes):
    rng = np.random.default_rng(row_bytes)
    src = rng.integers(0, 256, size=(5000, row_bytes), dtype=np.uint8)
    rows = rng.integers(-1, 5000, size=3001).astype(np.int32)
    rows[:7] = -1
    got = skv.gather_rows(h, dev(src), dev(rows), row_bytes=row_bytes).cpu().numpy()
    want = np.where(rows[:, None] >= 0, src[np.maximum(rows, 0)], 0).astype(np.uint8)
    assert np.array_equal(got, want)


# ------------------------------------------------------------ combine

@pytest.mark.parametrize("P,rows,D", [(1, 5, 64), (3, 37, 128), (17, 100, 128), (300, 40, 128), (2, 9, 64)])
def test_combine_matches_oracle(skv, h, oracle_mod, P, rows, D):
    rng = np.random.default_rng(P * 1000 + rows)
    o_parts = rng.standard_normal((P, rows, D)).astype(np.float32)
    lse_parts = (rng.standard_normal((P, rows)) * 3).astype(np.float32)
    lse_parts[rng.random((P, rows)) < 0.2] = -np.inf
    lse_parts[:, 0] = -np.inf                     # a row with no visible key
    o_parts[np.isneginf(lse_parts)] = np.nan      # never read
    o, l = skv.attn_combine(h, dev(o_parts), dev(lse_parts))
    want_o, want_l = oracle_mod.combine(np.nan_to_num(o_parts.astype(np.float64)), lse_parts.astype(np.float64))
    check_attention(o, l, want_o, want_l, float(np.nanmax(np.abs(o_parts))), "combine")


def test_combine_zero_parts(skv, h):
    import torch
    o = torch.full((4, 64), 7.0, device="cuda")
    l = torch.full((4,), 7.0, device="cuda")
    skv.attn_combine(h, torch.empty((0, 4, 64), device="cuda"), torch.empty((0, 4), device="cuda"), o=o, lse=l)
    assert torch.all(o == 0) and torch.all(torch.isneginf(l))


# ------------------------------------------------------------ attention: dense

def _oracle_dense(oracle_mod, w_q, K, V, D, H, Hk, n, **kw):
    return oracle_mod.attention(w_q, D=D, H=H, Hk=Hk, scale=1 / math.sqrt(D), k0=K, v0=V, n_rows0=n,
                                k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1], n_keys=n, **kw)


@pytest.mark.parametrize("D,H,Hk,nq,n", [
    (64, 4, 1, 1, 256),       # tiny decode geometry
    (128, 32, 8, 1, 1000),    # GQA 4:1, ragged tail tile
    (128, 40, 8, 1, 777),     # G = 5
    (128, 16, 2, 1, 5000),    # G = 8, many tiles and splits
    (64, 8, 1, 3, 300),       # three tokens x G=8 -> three column groups
    (128, 4, 4, 2, 65),       # G = 1, one key past a tile
    (64, 6, 3, 1, 1),         # one key
])
def test_attn_dense_f16(skv, h, oracle_mod, D, H, Hk, nq, n):
    rng = wl.generator(2, salt=D + H + n)
    q = wl.normal_f16(rng, (2, nq, H, D))
    K = wl.cache_rows(rng, wl.F16, n, Hk, D)
    V = wl.cache_rows(rng, wl.F16, n, Hk, D)
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk)
    want_o, want_l = _oracle_dense(oracle_mod, q, K, V, D, H, Hk, n)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, V, D), "dense")


def test_attn_dense_subrange_causal_mask(skv, h, oracle_mod):
    D, H, Hk, nq, n = 128, 8, 2, 4, 3000
    rng = wl.generator(4, salt=5)
    q = wl.normal_f16(rng, (1, nq, H, D))
    K = wl.cache_rows(rng, wl.F16, n, Hk, D)
    V = wl.cache_rows(rng, wl.F16, n, Hk, D)
    q_pos = np.array([[10, 1500, 2599, 5000]], np.int32)
    mask = (rng.standard_normal((1, nq, n)) * 2).astype(np.float16)
    mask[:, :, 100:164] = -np.inf
    b, e = 70, 2600
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, kv_begin=b, kv_end=e, q_pos=dev(q_pos),
                            key_pos0=3, mask=dev(mask))
    # oracle: keys b..e-1 as a row list, positions key_pos0 + logical index
    rows = np.arange(b, e, dtype=np.int32).reshape(1, -1)
    want_o, want_l = oracle_mod.attention(q, D=D, H=H, Hk=Hk, scale=1 / math.sqrt(D), k0=K, v0=V, n_rows0=n,
                                          k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1], n_keys=e - b,
                                          kv_rows=rows, q_pos=q_pos, key_pos0=3 + b, mask=mask[:, :, b:e])
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, V, D), "causal+mask")


# ------------------------------------------------------------ attention: row lists

@pytest.mark.parametrize("per_head", [False, True])
def test_attn_rows_padding(skv, h, oracle_mod, per_head):
    D, H, Hk, S, n_cache, n_list = 128, 16, 4, 5, 9000, 2304
    rng = wl.generator(2, salt=77 + per_head)
    q = wl.normal_f16(rng, (S, 1, H, D))
    K = wl.cache_rows(rng, wl.F16, n_cache, Hk, D)
    V = wl.cache_rows(rng, wl.F16, n_cache, Hk, D)
    shape = (S, Hk, n_list) if per_head else (S, n_list)
    rows = rng.integers(0, n_cache, size=shape).astype(np.int32)
    flat = rows.reshape(-1, n_list)
    flat[0, 2000:] = -1                   # ragged padding, 304 rows
    flat[1, :] = -1                       # a list of padding only
    flat[2, 64:1024] = -1                 # whole padding tiles inside the list
    flat[3, ::7] = -1                     # scattered padding
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, kv_rows=dev(rows), kv_rows_per_head=per_head)
    want_o, want_l = oracle_mod.attention(q, D=D, H=H, Hk=Hk, scale=1 / math.sqrt(D), k0=K, v0=V, n_rows0=n_cache,
                                          k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1], n_keys=n_list,
                                          kv_rows=rows, rows_per_head=per_head)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, V, D), "rows")


@pytest.mark.parametrize("S,H,Hk,n,b,e,per_head", [
    (2, 32, 8, 4096, 0, 4096, False),     # whole range, several splits
    (3, 40, 8, 3000, 0, 3000, True),      # G = 5, ragged last tile, per-head lists
    (1, 8, 2, 20000, 333, 19001, False),  # a sub-range starting mid-tile, many splits
])
def test_identity_rows_bitwise_equal_dense(skv, h, S, H, Hk, n, b, e, per_head):
    """An identity row list takes the same split plan and the same kernel as
    the dense range (both plan from the key count and the units alone), so
    the results must agree bit for bit: the gather changes only where the
    rows come from."""
    import torch
    D = 128
    rng = wl.generator(2, salt=3 + n)
    q = wl.normal_f16(rng, (S, 1, H, D))
    K = dev(wl.cache_rows(rng, wl.F16, n, Hk, D))
    V = dev(wl.cache_rows(rng, wl.F16, n, Hk, D))
    ident = np.arange(n, dtype=np.int32)
    rows = dev(np.tile(ident, (S, Hk, 1)) if per_head else np.tile(ident, (S, 1)))
    qd = dev(q)
    o1, l1 = skv.attn_partial(h, qd, K, V, Hk=Hk, kv_rows=rows, kv_rows_per_head=per_head, kv_begin=b, kv_end=e)
    o2, l2 = skv.attn_partial(h, qd, K, V, Hk=Hk, kv_begin=b, kv_end=e)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_unified_cache_reduced(skv, h, oracle_mod):
    w = wl.unified_decode(n_cache=16384, S=8, rows_per_seq=1900, H=32, Hk=8, D=128, salt=1)
    o, l = skv.attn_partial(h, dev(w.q), dev(w.k), dev(w.v), Hk=w.Hk, kv_rows=dev(w.kv_rows))
    want_o, want_l = oracle_mod.attention(w.q, D=w.D, H=w.H, Hk=w.Hk, scale=w.scale, k0=w.k, v0=w.v,
                                          n_rows0=w.k.shape[0], k_row_bytes0=w.k.shape[1],
                                          v_row_bytes0=w.v.shape[1], n_keys=w.n_keys, kv_rows=w.kv_rows)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, w.v, w.D), "unified reduced")


# ------------------------------------------------------------ attention: quantised

@pytest.mark.parametrize("kt,vt,D", [(wl.Q8_0, wl.Q4_0, 128), (wl.Q8_0, wl.Q4_0, 64), (wl.Q8_0, wl.Q8_0, 128),
                                     (wl.Q4_0, wl.Q4_0, 128), (wl.Q4_0, wl.Q8_0, 64)])
def test_attn_quant_dense_and_rows(skv, h, oracle_mod, kt, vt, D):
    H, Hk, n = 40, 8, 2500
    rng = wl.generator(3, salt=kt * 10 + vt + D)
    q = wl.normal_f16(rng, (1, 1, H, D))
    K = wl.cache_rows(rng, kt, n, Hk, D)
    V = wl.cache_rows(rng, vt, n, Hk, D)
    vmax = vmax_of(oracle_mod, vt, V, D)
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, k_type=kt, v_type=vt)
    want_o, want_l = oracle_mod.attention(q, D=D, H=H, Hk=Hk, scale=1 / math.sqrt(D), k_type=kt, v_type=vt,
                                          k0=K, v0=V, n_rows0=n, k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1],
                                          n_keys=n)
    check_attention(o, l, want_o, want_l, vmax, "quant dense")
    rows = rng.integers(-1, n, size=(1, 1024)).astype(np.int32)
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, k_type=kt, v_type=vt, kv_rows=dev(rows))
    want_o, want_l = oracle_mod.attention(q, D=D, H=H, Hk=Hk, scale=1 / math.sqrt(D), k_type=kt, v_type=vt,
                                          k0=K, v0=V, n_rows0=n, k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1],
                                          n_keys=1024, kv_rows=rows)
    check_attention(o, l, want_o, want_l, vmax, "quant rows")


# ------------------------------------------------------------ window + tail

def _oracle_wt(oracle_mod, w, **kw):
    return oracle_mod.attention(w.q, D=w.D, H=w.H, Hk=w.Hk, scale=w.scale, k_type=w.k_type, v_type=w.v_type,
                                k0=w.k, v0=w.v, n_rows0=w.k.shape[0], k_row_bytes0=w.k.shape[1],
                                v_row_bytes0=w.v.shape[1], k1=w.k_tail, v1=w.v_tail, n_rows1=w.k_tail.shape[0],
                                k_row_bytes1=w.k_tail.shape[1], v_row_bytes1=w.v_tail.shape[1], n_keys=w.n_keys,
                                **kw)


def test_tiny_decode_window_tail(skv, h, oracle_mod):
    w = wl.tiny_decode()
    o, l = skv.attn_window_tail(h, dev(w.q), dev(w.k), dev(w.v), pinned(w.k_tail), pinned(w.v_tail), Hk=w.Hk,
                                tile_rows=w.tile_rows)
    want_o, want_l = _oracle_wt(oracle_mod, w)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, np.concatenate([w.v, w.v_tail]), w.D), "tiny")


@pytest.mark.parametrize("tile_rows", [256, 512, 768, 1024, 1000])
def test_long_context_reduced_tiles(skv, h, oracle_mod, tile_rows):
    w = wl.long_context_decode(n_kv=6000, wc=1536, tile_rows=tile_rows, H=40, Hk=8, D=128)
    o, l = skv.attn_window_tail(h, dev(w.q), dev(w.k), dev(w.v), pinned(w.k_tail), pinned(w.v_tail), Hk=w.Hk,
                                tile_rows=tile_rows, k_type=w.k_type, v_type=w.v_type)
    want_o, want_l = _oracle_wt(oracle_mod, w)
    vmax = vmax_of(oracle_mod, wl.Q4_0, np.concatenate([w.v, w.v_tail]), w.D)
    check_attention(o, l, want_o, want_l, vmax, f"window+tail tile={tile_rows}")


def test_prefill_reduced_causal(skv, h, oracle_mod):
    w = wl.prefill_chunk(n_kv=2048, wc=1024, nq=24, H=8, Hk=2, D=128, tile_rows=384)
    o, l = skv.attn_window_tail(h, dev(w.q), dev(w.k), dev(w.v), pinned(w.k_tail), pinned(w.v_tail), Hk=w.Hk,
                                tile_rows=w.tile_rows, q_pos=dev(w.q_pos))
    want_o, want_l = _oracle_wt(oracle_mod, w, q_pos=w.q_pos)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, np.concatenate([w.v, w.v_tail]), w.D),
                    "prefill reduced")


def test_window_only_and_tail_only(skv, h, oracle_mod):
    w = wl.tiny_decode(n_kv=700, wc=700)
    empty = np.zeros((0, w.k.shape[1]), np.uint8)
    o, l = skv.attn_window_tail(h, dev(w.q), dev(w.k), dev(w.v), None, None, Hk=w.Hk, n_tail=0)
    want_o, want_l = _oracle_dense(oracle_mod, w.q, w.k, w.v, w.D, w.H, w.Hk, 700)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, w.v, w.D), "window only")
    o, l = skv.attn_window_tail(h, dev(w.q), None, None, pinned(w.k), pinned(w.v), Hk=w.Hk, n_win=0,
                                tile_rows=256)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, w.v, w.D), "tail only")
    del empty


def test_back_to_back_calls_reuse_ring(skv, h, oracle_mod):
    import torch
    ws = [wl.long_context_decode(n_kv=3000, wc=500, tile_rows=512, H=10, Hk=2, D=128) for _ in range(1)]
    w2 = wl.tiny_decode(n_kv=3000, wc=500, H=10, Hk=2, D=128)
    w1 = ws[0]
    o1, l1 = skv.attn_window_tail(h, dev(w1.q), dev(w1.k), dev(w1.v), pinned(w1.k_tail), pinned(w1.v_tail), Hk=2,
                                  tile_rows=512, k_type=w1.k_type, v_type=w1.v_type)
    o2, l2 = skv.attn_window_tail(h, dev(w2.q), dev(w2.k), dev(w2.v), pinned(w2.k_tail), pinned(w2.v_tail), Hk=2,
                                  tile_rows=512)
    torch.cuda.synchronize()
    check_attention(o1, l1, *_oracle_wt(oracle_mod, w1),
                    vmax_of(oracle_mod, wl.Q4_0, np.concatenate([w1.v, w1.v_tail]), 128), "first call")
    check_attention(o2, l2, *_oracle_wt(oracle_mod, w2),
                    vmax_of(oracle_mod, wl.F16, np.concatenate([w2.v, w2.v_tail]), 128), "second call")


def test_pageable_tail_rejected(skv, h):
    import torch
    w = wl.tiny_decode()
    with pytest.raises(skv.SplitKVError) as e:
        skv.attn_window_tail(h, dev(w.q), dev(w.k), dev(w.v), torch.from_numpy(w.k_tail),
                             torch.from_numpy(w.v_tail), Hk=w.Hk)
    assert e.value.status == 3


def test_bad_shape_rejected(skv, h):
    import torch
    q = torch.zeros((1, 1, 6, 128), dtype=torch.float16, device="cuda")
    k = torch.zeros((10, 4 * 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(skv.SplitKVError) as e:
        skv.attn_partial(h, q, k, k, Hk=4)        # H % Hk != 0
    assert e.value.status == 1
    q2 = torch.zeros((1, 1, 4, 96), dtype=torch.float16, device="cuda")
    with pytest.raises(skv.SplitKVError) as e:
        skv.attn_partial(h, q2, k, k, Hk=4)
    assert e.value.status == 2
