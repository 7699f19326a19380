"""Tensor-core prefill with software producers: quantised K/V and row lists.

* q8_0 / q4_0 rows (every K/V pairing the library builds), dense ranges with
  causal positions and sub-ranges, and window + pinned quantised tail;
* fp16 rows through per-sequence row lists with -1 padding (whole padding
  tiles included) for several sequences, and through per-KV-head lists;
* quantised rows through row lists; rows outside every list hold NaN bytes
  and must never be read; a sub-range [kv_begin, kv_end) of longer lists;
* the software producer writes the same operand tiles as the TMA producer: an
  identity row list reproduces the dense TMA result bit for bit.
All against the oracle at the attention tolerance; the status word stays clear.
"""
import math

import numpy as np
import pytest

from split_kv_flash_attn_gb300 import workloads as wl
from tests.gpu_util import check_attention, dev, pinned, vmax_of

pytestmark = pytest.mark.gpu

D = 128
PAIRS = [(wl.Q8_0, wl.Q4_0), (wl.Q8_0, wl.Q8_0), (wl.Q4_0, wl.Q4_0), (wl.Q4_0, wl.Q8_0)]


@pytest.fixture(scope="module")
def skv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import split_kv_flash_attn_gb300 as m
    return m


@pytest.fixture(scope="module")
def h(skv):
    return skv.Handle(0)


def _oracle(oracle_mod, q, H, Hk, kt, vt, K, V, n_rows, **kw):
    return oracle_mod.attention(q, D=D, H=H, Hk=Hk, scale=1 / math.sqrt(D), k_type=kt, v_type=vt, k0=K, v0=V,
                                n_rows0=n_rows, k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1], **kw)


@pytest.mark.parametrize("kt,vt", PAIRS)
def test_prefill_quant_dense(skv, h, oracle_mod, kt, vt):
    rng = wl.generator(4, salt=300 + 3 * kt + vt)
    S, nq, H, Hk, n = 1, 64, 32, 8, 1000
    q = wl.normal_f16(rng, (S, nq, H, D))
    K = wl.cache_rows(rng, kt, n, Hk, D)
    V = wl.cache_rows(rng, vt, n, Hk, D)
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, k_type=kt, v_type=vt)
    want_o, want_l = _oracle(oracle_mod, q, H, Hk, kt, vt, K, V, n, n_keys=n)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, vt, V, D), "quant dense")
    # causal positions over a sub-range, several splits
    b, e, kp0 = 37, 990, 3
    q_pos = np.sort(rng.integers(b + kp0 - 40, e + kp0 + 40, size=(S, nq))).astype(np.int32)
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, k_type=kt, v_type=vt, kv_begin=b, kv_end=e,
                            q_pos=dev(q_pos), key_pos0=kp0)
    rows = np.arange(b, e, dtype=np.int32).reshape(1, -1)
    want_o, want_l = _oracle(oracle_mod, q, H, Hk, kt, vt, K, V, n, n_keys=e - b, kv_rows=rows, q_pos=q_pos,
                             key_pos0=kp0 + b)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, vt, V, D), "quant causal")
    assert h.status() == 0


@pytest.mark.parametrize("kt", [wl.Q8_0, wl.Q4_0])
def test_prefill_quant_query_tile_pairs_ragged(skv, h, oracle_mod, kt):
    """Dense q8_0 / q4_0 keys with q4_0 values are served two query tiles a
    CTA: 80 tokens x 4 heads make three 128-row tiles, so the last pair has
    one tile, itself ragged (64 of its rows past the last token); two
    sequences, causal positions inside a sub-range whose ends are ragged
    against the 128-key tiles, and a range long enough to be split."""
    vt = wl.Q4_0
    rng = wl.generator(4, salt=330 + kt)
    S, nq, H, Hk, n = 2, 80, 16, 4, 9000
    q = wl.normal_f16(rng, (S, nq, H, D))
    K = wl.cache_rows(rng, kt, n, Hk, D)
    V = wl.cache_rows(rng, vt, n, Hk, D)
    b, e, kp0 = 45, 8931, 11
    q_pos = np.stack([np.sort(rng.integers(e + kp0 - 600, e + kp0 + 5, size=nq)) for _ in range(S)]).astype(np.int32)
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, k_type=kt, v_type=vt, kv_begin=b, kv_end=e,
                            q_pos=dev(q_pos), key_pos0=kp0)
    rows = np.tile(np.arange(b, e, dtype=np.int32), (S, 1))
    want_o, want_l = _oracle(oracle_mod, q, H, Hk, kt, vt, K, V, n, n_keys=e - b, kv_rows=rows, q_pos=q_pos,
                             key_pos0=kp0 + b)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, vt, V, D), "query-tile pairs")
    assert h.status() == 0


def test_prefill_quant_window_tail(skv, h, oracle_mod):
    """Prefill over a q8_0 / q4_0 window and a pinned quantised tail streamed
    in 768-row tiles (the long-context layout at reduced size)."""
    rng = wl.generator(4, salt=333)
    S, nq, H, Hk, nw, nt = 1, 64, 40, 8, 2048, 2500
    kt, vt = wl.Q8_0, wl.Q4_0
    q = wl.normal_f16(rng, (S, nq, H, D))
    Kw, Vw = wl.cache_rows(rng, kt, nw, Hk, D), wl.cache_rows(rng, vt, nw, Hk, D)
    Kt, Vt = wl.cache_rows(rng, kt, nt, Hk, D), wl.cache_rows(rng, vt, nt, Hk, D)
    q_pos = (nw + nt - nq + np.arange(nq, dtype=np.int32)).reshape(1, nq)
    o, l = skv.attn_window_tail(h, dev(q), dev(Kw), dev(Vw), pinned(Kt), pinned(Vt), Hk=Hk, tile_rows=768,
                                k_type=kt, v_type=vt, q_pos=dev(q_pos))
    want_o, want_l = oracle_mod.attention(q, D=D, H=H, Hk=Hk, scale=1 / math.sqrt(D), k_type=kt, v_type=vt,
                                          k0=Kw, v0=Vw, n_rows0=nw, k_row_bytes0=Kw.shape[1],
                                          v_row_bytes0=Vw.shape[1], k1=Kt, v1=Vt, n_rows1=nt,
                                          k_row_bytes1=Kt.shape[1], v_row_bytes1=Vt.shape[1], n_keys=nw + nt,
                                          q_pos=q_pos)
    vmax = max(vmax_of(oracle_mod, vt, Vw, D), vmax_of(oracle_mod, vt, Vt, D))
    check_attention(o, l, want_o, want_l, vmax, "quant window+tail")
    assert h.status() == 0


def _lists(rng, n_cache, lens, ld):
    """Per-sequence sorted row lists drawn from a shuffled cache, -1 padded to ld."""
    perm = rng.permutation(n_cache).astype(np.int32)
    out = np.full((len(lens), ld), -1, np.int32)
    at = 0
    for s, n in enumerate(lens):
        out[s, :n] = np.sort(perm[at:at + n])
        at += n
    return out


@pytest.mark.parametrize("kt,vt", [(wl.F16, wl.F16), (wl.Q8_0, wl.Q4_0)])
def test_prefill_row_lists(skv, h, oracle_mod, kt, vt):
    """Three sequences share one cache; each reads its own rows through a
    list padded with -1 (sequence 2 mostly padding: whole 128-key tiles of
    padding), with causal positions at the end of each list."""
    rng = wl.generator(4, salt=400 + kt)
    S, nq, H, Hk, n_cache = 3, 64, 16, 4, 6000
    lens, ld = [2000, 1333, 150], 2048
    q = wl.normal_f16(rng, (S, nq, H, D))
    K = wl.cache_rows(rng, kt, n_cache, Hk, D)
    V = wl.cache_rows(rng, vt, n_cache, Hk, D)
    rows = _lists(rng, n_cache, lens, ld)
    rows[1, 700:764] = -1                                   # padding inside a list too
    q_pos = np.stack([np.arange(nq, dtype=np.int32) + max(0, n - nq) for n in lens]).astype(np.int32)
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, k_type=kt, v_type=vt, kv_rows=dev(rows),
                            q_pos=dev(q_pos))
    want_o, want_l = _oracle(oracle_mod, q, H, Hk, kt, vt, K, V, n_cache, n_keys=ld, kv_rows=rows, q_pos=q_pos)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, vt, V, D), "row-list prefill")
    assert h.status() == 0


@pytest.mark.parametrize("kt,vt", [(wl.F16, wl.F16), (wl.Q8_0, wl.Q4_0)])
def test_prefill_row_lists_read_only_listed_rows(skv, h, oracle_mod, kt, vt):
    """Every cache row that no list names is all 0xFF bytes (an fp16 NaN, a
    NaN block scale): the result stays finite and equal to the oracle's, so
    neither padding entries (-1, inside a list and at its end) nor tile or
    split edges make the producers read a row outside the lists."""
    rng = wl.generator(4, salt=600 + kt)
    S, nq, H, Hk, n_cache = 2, 64, 32, 8, 5000
    lens, ld = [1400, 1100], 1536
    q = wl.normal_f16(rng, (S, nq, H, D))
    K = wl.cache_rows(rng, kt, n_cache, Hk, D)
    V = wl.cache_rows(rng, vt, n_cache, Hk, D)
    rows = _lists(rng, n_cache, lens, ld)
    rows[0, 300:420] = -1
    listed = np.zeros(n_cache, dtype=bool)
    listed[rows[rows >= 0]] = True
    Kp, Vp = K.copy(), V.copy()
    Kp[~listed] = 0xFF
    Vp[~listed] = 0xFF
    q_pos = np.stack([np.arange(nq, dtype=np.int32) + (n - nq) for n in lens]).astype(np.int32)
    o, l = skv.attn_partial(h, dev(q), dev(Kp), dev(Vp), Hk=Hk, k_type=kt, v_type=vt, kv_rows=dev(rows),
                            q_pos=dev(q_pos))
    want_o, want_l = _oracle(oracle_mod, q, H, Hk, kt, vt, K, V, n_cache, n_keys=ld, kv_rows=rows, q_pos=q_pos)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, vt, V, D), "row lists, NaN outside them")
    assert h.status() == 0


@pytest.mark.parametrize("kt,vt", [(wl.F16, wl.F16), (wl.Q4_0, wl.Q8_0)])
def test_prefill_row_list_subrange(skv, h, oracle_mod, kt, vt):
    """Entries [kv_begin, kv_end) of longer lists (both ends ragged against
    the 128-key tiles, sequence 1's end in its padding), a ragged last query
    tile (80 tokens x 4 heads), causal positions: the oracle takes the
    sliced lists with the positions shifted by kv_begin."""
    rng = wl.generator(4, salt=650 + kt)
    S, nq, H, Hk, n_cache = 2, 80, 16, 4, 6000
    lens, ld = [2900, 2500], 3000
    b, e = 333, 2777
    q = wl.normal_f16(rng, (S, nq, H, D))
    K = wl.cache_rows(rng, kt, n_cache, Hk, D)
    V = wl.cache_rows(rng, vt, n_cache, Hk, D)
    rows = _lists(rng, n_cache, lens, ld)
    q_pos = np.stack([np.arange(nq, dtype=np.int32) + (e - nq - 7 * s) for s in range(S)]).astype(np.int32)
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, k_type=kt, v_type=vt, kv_rows=dev(rows),
                            kv_begin=b, kv_end=e, q_pos=dev(q_pos))
    want_o, want_l = _oracle(oracle_mod, q, H, Hk, kt, vt, K, V, n_cache, n_keys=e - b,
                             kv_rows=np.ascontiguousarray(rows[:, b:e]), q_pos=q_pos, key_pos0=b)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, vt, V, D), "row-list sub-range")
    assert h.status() == 0


def test_prefill_per_head_lists(skv, h, oracle_mod):
    rng = wl.generator(4, salt=450)
    S, nq, H, Hk, n_cache, ld = 2, 64, 16, 4, 4096, 768
    q = wl.normal_f16(rng, (S, nq, H, D))
    K = wl.cache_rows(rng, wl.F16, n_cache, Hk, D)
    V = wl.cache_rows(rng, wl.F16, n_cache, Hk, D)
    rows = np.stack([np.stack([np.sort(rng.choice(n_cache, ld, replace=False)) for _ in range(Hk)])
                     for _ in range(S)]).astype(np.int32)
    rows[0, 1, 500:] = -1
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, kv_rows=dev(rows), kv_rows_per_head=True)
    want_o, want_l = _oracle(oracle_mod, q, H, Hk, wl.F16, wl.F16, K, V, n_cache, n_keys=ld, kv_rows=rows,
                             rows_per_head=True)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, V, D), "per-head lists")
    assert h.status() == 0


def test_identity_list_matches_tma_bitwise(skv, h):
    """One 128-row query tile per (sequence, KV head): the dense range and the
    identity row list both run the single-tile kernel (TMA producers against
    software producers) with the same split plan."""
    import torch
    rng = wl.generator(4, salt=500)
    S, nq, H, Hk, n = 2, 32, 32, 8, 3000
    q = wl.normal_f16(rng, (S, nq, H, D))
    K = wl.cache_rows(rng, wl.F16, n, Hk, D)
    V = wl.cache_rows(rng, wl.F16, n, Hk, D)
    qd, Kd, Vd = dev(q), dev(K), dev(V)
    q_pos = dev(np.tile(n - nq + np.arange(nq, dtype=np.int32), (S, 1)))
    o_tma, l_tma = skv.attn_partial(h, qd, Kd, Vd, Hk=Hk, q_pos=q_pos)
    rows = dev(np.tile(np.arange(n, dtype=np.int32), (S, 1)))
    o_sw, l_sw = skv.attn_partial(h, qd, Kd, Vd, Hk=Hk, kv_rows=rows, q_pos=q_pos)
    assert torch.equal(o_tma, o_sw) and torch.equal(l_tma, l_sw)
    assert h.status() == 0
