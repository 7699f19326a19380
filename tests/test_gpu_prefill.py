"""Parity of the tensor-core prefill path (tcgen05 / TMEM) against the oracle.

The path is taken for fp16 K/V, head dim 128, no additive mask and at least
64 query rows per KV head (nq x G); these cases cover partial 128-row query
tiles, partial 128-key tiles, G = 1/4/8, causal rows that see no key, key
sub-ranges, several key splits (merged in the kernel) and the full-size
prefill chunk on sampled tokens.  After each case the handle's device status
word must be clear (no bounded wait gave up)."""
import math

import numpy as np
import pytest

from split_kv_flash_attn_gb300 import workloads as wl
from tests.gpu_util import check_attention, dev, pinned, vmax_of

pytestmark = pytest.mark.gpu


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


def _case(seed, S, nq, H, Hk, n, D=128):
    rng = wl.generator(4, salt=seed)
    q = wl.normal_f16(rng, (S, nq, H, D))
    K = wl.cache_rows(rng, wl.F16, n, Hk, D)
    V = wl.cache_rows(rng, wl.F16, n, Hk, D)
    return rng, q, K, V


@pytest.mark.parametrize("S,nq,H,Hk,n", [
    (1, 64, 32, 8, 1000),      # G = 4: 256 rows, two full query tiles, ragged key tile
    (1, 40, 32, 8, 700),       # 160 rows: partial second query tile
    (2, 100, 4, 4, 513),       # G = 1, two sequences, one key past a tile
    (1, 17, 16, 2, 2048),      # G = 8: 136 rows
    (1, 128, 8, 2, 5000),      # several key splits
])
def test_prefill_dense(skv, h, oracle_mod, S, nq, H, Hk, n):
    _, q, K, V = _case(S * 7 + nq + n, S, nq, H, Hk, n)
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk)
    want_o, want_l = oracle_mod.attention(q, D=128, H=H, Hk=Hk, scale=1 / math.sqrt(128), k0=K, v0=V, n_rows0=n,
                                          k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1], n_keys=n)
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, V, 128), "prefill dense")
    assert h.status() == 0


def test_prefill_causal_subrange(skv, h, oracle_mod):
    S, nq, H, Hk, n = 1, 96, 16, 4, 3000
    rng, q, K, V = _case(91, S, nq, H, Hk, n)
    b, e, kp0 = 200, 2900, 5
    # positions: some rows see nothing (q_pos below the first key), some see all
    q_pos = np.sort(rng.integers(b + kp0 - 50, e + kp0 + 50, size=(S, nq))).astype(np.int32)
    q_pos[0, :3] = b + kp0 - 1 - np.arange(3)
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, kv_begin=b, kv_end=e, q_pos=dev(q_pos),
                            key_pos0=kp0)
    rows = np.arange(b, e, dtype=np.int32).reshape(1, -1)
    want_o, want_l = oracle_mod.attention(q, D=128, H=H, Hk=Hk, scale=1 / math.sqrt(128), k0=K, v0=V, n_rows0=n,
                                          k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1], n_keys=e - b,
                                          kv_rows=rows, q_pos=q_pos, key_pos0=kp0 + b)
    assert np.isneginf(want_l[0, :3]).all()
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, V, 128), "prefill causal")
    assert h.status() == 0


@pytest.mark.parametrize("rows_list", [False, True])
def test_prefill_reference_moves_on_a_later_tile(skv, h, oracle_mod, rows_list):
    """Keys of later 128-key tiles scaled up (x4 in tile 3, x12 in tile 6,
    x40 on four keys of tile 9) so that row maxima grow by far more than 2^8
    after the first tile: the kernel's lazy reference moves mid-walk, O is
    rescaled in tensor memory and the tile's exponentials are taken again
    against the new reference (the dense range runs the TMA kernel, the
    identity row list the copy-warp kernel)."""
    S, nq, H, Hk, n = 1, 64, 32, 8, 1400
    rng, q, K, V = _case(812, S, nq, H, Hk, n)
    Kf = K.view(np.float16).reshape(n, Hk * 128).astype(np.float32)
    Kf[3 * 128:4 * 128] *= 4.0
    Kf[6 * 128:7 * 128] *= 12.0
    Kf[9 * 128 + 5:9 * 128 + 9] *= 40.0
    K = Kf.astype(np.float16).view(np.uint8).reshape(n, Hk * 256)
    kw = {"kv_rows": dev(np.arange(n, dtype=np.int32).reshape(1, n))} if rows_list else {}
    o, l = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk, **kw)
    want_o, want_l = oracle_mod.attention(q, D=128, H=H, Hk=Hk, scale=1 / math.sqrt(128), k0=K, v0=V, n_rows0=n,
                                          k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1], n_keys=n)
    # the maxima did move by more than 2^8 (log2 units) after the first tile
    first = oracle_mod.attention(q, D=128, H=H, Hk=Hk, scale=1 / math.sqrt(128), k0=K[:128], v0=V[:128],
                                 n_rows0=128, k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1], n_keys=128)[1]
    assert float(np.max(want_l - first)) / math.log(2) > 8
    check_attention(o, l, want_o, want_l, vmax_of(oracle_mod, wl.F16, V, 128), "reference moves")
    assert h.status() == 0


@pytest.mark.parametrize("tile_rows", [384, 1024])
def test_prefill_window_tail_reduced(skv, h, oracle_mod, tile_rows):
    w = wl.prefill_chunk(n_kv=4096, wc=2048, nq=64, H=32, Hk=8, D=128, tile_rows=tile_rows)
    o, l = skv.attn_window_tail(h, dev(w.q), dev(w.k), dev(w.v), pinned(w.k_tail), pinned(w.v_tail), Hk=w.Hk,
                                tile_rows=tile_rows, q_pos=dev(w.q_pos))
    want_o, want_l = oracle_mod.attention(w.q, D=w.D, H=w.H, Hk=w.Hk, scale=w.scale, k0=w.k, v0=w.v,
                                          n_rows0=w.k.shape[0], k_row_bytes0=w.k.shape[1],
                                          v_row_bytes0=w.v.shape[1], k1=w.k_tail, v1=w.v_tail,
                                          n_rows1=w.k_tail.shape[0], k_row_bytes1=w.k_tail.shape[1],
                                          v_row_bytes1=w.v_tail.shape[1], n_keys=w.n_keys, q_pos=w.q_pos)
    vmax = vmax_of(oracle_mod, wl.F16, np.concatenate([w.v, w.v_tail]), w.D)
    check_attention(o, l, want_o, want_l, vmax, "prefill window+tail")
    assert h.status() == 0


def test_prefill_full_size_sampled_tokens(skv, h, oracle_mod):
    """512 tokens at positions 65024..65535 over 65536 keys (32768 window +
    32768 pinned tail, 8192-row tiles); the oracle checks 12 sampled tokens."""
    w = wl.prefill_chunk()
    o, l = skv.attn_window_tail(h, dev(w.q), dev(w.k), dev(w.v), pinned(w.k_tail), pinned(w.v_tail), Hk=w.Hk,
                                tile_rows=w.tile_rows, q_pos=dev(w.q_pos))
    o = o.cpu().numpy()
    l = l.cpu().numpy()
    rng = np.random.default_rng(4)
    toks = np.unique(np.r_[0, 1, 255, 511, rng.choice(512, 8, replace=False)])
    qs = np.ascontiguousarray(w.q[:, toks])
    want_o, want_l = oracle_mod.attention(qs, D=w.D, H=w.H, Hk=w.Hk, scale=w.scale, k0=w.k, v0=w.v,
                                          n_rows0=w.k.shape[0], k_row_bytes0=w.k.shape[1],
                                          v_row_bytes0=w.v.shape[1], k1=w.k_tail, v1=w.v_tail,
                                          n_rows1=w.k_tail.shape[0], k_row_bytes1=w.k_tail.shape[1],
                                          v_row_bytes1=w.v_tail.shape[1], n_keys=w.n_keys,
                                          q_pos=np.ascontiguousarray(w.q_pos[:, toks]))
    import torch
    vmax = float(np.abs(np.concatenate([w.v, w.v_tail]).view(np.float16)).max())
    check_attention(torch.from_numpy(o[:, toks]), torch.from_numpy(l[:, toks]), want_o, want_l, vmax,
                    "prefill full size")
    assert h.status() == 0


def test_prefill_matches_decode_path_on_one_token(skv, h, oracle_mod):
    """One query token per head group routes to the decode kernel; 64 tokens
    route to the tensor-core kernel.  Token 0's rows must agree between the
    two paths (and with the oracle) within the attention tolerance."""
    S, nq, H, Hk, n = 1, 64, 32, 8, 2000
    _, q, K, V = _case(5, S, nq, H, Hk, n)
    Kd, Vd = dev(K), dev(V)
    o_tc, l_tc = skv.attn_partial(h, dev(q), Kd, Vd, Hk=Hk)
    o_dec, l_dec = skv.attn_partial(h, dev(np.ascontiguousarray(q[:, :1])), Kd, Vd, Hk=Hk)
    vmax = vmax_of(oracle_mod, wl.F16, V, 128)
    want_o, want_l = oracle_mod.attention(q[:, :1], D=128, H=H, Hk=Hk, scale=1 / math.sqrt(128), k0=K, v0=V,
                                          n_rows0=n, k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1], n_keys=n)
    check_attention(o_tc[:, :1], l_tc[:, :1], want_o, want_l, vmax, "tc token 0")
    check_attention(o_dec, l_dec, want_o, want_l, vmax, "decode token 0")
