"""Appending rows: write routing, quantise-on-append and write-through.

* skv_kv_append writes the same bytes as the oracle (bit-exact) for fp16, q8_0
  and q4_0 rows, into a device window and a pinned host tail, with padded row
  strides, skipped and out-of-range positions;
* a live decode loop (a prefill chunk appended, then one row per step, then
  window + tail attention) matches the oracle over the oracle-appended cache;
* skv_bcache_append keeps the host copy authoritative (bit-exact against the
  oracle's paged append) and every resident page equal to its host page, so
  attention through the cache after appends, with no fetch, matches the oracle.
"""
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
    import split_kv_flash_attn_gb300 as m
    return m


@pytest.fixture(scope="module")
def h(skv):
    return skv.Handle(0)


def _regions(n0, n1, row_bytes, fill0=0xAB, fill1=0xCD):
    return np.full(n0 * row_bytes, fill0, np.uint8), np.full(n1 * row_bytes, fill1, np.uint8)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("type_,pad", [(wl.F16, 0), (wl.F16, 4), (wl.Q8_0, 2), (wl.Q4_0, 6)])
def test_kv_append_bit_exact(skv, h, D, type_, pad):
    import torch
    rng = wl.generator(6, salt=D + 3 * type_ + pad)
    Hk, n0, n1 = 8, 300, 500
    row_bytes = Hk * wl.segment_bytes(type_, D) + pad
    r0, r1 = _regions(n0, n1, row_bytes)
    pos = rng.permutation(n0 + n1)[:256].astype(np.int32)
    pos[7] = -1                                              # skipped
    k, _ = wl.new_kv_values(rng, pos.size, Hk, D)
    d0, d1 = dev(r0), pinned(r1)
    skv.kv_append(h, dev(k), dev(pos), d0, d1, type_=type_, n_rows0=n0, n_rows1=n1, row_bytes=row_bytes)
    torch.cuda.synchronize()
    assert h.status() == 0
    bad = oracle.kv_append(type_, k, pos, r0, n0, r1, n1, row_bytes)
    assert bad == 0
    assert np.array_equal(d0.cpu().numpy(), r0), "window bytes differ from the oracle"
    assert np.array_equal(d1.numpy(), r1), "tail bytes differ from the oracle"


def _tie_blocks(rng, x, qmax):
    """Overwrite blocks of x (float32 [..., D], 32-value blocks) with the cases
    where a product with a reciprocal and the fp32 quotient could decide
    differently: values on and within 3 ulps of half-integer multiples of the
    block's scale (exact ties included), block maxima whose amax/qmax falls
    exactly between two fp16 values, and blocks with fp16-subnormal scales --
    some so small that the rounded scale leaves |x / d| past qmax + 0.5 (the
    clamps: q8_0 at +-127, q4_0 at 0 and 15) or rounds to zero."""
    blocks = x.reshape(-1, 32)
    nb = blocks.shape[0]
    # 0: untouched, 1: ties, 2: fp16-midpoint scale, 3: subnormal scale, 4: a few fp16 ulps of scale
    kind = rng.integers(0, 5, nb)
    d = rng.uniform(1e-3, 0.05, nb).astype(np.float16).astype(np.float32)
    k = rng.integers(-qmax, qmax, (nb, 32)).astype(np.float32)
    t = (k + 0.5) * d[:, None]                 # exact in fp32 (9-bit x 11-bit products)
    nudge = rng.integers(-3, 4, (nb, 32)).astype(np.int32)
    nudge[:, ::4] = 0                          # a quarter stay exact ties
    t = (t.view(np.int32) + nudge).view(np.float32)
    t[:, 0] = qmax * d                         # the block maximum: amax / qmax = d exactly
    ties = kind == 1
    blocks[ties] = t[ties]
    # amax / qmax exactly halfway between two fp16 values
    mid = kind == 2
    h = d.astype(np.float16)
    up = np.nextafter(h, np.float16(np.inf)).astype(np.float32)
    m = (d + up) / 2                           # exact: 12 significant bits
    blocks[mid] = np.clip(blocks[mid], -0.99 * qmax * m[mid, None], 0.99 * qmax * m[mid, None])
    blocks[mid, 5] = -qmax * m[mid]            # exact: 12-bit x 7-bit product
    sub = kind == 3
    blocks[sub] *= np.float32(2e-5)
    tiny = kind == 4
    blocks[tiny] *= np.float32(1e-6)
    return x


@pytest.mark.parametrize("type_", [wl.Q8_0, wl.Q4_0])
def test_kv_append_quant_near_ties_bit_exact(skv, h, type_):
    """Quantise-on-append decides each code without dividing unless the value
    is near a rounding boundary; on blocks built to sit on those boundaries,
    and on 32768 ordinary rows, every stored byte equals the oracle's fp32
    division rule."""
    import torch
    rng = wl.generator(6, salt=4242 + type_)
    qmax = 127 if type_ == wl.Q8_0 else 7
    Hk, D = 8, 128
    row_bytes = Hk * wl.segment_bytes(type_, D)
    for n, ties in ((4096, True), (32768, False)):
        x, _ = wl.new_kv_values(rng, n, Hk, D)
        if ties:
            x = _tie_blocks(rng, x, qmax)
        pos = np.arange(n, dtype=np.int32)
        r0 = np.zeros(n * row_bytes, np.uint8)
        d0 = dev(r0)
        skv.kv_append(h, dev(x), dev(pos), d0, None, type_=type_, n_rows0=n, n_rows1=0, row_bytes=row_bytes)
        torch.cuda.synchronize()
        assert h.status() == 0
        assert oracle.kv_append(type_, x, pos, r0, n, np.zeros(1, np.uint8), 0, row_bytes) == 0
        got = d0.cpu().numpy()
        assert np.array_equal(got, r0), f"{int((got != r0).sum())} bytes differ from the oracle (ties={ties})"


def test_kv_append_out_of_range_sets_status(skv, h):
    import torch
    Hk, D, n0, n1 = 2, 64, 8, 8
    row_bytes = Hk * 2 * D
    r0, r1 = _regions(n0, n1, row_bytes)
    d0, d1 = dev(r0), pinned(r1)
    pos = np.array([3, 16, 40, 12], np.int32)                # 16 and 40 are past the end
    k, _ = wl.new_kv_values(wl.generator(6, salt=99), pos.size, Hk, D)
    skv.kv_append(h, dev(k), dev(pos), d0, d1, n_rows0=n0, n_rows1=n1, row_bytes=row_bytes)
    torch.cuda.synchronize()
    with pytest.raises(skv.SplitKVError) as e:
        h.status()
    assert e.value.status == 8                               # SKV_EDEVICE
    assert h.status() == 0                                   # the word was cleared
    oracle.kv_append(wl.F16, k, pos, r0, n0, r1, n1, row_bytes)
    assert np.array_equal(d0.cpu().numpy(), r0) and np.array_equal(d1.numpy(), r1)


def test_kv_append_rejects_pageable_tail(skv, h):
    import torch
    Hk, D = 2, 64
    x = torch.zeros((1, Hk, D), dtype=torch.float32, device="cuda")
    pos = torch.zeros((1,), dtype=torch.int32, device="cuda")
    tail = torch.zeros((4, Hk * 2 * D), dtype=torch.uint8)   # not page-locked
    with pytest.raises(skv.SplitKVError) as e:
        skv.kv_append(h, x, pos, None, tail, n_rows0=0, n_rows1=4)
    assert e.value.status == 3                               # SKV_ENOTPINNED


@pytest.mark.parametrize("k_type,v_type", [(wl.F16, wl.F16), (wl.Q8_0, wl.Q4_0), (wl.Q8_0, wl.Q8_0)])
def test_decode_loop_append_then_attention(skv, h, oracle_mod, k_type, v_type):
    """A prefill chunk of 1500 rows, then 6 single-row decode steps, appended
    across the window/tail boundary (window 1024 rows); after the last step,
    window + tail attention over all rows against the oracle."""
    import torch
    rng = wl.generator(6, salt=1000 + 3 * k_type + v_type)
    Hk, H, D, n0, n1 = 4, 16, 128, 1024, 1024
    kb, vb = Hk * wl.segment_bytes(k_type, D), Hk * wl.segment_bytes(v_type, D)
    rk0, rk1 = _regions(n0, n1, kb, 0, 0)
    rv0, rv1 = _regions(n0, n1, vb, 0, 0)
    dk0, dk1, dv0, dv1 = dev(rk0), pinned(rk1), dev(rv0), pinned(rv1)
    n_cur = 0
    for n_new in [1500] + [1] * 6:
        pos = np.arange(n_cur, n_cur + n_new, dtype=np.int32)
        k, v = wl.new_kv_values(rng, n_new, Hk, D)
        pos_d = dev(pos)
        skv.kv_append(h, dev(k), pos_d, dk0, dk1, type_=k_type, n_rows0=n0, n_rows1=n1)
        skv.kv_append(h, dev(v), pos_d, dv0, dv1, type_=v_type, n_rows0=n0, n_rows1=n1)
        oracle.kv_append(k_type, k, pos, rk0, n0, rk1, n1, kb)
        oracle.kv_append(v_type, v, pos, rv0, n0, rv1, n1, vb)
        n_cur += n_new
    q = wl.normal_f16(rng, (1, 1, H, D))
    o, lse = skv.attn_window_tail(h, dev(q), dk0.view(n0, kb), dv0.view(n0, vb), dk1.view(n1, kb),
                                  dv1.view(n1, vb), Hk=Hk, n_win=n0, n_tail=n_cur - n0, tile_rows=256,
                                  k_type=k_type, v_type=v_type)
    torch.cuda.synchronize()
    assert h.status() == 0
    assert np.array_equal(dk0.cpu().numpy(), rk0) and np.array_equal(dk1.numpy(), rk1)
    assert np.array_equal(dv0.cpu().numpy(), rv0) and np.array_equal(dv1.numpy(), rv1)
    want_o, want_l = oracle_mod.attention(q, D=D, H=H, Hk=Hk, scale=1 / math.sqrt(D), k_type=k_type,
                                          v_type=v_type, k0=rk0, v0=rv0, n_rows0=n0, k_row_bytes0=kb,
                                          v_row_bytes0=vb, k1=rk1, v1=rv1, n_rows1=n_cur - n0, k_row_bytes1=kb,
                                          v_row_bytes1=vb, n_keys=n_cur)
    vmax = max(vmax_of(oracle_mod, v_type, rv0, D), vmax_of(oracle_mod, v_type, rv1[:(n_cur - n0) * vb], D))
    check_attention(o, lse, want_o, want_l, vmax, "append loop")


def _pool_pages(skv, h, c, page_ids, page_bytes):
    """Copies of the pool pages named by page_ids (K, V) as uint8 [n][page_bytes]."""
    import torch
    k_ptr, v_ptr, _, _ = c.pool()
    ids = page_ids.reshape(-1).to(torch.int32)
    out_k = torch.empty((ids.numel(), page_bytes), dtype=torch.uint8, device="cuda")
    out_v = torch.empty_like(out_k)
    skv.gather_rows(h, k_ptr, ids, row_bytes=page_bytes, out=out_k)
    skv.gather_rows(h, v_ptr, ids, row_bytes=page_bytes, out=out_v)
    return out_k.cpu().numpy(), out_v.cpu().numpy()


@pytest.mark.parametrize("n_slots", [64, 12])
def test_block_cache_write_through(skv, h, oracle_mod, n_slots):
    import torch
    rng = wl.generator(6, salt=2000 + n_slots)
    Hk, H, D, br, n_blocks, S, n_sel = 4, 16, 128, 64, 32, 2, 6
    host_k = wl.normal_f16(rng, (n_blocks, Hk, br, D))
    host_v = wl.normal_f16(rng, (n_blocks, Hk, br, D))
    hk, hv = pinned(host_k), pinned(host_v)
    ref_k, ref_v = host_k.view(np.uint16).copy(), host_v.view(np.uint16).copy()
    c = skv.BlockCache(h, hk, hv, n_blocks=n_blocks, block_rows=br, Hk=Hk, D=D, n_slots=n_slots,
                       max_lookups=S * Hk * n_sel)
    sel = np.stack([np.stack([rng.choice(n_blocks, n_sel, replace=False) for _ in range(Hk)])
                    for _ in range(S)]).astype(np.int32)
    q = wl.normal_f16(rng, (S, 1, H, D))
    q_d, sel_d = dev(q), dev(sel)
    page_ids = torch.empty((S, Hk, n_sel), dtype=torch.int32, device="cuda")
    c.resolve(sel_d, page_ids)                              # make the selected pages resident
    st0 = c.stats()
    # appends at rows of selected (resident) blocks and of other blocks, incl. skipped ones
    chosen = np.unique(np.concatenate([sel[0, 0, :3] * br + rng.integers(0, br, 3),
                                       rng.integers(0, n_blocks * br, 40)]))
    pos = np.concatenate([chosen, [-1]]).astype(np.int32)
    k_new, v_new = wl.new_kv_values(rng, pos.size, Hk, D)
    c.append(dev(k_new), dev(v_new), dev(pos))
    torch.cuda.synchronize()
    assert h.status() == 0
    assert oracle.paged_append(k_new, pos, ref_k, block_rows=br, n_blocks=n_blocks) == 0
    assert oracle.paged_append(v_new, pos, ref_v, block_rows=br, n_blocks=n_blocks) == 0
    assert np.array_equal(hk.numpy().view(np.uint16), ref_k), "host copy (K) differs from the oracle"
    assert np.array_equal(hv.numpy().view(np.uint16), ref_v), "host copy (V) differs from the oracle"
    # every resident page named by the resolve equals its host page
    ids = page_ids.cpu().numpy()
    pk, pv = _pool_pages(skv, h, c, page_ids, br * D * 2)
    host_pages_k = ref_k.reshape(n_blocks * Hk, br * D)
    host_pages_v = ref_v.reshape(n_blocks * Hk, br * D)
    flat_sel = sel.reshape(-1)
    heads = np.broadcast_to(np.arange(Hk)[None, :, None], sel.shape).reshape(-1)
    resident = ids.reshape(-1) < n_slots
    assert resident.any()
    for i in np.nonzero(resident)[0]:
        page = flat_sel[i] * Hk + heads[i]
        assert np.array_equal(pk[i].view(np.uint16), host_pages_k[page]), f"stale resident K page {page}"
        assert np.array_equal(pv[i].view(np.uint16), host_pages_v[page]), f"stale resident V page {page}"
    # attention through the cache: resident pages read as they are, misses fetched
    o, lse = c.attn(q_d, sel_d)
    st1 = c.stats()
    if n_slots >= S * Hk * n_sel:
        assert st1["misses"] == st0["misses"], "every selected page should have stayed resident"
    assert c.check() == 0
    rows = (sel[..., None] * br + np.arange(br, dtype=np.int32)).reshape(S, Hk, -1).astype(np.int32)
    want_o, want_l = oracle_mod.attention(q, D=D, H=H, Hk=Hk, scale=1 / math.sqrt(D), k0=ref_k, v0=ref_v,
                                          n_rows0=n_blocks * br, layout=oracle_mod.PAGED, page_rows=br,
                                          n_keys=rows.shape[-1], kv_rows=rows, rows_per_head=True)
    vmax = float(np.abs(ref_v.view(np.float16).astype(np.float64)).max())
    check_attention(o, lse, want_o, want_l, vmax, "after write-through")
    c.close()
