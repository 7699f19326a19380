"""Parity at the benchmark's full sizes, in the launch configuration that
bench.py times.

* Unified-cache decode (262144-row shared cache, 8 sequences x 32768 rows,
  32 q heads, 8 KV heads, D = 128): every output row against the oracle.
* Block-sparse decode through the block cache, cold and warm, against the
  oracle and bit for bit against an all-resident run split the same way.
* Long-context window + host tail (1,048,576 rows, q8_0 K / q4_0 V, window
  131072, 28 tail tiles of 32768 rows chosen by the library's planner): the
  full call on the GPU; the oracle recomputes every KV head's rows, one head
  group at a time.
"""
import numpy as np
import pytest

from split_kv_flash_attn_gb300 import workloads as wl
from tests.gpu_util import check_attention, dev, head_columns, oracle_one_head, pinned, vmax_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import split_kv_flash_attn_gb300 as m
    return m


def test_unified_cache_full_size(skv, oracle_mod):
    w = wl.unified_decode()
    h = skv.Handle(0)
    o, l = skv.attn_partial(h, dev(w.q), dev(w.k), dev(w.v), Hk=w.Hk, kv_rows=dev(w.kv_rows))
    want_o, want_l = oracle_mod.attention(w.q, D=w.D, H=w.H, Hk=w.Hk, scale=w.scale, k0=w.k, v0=w.v,
                                          n_rows0=w.k.shape[0], k_row_bytes0=w.k.shape[1],
                                          v_row_bytes0=w.v.shape[1], n_keys=w.n_keys, kv_rows=w.kv_rows)
    vmax = float(np.abs(w.v.view(np.float16)).max())
    check_attention(o, l, want_o, want_l, vmax, "unified full")
    h.close()


def test_block_sparse_full_size(skv, oracle_mod):
    """4 sequences x 4 KV heads x 512 of 4096 64-row blocks from a pinned
    paged cache of 262144 rows through a 2048-page block cache (demand above
    capacity): every output row against the oracle, cold and warm, and bit
    for bit against the same call with every page resident."""
    import torch
    w = wl.block_sparse_decode()
    sel = w.extra["sel"]
    h = skv.Handle(0)
    hk, hv = pinned(w.k), pinned(w.v)
    c = skv.BlockCache(h, hk, hv, n_blocks=w.extra["n_blocks"], block_rows=64, Hk=w.Hk, D=w.D,
                       n_slots=w.extra["cache_pages"], max_lookups=sel.size)
    q = dev(w.q)
    o, l = c.attn(q, dev(sel))
    br = w.extra["block_rows"]
    rows = (sel[..., None] * br + np.arange(br, dtype=np.int32)).reshape(w.S, w.Hk, -1).astype(np.int32)
    want_o, want_l = oracle_mod.attention(w.q, D=w.D, H=w.H, Hk=w.Hk, scale=w.scale, k0=w.k, v0=w.v,
                                          n_rows0=w.extra["n_kv"], layout=oracle_mod.PAGED, page_rows=br,
                                          n_keys=rows.shape[-1], kv_rows=rows, rows_per_head=True)
    check_attention(o, l, want_o, want_l, float(np.abs(w.v.view(np.float16)).max()), "block sparse full")
    from tests.test_gpu_bcache import AllResident
    resident = AllResident(skv, h, w, hk, hv, sel.size)
    r_o, r_l = resident(q, sel)
    assert torch.equal(o, r_o) and torch.equal(l, r_l)
    o2, l2 = c.attn(q, dev(sel))                       # warm call: hits and misses mixed
    assert torch.equal(o2, r_o) and torch.equal(l2, r_l)
    resident.close()
    check_attention(o2, l2, want_o, want_l, float(np.abs(w.v.view(np.float16)).max()), "block sparse warm")
    st = c.stats()
    assert st["last_misses"] > 0 and st["last_overflow"] > 0 and st["hits"] > 0
    assert c.check() == 0
    c.close()
    h.close()


def test_long_context_full_size_all_heads(skv, oracle_mod):
    """The whole window + tail call, tail tiles sized by the library's own
    planner (tile_rows = 0 -> skv_plan_tail_tile: 28 tiles of 32768 rows),
    against the oracle on every KV head."""
    w = wl.long_context_decode()
    assert skv.plan_tail_tile(w.k_tail.shape[0], w.k_tail.shape[1] + w.v_tail.shape[1]) == (32768, 28)
    h = skv.Handle(0)
    o, l = skv.attn_window_tail(h, dev(w.q), dev(w.k), dev(w.v), pinned(w.k_tail), pinned(w.v_tail), Hk=w.Hk,
                                k_type=w.k_type, v_type=w.v_type)
    o = o.cpu()
    l = l.cpu()
    G = w.H // w.Hk
    sv = wl.segment_bytes(w.v_type, w.D)
    for kh in range(w.Hk):
        want_o, want_l = oracle_one_head(oracle_mod, w, kh, k_type=w.k_type, v_type=w.v_type, k0=w.k, v0=w.v,
                                         k1=w.k_tail, v1=w.v_tail, n_keys=w.n_keys)
        vmax = max(vmax_of(oracle_mod, w.v_type, head_columns(w.v, kh, sv), w.D),
                   vmax_of(oracle_mod, w.v_type, head_columns(w.v_tail, kh, sv), w.D))
        check_attention(o[:, :, kh * G:(kh + 1) * G], l[:, :, kh * G:(kh + 1) * G], want_o, want_l, vmax,
                        f"long context head {kh}")
    assert h.status() == 0
    h.close()
