"""Ring layout of the block cache (static table block -> block % ring_blocks).

* after a restore, attention over the last cells through the ring equals the
  oracle over the same cells of the host copy, for windows that start mid-block
  and for the whole ring;
* a decode loop (one row appended per step across block boundaries, so newer
  blocks overwrite older ring pages) keeps the ring equal to the host copy;
* after the ring's pages are wiped, a restore brings the same results back
  (bitwise) -- the resume path;
* a window reaching past the ring is rejected, and the table stays static.
"""
import math

import numpy as np
import pytest

import oracle
from split_kv_flash_attn_gb300 import workloads as wl
from tests.gpu_util import check_attention, dev, pinned

pytestmark = pytest.mark.gpu

HK, H, D, BR, NB, R = 4, 16, 128, 64, 64, 8


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


def _oracle_window(oracle_mod, q, ref_k, ref_v, lo, hi):
    S = q.shape[0]
    rows = np.broadcast_to(np.arange(lo, hi, dtype=np.int32), (S, HK, hi - lo)).copy()
    return oracle_mod.attention(q, D=D, H=H, Hk=HK, scale=1 / math.sqrt(D), k0=ref_k, v0=ref_v,
                                n_rows0=NB * BR, layout=oracle_mod.PAGED, page_rows=BR, n_keys=hi - lo,
                                kv_rows=rows, rows_per_head=True)


def _setup(skv, h, seed):
    rng = wl.generator(7, salt=seed)
    host_k = wl.normal_f16(rng, (NB, HK, BR, D))
    host_v = wl.normal_f16(rng, (NB, HK, BR, D))
    hk, hv = pinned(host_k), pinned(host_v)
    c = skv.BlockCache(h, hk, hv, n_blocks=NB, block_rows=BR, Hk=HK, D=D, ring_blocks=R, max_seqs=2)
    return rng, hk, hv, c


def test_ring_restore_and_windows(skv, h, oracle_mod):
    import torch
    rng, hk, hv, c = _setup(skv, h, 1)
    ref_k, ref_v = hk.numpy().view(np.uint16), hv.numpy().view(np.uint16)
    vmax = float(np.abs(hv.numpy().astype(np.float64)).max())
    q = wl.normal_f16(rng, (2, 1, H, D))
    n_keys = 3000                                   # last block 46; the ring holds blocks 39..46
    c.ring_restore(n_keys)
    ring_first = (n_keys - 1) // BR - R + 1
    for window in (1, 100, 256, n_keys - ring_first * BR, 0):
        o, lse = c.ring_attn(dev(q), n_keys, window)
        lo = n_keys - window if window > 0 else ring_first * BR
        want_o, want_l = _oracle_window(oracle_mod, q, ref_k, ref_v, lo, n_keys)
        check_attention(o, lse, want_o, want_l, vmax, f"window {window}")
    with pytest.raises(skv.SplitKVError) as e:
        c.ring_attn(dev(q), n_keys, n_keys - ring_first * BR + 1)
    assert e.value.status == 1
    # short cache: fewer blocks than the ring holds
    c.ring_restore(130)
    o, lse = c.ring_attn(dev(q), 130, 0)
    want_o, want_l = _oracle_window(oracle_mod, q, ref_k, ref_v, 0, 130)
    check_attention(o, lse, want_o, want_l, vmax, "short")
    assert c.check() == 0
    torch.cuda.synchronize()
    c.close()


def test_ring_decode_loop_and_resume(skv, h, oracle_mod):
    import torch
    rng, hk, hv, c = _setup(skv, h, 2)
    ref_k, ref_v = hk.numpy().view(np.uint16).copy(), hv.numpy().view(np.uint16).copy()
    q = wl.normal_f16(rng, (1, 1, H, D))
    q_d = dev(q)
    n_keys, window = 2950, 300
    c.ring_restore(n_keys)
    results = []
    for step in range(140):                         # crosses blocks 46 -> 48 (ring pages of 38, 39 reused)
        k_new, v_new = wl.new_kv_values(rng, 1, HK, D)
        pos = np.array([n_keys], np.int32)
        c.append(dev(k_new), dev(v_new), dev(pos))
        oracle.paged_append(k_new, pos, ref_k, block_rows=BR, n_blocks=NB)
        oracle.paged_append(v_new, pos, ref_v, block_rows=BR, n_blocks=NB)
        n_keys += 1
        o, lse = c.ring_attn(q_d, n_keys, window)
        if step % 20 == 19:
            vmax = float(np.abs(ref_v.view(np.float16).astype(np.float64)).max())
            want_o, want_l = _oracle_window(oracle_mod, q, ref_k, ref_v, n_keys - window, n_keys)
            check_attention(o, lse, want_o, want_l, vmax, f"step {step}")
            results.append((n_keys, o.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert h.status() == 0
    assert np.array_equal(hk.numpy().view(np.uint16), ref_k) and np.array_equal(hv.numpy().view(np.uint16), ref_v)
    # resume: wipe the ring pages, restore from the host copy, same results bitwise
    k_ptr, v_ptr, n_pool, _ = c.pool()
    assert n_pool == R * HK
    wipe = torch.full((n_pool,), -1, dtype=torch.int32, device="cuda")
    for ptr in (k_ptr, v_ptr):
        skv.gather_rows(h, ptr, wipe, row_bytes=BR * D * 2, out=ptr)
    o_w, _ = c.ring_attn(q_d, n_keys, window)
    assert not torch.equal(o_w, results[-1][1])
    c.ring_restore(n_keys)
    o2, l2 = c.ring_attn(q_d, n_keys, window)
    assert torch.equal(o2, results[-1][1]) and torch.equal(l2, results[-1][2])
    assert c.check() == 0
    c.close()


def test_ring_rejects_resolve(skv, h):
    _, _, _, c = _setup(skv, h, 3)
    sel = dev(np.zeros((1, HK, 1), np.int32))
    with pytest.raises(skv.SplitKVError) as e:
        c.resolve(sel)
    assert e.value.status == 2
    c.close()
