"""Block cache (selection-driven residency over a pinned paged host copy).

Parity is against the oracle over the selected rows, and bitwise against the
same call with every page resident, the check the Strata KV-streaming parity
test makes: a second cache that holds all pages, called twice with the
selection so that the second call reads every page from its pool.  The
resolve-then-attend path (skv_bcache_resolve, then skv_attn_paged through the
pool) is checked bitwise against skv_attn_paged over the whole cache on the
device (identity page table).  After every resolve the page table and the
slot map must be inverse maps, and the counters must add up.  The residency
decisions themselves (the slot of every page, the overflow, the hand) are
compared call by call with a plain sequential CLOCK model of the page's
resolve rules (oracle/bcache_model.py)."""
import math

import numpy as np
import pytest

from oracle.bcache_model import ClockCache
from split_kv_flash_attn_gb300 import workloads as wl
from tests.gpu_util import check_attention, dev, pinned

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


class AllResident:
    """The same block-cache call with every page resident: a cache with a slot
    for every page, called twice with the selection (the first call fetches
    what is not resident yet, the second reads every page from the pool)."""

    def __init__(self, skv, h, w, hk, hv, max_lookups):
        self.c = skv.BlockCache(h, hk, hv, n_blocks=w.extra["n_blocks"], block_rows=w.extra["block_rows"], Hk=w.Hk,
                                D=w.D, n_slots=w.extra["n_blocks"] * w.Hk, max_lookups=max_lookups)

    def __call__(self, q_d, sel):
        self.c.attn(q_d, dev(sel))
        o, l = self.c.attn(q_d, dev(sel))
        assert self.c.stats()["last_misses"] == 0
        return o, l

    def close(self):
        self.c.close()


def _identity(skv, h, w, q_d, sel, k_full, v_full):
    """skv_attn_paged with every page resident on the device (identity page
    table: page id = block * Hk + head)."""
    ids = (sel * w.Hk + np.arange(w.Hk, dtype=np.int32)[None, :, None]).astype(np.int32)
    return skv.attn_paged(h, q_d, k_full, v_full, dev(ids), Hk=w.Hk, page_rows=w.extra["block_rows"])


def _resolved(skv, h, c, w, q_d, sel):
    """skv_bcache_resolve, then skv_attn_paged through the cache's pool."""
    import torch
    ids = torch.empty(sel.shape, dtype=torch.int32, device="cuda")
    c.resolve(dev(sel), ids)
    k_pool, v_pool, _, _ = c.pool()
    return skv.attn_paged(h, q_d, k_pool, v_pool, ids, Hk=w.Hk, page_rows=w.extra["block_rows"])


def _oracle(oracle_mod, w, sel):
    br = w.extra["block_rows"]
    rows = np.where(sel[..., None] >= 0, sel[..., None] * br + np.arange(br, dtype=np.int32), -1)
    rows = rows.reshape(sel.shape[0], sel.shape[1], -1)
    return oracle_mod.attention(w.q, D=w.D, H=w.H, Hk=w.Hk, scale=w.scale, k0=w.k, v0=w.v,
                                n_rows0=w.extra["n_kv"], layout=oracle_mod.PAGED, page_rows=br,
                                n_keys=rows.shape[-1], kv_rows=rows.astype(np.int32), rows_per_head=True)


@pytest.mark.parametrize("n_slots", [128, 1024])
def test_block_cache_cold_warm_drift(skv, h, oracle_mod, n_slots):
    import torch
    w = wl.block_sparse_decode(n_kv=64 * 512, S=4, H=32, Hk=4, D=128, n_sel=64, cache_pages=n_slots)
    sel = w.extra["sel"]
    n_blocks = w.extra["n_blocks"]
    hk, hv = pinned(w.k), pinned(w.v)
    c = skv.BlockCache(h, hk, hv, n_blocks=n_blocks, block_rows=64, Hk=w.Hk, D=w.D, n_slots=n_slots,
                       max_lookups=w.S * w.Hk * sel.shape[-1])
    q_d = dev(w.q)
    vmax = float(np.abs(w.v.view(np.float16)).max())
    lookups = w.S * w.Hk * sel.shape[-1]
    distinct = len({(int(b), k) for s in range(w.S) for k in range(w.Hk) for b in sel[s, k]})
    resident = AllResident(skv, h, w, hk, hv, lookups)

    o0, l0 = c.attn(q_d, dev(sel))                            # cold
    want_o, want_l = _oracle(oracle_mod, w, sel)
    check_attention(o0, l0, want_o, want_l, vmax, "cold")
    r_o, r_l = resident(q_d, sel)
    assert torch.equal(o0, r_o) and torch.equal(l0, r_l), "cold call differs from the all-resident run"
    assert c.check() == 0
    st = c.stats()
    assert st["calls"] == 1 and st["lookups"] == lookups and st["hits"] == 0
    assert st["misses"] == distinct and st["overflow"] == max(0, distinct - n_slots)

    o1, l1 = c.attn(q_d, dev(sel))                            # warm, same selection
    r_o, r_l = resident(q_d, sel)
    assert torch.equal(o1, r_o) and torch.equal(l1, r_l), "warm call differs from the all-resident run"
    check_attention(o1, l1, want_o, want_l, vmax, "warm")
    assert c.check() == 0
    st1 = c.stats()
    new_hits = st1["hits"] - st["hits"]
    new_miss = st1["misses"] - st["misses"]
    if n_slots >= distinct:
        assert new_miss == 0 and new_hits == lookups      # everything stayed resident
    else:
        assert 0 < new_miss < distinct and new_hits > 0
    assert st1["calls"] == 2 and st1["lookups"] == 2 * lookups

    rng = np.random.default_rng(55)
    cur = sel
    for step in range(3):                                     # drift: 10% of the blocks redrawn per step
        cur = wl.redraw_selection(cur, n_blocks, 0.1, rng)
        o2, l2 = c.attn(q_d, dev(cur))
        r_o, r_l = resident(q_d, cur)
        assert torch.equal(o2, r_o) and torch.equal(l2, r_l), f"drift step {step}"
        assert c.check() == 0
    want_o, want_l = _oracle(oracle_mod, w, cur)
    check_attention(o2, l2, want_o, want_l, vmax, "drift")

    c.reset()
    o3, l3 = c.attn(q_d, dev(sel))                            # after a reset: cold again, the same decisions
    assert torch.equal(o3, o0) and torch.equal(l3, l0)
    st3 = c.stats()
    assert st3["calls"] == 1 and st3["hits"] == 0

    # resolve, then paged attention through the pool (the path for shapes the
    # call does not fuse): bitwise the same as over the whole cache on the device
    k_full, v_full = dev(w.k), dev(w.v)
    for sl in (sel, cur):
        p_o, p_l = _resolved(skv, h, c, w, q_d, sl)
        i_o, i_l = _identity(skv, h, w, q_d, sl, k_full, v_full)
        assert torch.equal(p_o, i_o) and torch.equal(p_l, i_l), "resolve + paged attention differs"
    assert c.check() == 0
    resident.close()
    c.close()


@pytest.mark.parametrize("n_slots,D", [(40, 128), (4096, 128), (40, 64)])
def test_block_cache_repeats_and_absent_blocks(skv, h, oracle_mod, n_slots, D):
    """Selections that name a block twice in one list (a later lookup of a
    page the same work item fetches), name the same blocks in every list, and
    hold absent entries (-1, and ids past the cache): against the oracle, and
    bit for bit against the same call with every page resident, cold and
    warm; 40 slots overflow, 4096 hold everything; head dims 128 and 64."""
    import torch
    w = wl.block_sparse_decode(n_kv=64 * 256, S=3, H=16, Hk=2, D=D, n_sel=40, cache_pages=n_slots)
    n_blocks = w.extra["n_blocks"]
    sel = w.extra["sel"].copy()
    sel[0, 0, 3] = sel[0, 0, 1]                 # same work item (8 pages a work item)
    sel[0, 1, 30] = sel[0, 1, 2]                # a later work item of the same list
    sel[1, 0, :10] = sel[0, 0, :10]             # the first lookups are in list (0, 0)
    sel[2, 1, 5] = -1
    sel[2, 1, 17] = n_blocks + 3                # past the cache: absent
    sel[1, 1, 39] = -1
    hk, hv = pinned(w.k), pinned(w.v)
    lookups = w.S * w.Hk * sel.shape[-1]
    c = skv.BlockCache(h, hk, hv, n_blocks=n_blocks, block_rows=64, Hk=w.Hk, D=w.D, n_slots=n_slots,
                       max_lookups=lookups)
    resident = AllResident(skv, h, w, hk, hv, lookups)
    q_d = dev(w.q)
    vmax = float(np.abs(w.v.view(np.float16)).max())
    want_o, want_l = _oracle(oracle_mod, w, np.where(sel < n_blocks, sel, -1))
    r_o, r_l = resident(q_d, sel)
    for what in ("cold", "warm"):
        o, l = c.attn(q_d, dev(sel))
        torch.cuda.synchronize()
        assert h.status() == 0
        check_attention(o, l, want_o, want_l, vmax, what)
        assert torch.equal(o, r_o) and torch.equal(l, r_l), f"{what} call differs from the all-resident run"
        assert c.check() == 0
    resident.close()
    c.close()


@pytest.mark.parametrize("n_slots", [96, 700, 5000])
def test_resolve_matches_clock_model(skv, h, n_slots):
    """Every resolve's page ids and counters against the plain sequential
    CLOCK model (oracle/bcache_model.py): cold, warm, three drift steps, a
    selection of already-resident pages, a reset, cold again.  96 slots wrap
    the sweep and overflow, 700 take cold slots only after the first calls,
    5000 hold everything."""
    import torch
    w = wl.block_sparse_decode(n_kv=64 * 512, S=4, H=32, Hk=4, D=128, n_sel=64, cache_pages=n_slots)
    n_blocks, Hk = w.extra["n_blocks"], w.Hk
    c = skv.BlockCache(h, pinned(w.k), pinned(w.v), n_blocks=n_blocks, block_rows=64, Hk=Hk, D=w.D,
                       n_slots=n_slots, max_lookups=w.S * Hk * 64)
    model = ClockCache(n_blocks * Hk, n_slots)
    rng = np.random.default_rng(31)
    sels = [w.extra["sel"], w.extra["sel"]]
    for _ in range(3):
        sels.append(wl.redraw_selection(sels[-1], n_blocks, 0.1, rng))
    sels.append(np.ascontiguousarray(sels[-1][:, :, :16]))
    sels += ["reset", w.extra["sel"]]
    for i, sel in enumerate(sels):
        if isinstance(sel, str):
            c.reset()
            model.reset()
            continue
        ids = torch.empty(sel.shape, dtype=torch.int32, device="cuda")
        c.resolve(dev(sel), ids)
        pages = (sel.astype(np.int64) * Hk + np.arange(Hk)[None, :, None]).reshape(-1).tolist()
        want = np.array(model.resolve(pages), dtype=np.int32).reshape(sel.shape)
        assert np.array_equal(ids.cpu().numpy(), want), f"call {i}: page ids differ from the CLOCK model"
        st = c.stats()
        assert (st["calls"], st["lookups"], st["hits"], st["misses"], st["overflow"]) == \
            (model.calls, model.lookups, model.hits, model.misses, model.overflow), f"call {i}: counters"
        assert c.check() == 0
    c.close()


def test_paged_attention_padding_pages(skv, h, oracle_mod):
    import torch
    rng = np.random.default_rng(7)
    Hk, D, br, n_pages, S, H = 2, 128, 64, 40, 3, 8
    pool_k = rng.standard_normal((n_pages, br, D)).astype(np.float16)
    pool_v = rng.standard_normal((n_pages, br, D)).astype(np.float16)
    ids = rng.integers(0, n_pages, size=(S, Hk, 12)).astype(np.int32)
    ids[0, 0, 5:] = -1
    ids[1, :, :] = -1
    q = rng.standard_normal((S, 1, H, D)).astype(np.float16)
    o, l = skv.attn_paged(h, dev(q), dev(pool_k), dev(pool_v), dev(ids), Hk=Hk, page_rows=br)
    # oracle: the pool as a paged cache with Hk = 1 (one head per page); rows per (s, k)
    rows = np.where(ids[..., None] >= 0, ids[..., None] * br + np.arange(br), -1).reshape(S, Hk, -1)
    want_o = np.zeros((S, 1, H, D))
    want_l = np.zeros((S, 1, H))
    G = H // Hk
    for k in range(Hk):
        qk = np.ascontiguousarray(q[:, :, k * G:(k + 1) * G])
        oo, ll = oracle_mod.attention(qk, D=D, H=G, Hk=1, scale=1 / math.sqrt(D), k0=pool_k, v0=pool_v,
                                      n_rows0=n_pages * br, k_row_bytes0=2 * D, v_row_bytes0=2 * D,
                                      n_keys=rows.shape[-1], kv_rows=np.ascontiguousarray(rows[:, k]).astype(np.int32))
        want_o[:, :, k * G:(k + 1) * G] = oo
        want_l[:, :, k * G:(k + 1) * G] = ll
    check_attention(o, l, want_o, want_l, float(np.abs(pool_v).max()), "paged")
    assert torch.all(torch.isneginf(l[1]))


def test_block_cache_rejects_pageable_host_copy(skv, h):
    import torch
    k = torch.zeros((4, 2, 64, 128), dtype=torch.float16)
    with pytest.raises(skv.SplitKVError) as e:
        skv.BlockCache(h, k, k, n_blocks=4, block_rows=64, Hk=2, D=128, n_slots=2, max_lookups=8)
    assert e.value.status == 3
