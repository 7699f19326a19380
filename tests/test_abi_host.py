"""Host-only checks of the C ABI (no GPU): the library builds and loads, it
exports every function include/splitkv.h declares, and the pure-host split
planner keeps its contract."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from split_kv_flash_attn_gb300 import build as b
    b.build()
    from split_kv_flash_attn_gb300 import _lib
    return _lib.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(skv_\w+)\s*\(", txt, re.M))
    return names


def test_header_declares_entry_points():
    names = _declared()
    for must in ("skv_attn_partial", "skv_attn_combine", "skv_attn_window_tail",
                 "skv_kv_dequant_q8_0", "skv_kv_dequant_q4_0"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in sorted(_declared()) if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_lists_every_export():
    from split_kv_flash_attn_gb300 import _lib
    assert set(_lib.EXPORTS) == _declared()


def test_status_strings(lib):
    assert lib.skv_status_string(0) == b"ok"
    assert b"page-locked" in lib.skv_status_string(3)
    assert lib.skv_status_string(99) == b"unknown status"


def test_null_handle_rejected(lib):
    assert lib.skv_attn_combine(None, 1, None, None, 1, 64, None, None, None) == 1
    assert lib.skv_destroy(None) == 0


def _plan(n_keys, units, sms=152, ctas=2, tile=64, max_split=0):
    from split_kv_flash_attn_gb300 import plan_splits
    return plan_splits(n_keys, units, sms, ctas, tile, max_split)


@pytest.mark.parametrize("n_keys,units,max_split", [
    (32768, 64, 2048), (131072, 8, 0), (32768, 8, 0), (256, 1, 0), (1, 1, 0), (65, 3, 0),
    (1000003, 7, 2048), (4096, 1000, 2048), (512 * 64, 16, 2048), (64, 152 * 2, 0)])
def test_planner_covers_range(n_keys, units, max_split):
    sl, ns = _plan(n_keys, units, max_split=max_split)
    assert sl % 64 == 0 and sl > 0
    assert ns * sl >= n_keys and (ns - 1) * sl < n_keys     # covers, no empty split
    if max_split:
        assert sl <= max_split


def test_planner_fills_waves_for_unified_cache():
    # 64 (sequence, KV head) units of 32768 gathered keys on 152 SMs x 2 CTAs:
    # 19 splits of 1728 keys make exactly four waves of 304 CTAs.
    sl, ns = _plan(32768, 64, max_split=2048)
    assert (sl, ns) == (1728, 19)
    assert (64 * ns) % 304 == 0


def test_planner_window_one_wave():
    sl, ns = _plan(131072, 8)
    assert 8 * ns == 304 or (8 * ns) % 304 == 0


def test_planner_empty_and_bad_args():
    from split_kv_flash_attn_gb300 import SplitKVError, plan_splits
    assert plan_splits(0, 4, 152, 2)[1] == 0
    with pytest.raises(SplitKVError):
        plan_splits(10, 0, 152, 2)
    with pytest.raises(SplitKVError):
        plan_splits(10, 1, 152, 2, tile=64, max_split=32)


def test_prefill_plan_head_and_tail():
    # 512 tokens x 32 q heads over 8 KV heads make 128 query tiles (16 per KV
    # head) over 32768 keys on 152 SMs: one split leaves 24 SMs idle.  A head
    # of 227 tiles per query tile and a tail of 29 let the 24 free SMs run
    # six tails each (6 x (29 + 10) = 234 tile-times) within one head (227 +
    # 10 = 237), against 256 + 10 for one split.  Over q8_0 keys and values
    # (4 tiles of fixed cost): 223 + 33, against seven even splits of 37
    # tiles in six waves (6 x 41 = 246).  Over q8_0 keys with q4_0 values the
    # CTAs take query-tile pairs (64 units, 10 tiles of fixed cost): two heads
    # of 113 tiles per pair fill 128 SMs and the 24 others run the 64 tails of
    # 30, three each (3 x 40 = 120 <= 113 + 10), against 128 + 10 for two
    # even splits.  Eight sequences of 64 tokens through row lists: 128 units
    # again.
    from split_kv_flash_attn_gb300 import F16, Q4_0, Q8_0, plan_prefill_splits
    assert plan_prefill_splits(1, 512, 32, 8, 32768, 152) == (227 * 128, 2, 256)
    assert plan_prefill_splits(1, 512, 32, 8, 32768, 152, k_type=Q8_0, v_type=Q8_0) == (223 * 128, 2, 256)
    assert plan_prefill_splits(1, 512, 32, 8, 32768, 152, k_type=Q8_0, v_type=Q4_0) == (113 * 128, 3, 192)
    assert plan_prefill_splits(8, 64, 32, 8, 32768, 152, rows=True) == (227 * 128, 2, 256)
    # row lists of quantised rows stay one query tile a CTA
    assert plan_prefill_splits(1, 512, 32, 8, 32768, 152, k_type=Q8_0, v_type=Q4_0, rows=True)[2] % 128 == 0


@pytest.mark.parametrize("S,nq,n_keys", [
    (1, 512, 32768), (1, 512 * 19 // 16, 32768), (4, 512, 32768), (1, 1024, 65536), (8, 64, 1000), (1, 32, 128),
    (2, 80, 129), (1, 152 * 8, 5 * 128), (1, 480, 1 << 20), (1, 64, 32768)])
@pytest.mark.parametrize("kt,vt", [(0, 0), (1, 1), (1, 2), (2, 2), (2, 1)])
def test_prefill_plan_properties(S, nq, n_keys, kt, vt):
    from split_kv_flash_attn_gb300 import plan_prefill_splits
    H, Hk = 32, 8
    sl, ns, nc = plan_prefill_splits(S, nq, H, Hk, n_keys, 152, k_type=kt, v_type=vt)
    tiles = -(-n_keys // 128)
    q_tiles = Hk * -(-nq * (H // Hk) // 128)
    pairs = kt != 0 and vt == 2 and q_tiles // Hk >= 2
    units = S * (Hk * -(-(q_tiles // Hk) // 2) if pairs else q_tiles)
    assert nc == units * ns
    assert sl % 128 == 0 and sl > 0
    assert ns * sl >= n_keys and (ns - 1) * sl < n_keys     # covers, no empty split
    if units >= 152:
        assert ns == 1 or 2 * sl <= n_keys + 128 * (ns - 1)   # no heads-and-tail plan once the SMs are full
    head, tail = sl // 128, tiles - (ns - 1) * (sl // 128)
    if ns >= 2 and units * (ns - 1) < 152 and 2 * tail < head:
        # heads and a much shorter tail: the free SMs' tails fit beside the heads
        c = 10 if (kt == 0 or pairs) else 4
        k = -(-units // (152 - units * (ns - 1)))
        assert k * (tail + c) <= head + c + k * (ns - 1) + 1


def test_prefill_plan_bad_args():
    from split_kv_flash_attn_gb300 import SplitKVError, plan_prefill_splits
    assert plan_prefill_splits(1, 512, 32, 8, 0, 152)[1] == 0
    for args, kw in (((1, 512, 32, 8, -1, 152), {}), ((1, 512, 32, 8, 10, 0), {}), ((0, 512, 32, 8, 10, 152), {}),
                     ((1, 512, 32, 7, 10, 152), {}), ((1, 512, 32, 8, 10, 152), {"D": 64}),
                     ((1, 8, 32, 8, 10, 152), {})):
        with pytest.raises(SplitKVError):
            plan_prefill_splits(*args, **kw)


def test_product_path_fails_loudly_without_library(tmp_path):
    from split_kv_flash_attn_gb300 import _lib
    with pytest.raises(ImportError):
        _lib.load(str(tmp_path / "missing.so"))


def test_product_package_never_imports_oracle():
    pkg = os.path.join(ROOT, "split_kv_flash_attn_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f
                assert "splitkv_oracle" not in txt, f
