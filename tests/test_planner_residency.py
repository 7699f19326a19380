"""Residency planning (host logic, no GPU): the resident window and the tail
tiles.  The library's planner is written as closed forms of the constraints;
oracle/planner.py restates the Rolling KV page's rules step by step in the
page's order.  The two codings must agree on random inputs (bit-exact), both
must meet the constraints (alignment, budget, a step of tail, coverage, the
slot cap), and both must give the numbers the page states: 32768-key tiles
(the coarsening from 2048 keys, which gave 128 tiles at 256k keys), four slots
of a tile within 512 MiB, windows aligned to the 256-key stride, and the
long-context workload's 32768-row tiles of raw q8_0/q4_0 bytes."""
import numpy as np
import pytest

from oracle import planner as ref

MIB = 1 << 20


@pytest.fixture(scope="module")
def skv():
    from split_kv_flash_attn_gb300 import build as b
    b.build()
    import split_kv_flash_attn_gb300 as m
    return m


def test_window_fits_whole_cache(skv):
    assert skv.plan_window(1024, 100000, 80 << 30) == 100000
    assert skv.plan_window(0, 5, 0) == 5


def test_window_rounds_down_and_clamps(skv):
    # 10 GiB free, 1.5 GiB reserve, 1 MiB per cell -> 8704 cells, already a multiple of 256
    assert skv.plan_window(MIB, 1 << 20, 10 << 30) == 8704
    # a budget below one cell -> one 256-cell step
    assert skv.plan_window(MIB, 1 << 20, 1536 * MIB + 5) == 256
    # nearly everything fits -> one step of tail is left
    assert skv.plan_window(1024, 10000, 1536 * MIB + 9999 * 1024) == 9728
    # target caps the free memory
    assert skv.plan_window(MIB, 1 << 20, 80 << 30, target_bytes=2048 * MIB) == 512
    # padding above 256 sets the alignment
    assert skv.plan_window(MIB, 1 << 20, 10 << 30, n_pad=1024) == 8192


def test_window_non_power_of_two_padding(skv):
    # the alignment must be a multiple of both the padding and the 256-key
    # stride: lcm(384, 256) = 768, where the page's larger-of-the-two rule
    # (written for power-of-two paddings) would give 384
    got = skv.plan_window(MIB, 1 << 20, 10 << 30, n_pad=384)
    assert got % 768 == 0 and got == 8448
    rng = np.random.default_rng(2)
    for _ in range(2000):
        per_cell = int(rng.integers(1, 1 << 22))
        kv = int(rng.integers(1, 1 << 21))
        free = int(rng.integers(0, 1 << 40))
        n_pad = int(rng.integers(1, 2000))
        step = np.lcm(n_pad, 256)
        got = skv.plan_window(per_cell, kv, free, 0, 1536 * MIB, n_pad)
        budget = max(0, free - 1536 * MIB)
        if per_cell * kv <= budget:
            assert got == kv
            continue
        assert got % step == 0 and got >= step
        if got > step:
            assert got * per_cell <= budget          # above one step only while it fits
        if kv > step:
            assert got <= max(step, kv - step)       # a step of tail stays (or one step)


def test_window_matches_restated_rules(skv):
    rng = np.random.default_rng(0)
    for _ in range(3000):
        per_cell = int(rng.integers(0, 1 << 22))
        kv = int(rng.integers(0, 1 << 21))
        free = int(rng.integers(0, 1 << 40))
        target = int(rng.choice([0, int(rng.integers(0, 1 << 38))]))
        reserve = int(rng.choice([0, 1536 * MIB, int(rng.integers(0, 1 << 32))]))
        n_pad = int(rng.choice([0, 32, 256, 512]))
        got = skv.plan_window(per_cell, kv, free, target, reserve, n_pad)
        assert got == ref.window_cells(per_cell, kv, free, target, reserve, n_pad)
        if 0 < got < kv:
            assert got % max(n_pad or 32, 256) == 0


def test_tail_tiles_page_numbers(skv):
    # 262144 keys at the old 2048-key target: 128 tiles (the launch slack the page removes)
    assert skv.plan_tail_tile(262144, 64, target_keys=2048) == (2048, 128)
    # at the 32768-key target: 8 tiles
    assert skv.plan_tail_tile(262144, 64) == (32768, 8)
    # long-context tail: 917504 rows of 1088 + 576 raw bytes -> 28 tiles of 32768 rows
    assert skv.plan_tail_tile(917504, 1088 + 576) == (32768, 28)
    # fp16 rows of 8 KV heads x 128 x 2 (K+V) = 4 KiB per key: 4 slots x 32768 keys = 512 MiB, fits
    assert skv.plan_tail_tile(65536, 4096) == (32768, 2)
    # 8 KiB per key: the 512 MiB cap halves the tile
    assert skv.plan_tail_tile(65536, 8192) == (16384, 4)


def test_tail_tiles_match_restated_rules(skv):
    rng = np.random.default_rng(1)
    for _ in range(3000):
        n = int(rng.integers(0, 1 << 22))
        per_key = int(rng.integers(0, 1 << 16))
        slots = int(rng.integers(1, 5))
        cap = int(rng.integers(0, 1 << 32))
        target = int(rng.integers(1, 1 << 17))
        align = int(rng.choice([1, 64, 128, 256]))
        rows, tiles = skv.plan_tail_tile(n, per_key, slots, cap, target, align)
        assert (rows, tiles) == ref.tail_tile(n, per_key, slots, cap, target, align)
        if n:
            assert rows % align == 0 and tiles * rows >= n and (tiles - 1) * rows < n
            # no more tiles than the target count or the slot cap asks for
            # (whole blocks, spread evenly), nor fewer than the target asks for
            n_blk = -(-n // align)
            cap_keys = max(align, cap // (per_key * slots)) if per_key else n
            want = min(n_blk, max(1, -(-n // target), -(-n // cap_keys)))
            assert tiles <= want and -(-n_blk // tiles) == -(-n_blk // want)
