"""Residency planning rules restated in plain Python (test infrastructure).

Follows the position-axis residency sizing and the tail-tile sizing of the
"Rolling KV -- position-windowed KV residency" page, step by step in the
page's order, so that the library's C planner can be compared with it bit for
bit on any inputs.
"""


def window_cells(per_cell, kv_size, free, target, reserve, n_pad):
    """Cells [0, C) kept resident; kv_size when everything fits."""
    if kv_size == 0 or per_cell == 0:
        return kv_size
    budget = free
    if target > 0:
        budget = min(budget, target)
    budget = budget - reserve if budget > reserve else 0
    if per_cell * kv_size <= budget:
        return kv_size
    pad = n_pad if n_pad else 32
    align = max(pad, 256)             # lcm with the 256-key stride for power-of-two paddings
    cells = budget // per_cell
    cells = (cells // align) * align  # round down
    if cells < align:
        cells = align                 # never below one stride
    if kv_size > align and cells > kv_size - align:
        cells = ((kv_size - align) // align) * align   # keep one stride of tail
        if cells < align:
            cells = align
    return cells


def tail_tile(n_keys, per_key, n_slots, slot_cap, target_keys, align):
    """(tile_rows, n_tiles) of the streamed tail."""
    if n_keys == 0:
        return align, 0
    n_blk = -(-n_keys // align)
    tiles = -(-n_keys // target_keys)
    denom = per_key * n_slots
    max_keys = n_keys if denom == 0 else slot_cap // denom
    max_keys = max(max_keys, align)
    tiles = max(tiles, -(-n_keys // max_keys))
    tiles = min(max(tiles, 1), n_blk)
    rows = -(-n_blk // tiles) * align
    return rows, -(-n_keys // rows)
