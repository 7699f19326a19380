// planner.cu -- residency planning on the host: how many position cells stay
// resident in device memory (the window), and how large the streamed tail's
// tiles are.  Pure integer logic; no GPU needed.
//
// Window ("Rolling KV -- position-windowed KV residency", the position-axis
// residency sizing of the KV cache): budget = min(free, target) minus a
// reserve; the whole cache stays resident when it fits; otherwise the window
// is the largest cell count that fits, rounded down to the alignment (the
// larger of the cache padding and 256, the attention kernels' key stride), no
// smaller than one alignment step and leaving at least one step of tail.
//
// Tail tiles (same page, streaming forward's tile sizing): tiles of about
// target_keys keys (32768 there, to keep launches few), enlarged in count
// until n_slots slots of one tile fit the slot-memory cap (512 MiB there), at
// most one tile per alignment block, each tile a whole number of blocks.
#include "internal.h"

extern "C" {

int skv_plan_window(int64_t per_cell_bytes, int64_t kv_size, int64_t free_bytes, int64_t target_bytes,
                    int64_t reserve_bytes, int32_t n_pad, int64_t *window_cells)
{
    if (!window_cells || per_cell_bytes < 0 || kv_size < 0 || free_bytes < 0 || target_bytes < 0 ||
        reserve_bytes < 0 || n_pad < 0)
        return SKV_EINVAL;
    if (kv_size == 0 || per_cell_bytes == 0) {
        *window_cells = kv_size;
        return SKV_OK;
    }
    int64_t budget = free_bytes;
    if (target_bytes > 0 && target_bytes < budget) budget = target_bytes;
    budget = budget > reserve_bytes ? budget - reserve_bytes : 0;
    if (per_cell_bytes <= budget / kv_size) {          // per_cell * kv_size <= budget, without overflow
        *window_cells = kv_size;
        return SKV_OK;
    }
    const int64_t pad = n_pad ? n_pad : 32;
    const int64_t align = pad >= 256 ? pad : 256;
    int64_t cells = budget / per_cell_bytes;
    cells = cells / align * align;
    if (cells < align) cells = align;
    if (kv_size > align && cells > kv_size - align) {
        cells = (kv_size - align) / align * align;
        if (cells < align) cells = align;
    }
    *window_cells = cells;
    return SKV_OK;
}

int skv_plan_tail_tile(int64_t n_keys, int64_t per_key_bytes, int32_t n_slots, int64_t slot_cap_bytes,
                       int64_t target_keys, int32_t align, int64_t *tile_rows, int32_t *n_tiles)
{
    if (!tile_rows || !n_tiles || n_keys < 0 || per_key_bytes < 0 || n_slots <= 0 || slot_cap_bytes < 0 ||
        target_keys <= 0 || align <= 0)
        return SKV_EINVAL;
    if (n_keys == 0) {
        *tile_rows = align;
        *n_tiles = 0;
        return SKV_OK;
    }
    const int64_t n_blk = (n_keys + align - 1) / align;
    int64_t tiles = (n_keys + target_keys - 1) / target_keys;
    const int64_t denom = per_key_bytes * n_slots;
    int64_t max_keys = denom == 0 ? n_keys : slot_cap_bytes / denom;
    if (max_keys < align) max_keys = align;
    const int64_t tiles_cap = (n_keys + max_keys - 1) / max_keys;
    if (tiles < tiles_cap) tiles = tiles_cap;
    if (tiles < 1) tiles = 1;
    if (tiles > n_blk) tiles = n_blk;
    const int64_t blk_per_tile = (n_blk + tiles - 1) / tiles;
    const int64_t rows = blk_per_tile * align;
    const int64_t count = (n_keys + rows - 1) / rows;
    if (count > 0x7fffffff) return SKV_EUNSUPPORTED;
    *tile_rows = rows;
    *n_tiles = static_cast<int32_t>(count);
    return SKV_OK;
}

}  // extern "C"
