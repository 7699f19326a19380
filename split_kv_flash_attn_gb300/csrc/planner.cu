// planner.cu -- residency planning on the host: how many position cells stay
// resident in device memory (the window), and how large the streamed tail's
// tiles are.  Pure integer logic; no GPU needed.
//
// Both answers are closed forms of the constraints the "Rolling KV --
// position-windowed KV residency" page puts on them (position-axis residency
// sizing; streaming forward's tile sizing):
//
//  window: the largest multiple of the alignment whose cells fit the budget,
//          never below one alignment step, and -- when the cache is longer
//          than one step -- never above the last aligned cell count that still
//          leaves a whole step of tail.  The alignment is a multiple of both the
//          cache padding and the attention kernels' 256-key stride, i.e. their
//          least common multiple (the page takes the larger of the two, which
//          is the same number for the power-of-two paddings it uses).
//  tiles:  as many tiles as the larger of two demands -- one tile per target
//          count of keys, and enough tiles that n_slots copies of one tile fit
//          the slot-memory cap -- but no more tiles than alignment blocks; the
//          blocks are then spread evenly, so every tile but the last holds the
//          same whole number of blocks.
#include "internal.h"

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t gcd64(int64_t a, int64_t b)
{
    while (b) {
        const int64_t r = a % b;
        a = b;
        b = r;
    }
    return a;
}

int64_t clamp64(int64_t x, int64_t lo, int64_t hi) { return x < lo ? lo : (x > hi ? hi : x); }

}  // namespace

extern "C" {

int skv_plan_window(int64_t per_cell_bytes, int64_t kv_size, int64_t free_bytes, int64_t target_bytes,
                    int64_t reserve_bytes, int32_t n_pad, int64_t *window_cells)
{
    if (!window_cells || per_cell_bytes < 0 || kv_size < 0 || free_bytes < 0 || target_bytes < 0 ||
        reserve_bytes < 0 || n_pad < 0)
        return SKV_EINVAL;
    // Nothing to size: an empty cache, or cells that cost nothing.
    if (kv_size == 0 || per_cell_bytes == 0) {
        *window_cells = kv_size;
        return SKV_OK;
    }
    const int64_t cap = target_bytes > 0 ? (target_bytes < free_bytes ? target_bytes : free_bytes) : free_bytes;
    const int64_t budget = cap > reserve_bytes ? cap - reserve_bytes : 0;
    const int64_t fit = budget / per_cell_bytes;              // whole cells the budget holds
    if (fit >= kv_size) {                                     // the whole cache stays resident
        *window_cells = kv_size;
        return SKV_OK;
    }
    const int64_t pad = n_pad > 0 ? n_pad : 32;
    const int64_t step = pad / gcd64(pad, 256) * 256;         // lcm(pad, 256)
    const int64_t lo = step;                                  // at least one step resident
    const int64_t hi = kv_size > step ? (kv_size - step) / step * step : 0;   // a step of tail stays
    const int64_t want = fit / step * step;
    *window_cells = kv_size > step ? clamp64(want, lo, hi > lo ? hi : lo) : (want > lo ? want : lo);
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
    const int64_t blocks = ceil_div(n_keys, align);
    // Most keys one tile may hold so that n_slots tiles fit the cap; a single
    // alignment block is allowed even when it alone exceeds the cap.
    const int64_t per_tile_slots = per_key_bytes * n_slots;
    const int64_t cap_keys =
        per_tile_slots == 0 ? n_keys : (slot_cap_bytes / per_tile_slots > align ? slot_cap_bytes / per_tile_slots : align);
    const int64_t by_target = ceil_div(n_keys, target_keys);
    const int64_t by_cap = ceil_div(n_keys, cap_keys);
    const int64_t tiles = clamp64(by_target > by_cap ? by_target : by_cap, 1, blocks);
    const int64_t rows = ceil_div(blocks, tiles) * align;     // blocks spread evenly
    const int64_t count = ceil_div(n_keys, rows);
    if (count > 0x7fffffff) return SKV_EUNSUPPORTED;
    *tile_rows = rows;
    *n_tiles = static_cast<int32_t>(count);
    return SKV_OK;
}

}  // extern "C"
