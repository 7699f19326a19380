// internal.h -- handle layout and kernel launchers shared by the library's
// translation units (not part of the public ABI).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <mutex>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "../../include/splitkv.h"

#define SKV_MAX_SLOTS 4

struct skv_handle {
    int device = 0;
    int sm_count = 0;
    int max_smem_optin = 0;
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t entry = nullptr;                       // orders the copy stream after the caller's work
    cudaEvent_t copy_done[SKV_MAX_SLOTS] = {};
    cudaEvent_t compute_done[SKV_MAX_SLOTS] = {};
    int *counters = nullptr;                           // per-unit arrival counters of the fused split merge
    void *workspace = nullptr;                         // partial outputs (grow-only)
    size_t ws_cap = 0;
    void *ring[SKV_MAX_SLOTS] = {};                    // tail-tile slots: [K bytes | V bytes]
    size_t ring_cap = 0;                               // bytes per slot
    int n_ring = 0;
    int *status = nullptr;                             // device status word (bit 0: a bounded wait gave up)
    cudaEvent_t prof_before = nullptr;                 // optional timing hook around attention kernels
    cudaEvent_t prof_after = nullptr;
    char err[512] = {0};
};

namespace skv {

// Record a formatted error on the handle and return `code`.
int fail(skv_handle *h, int code, const char *fmt, ...);
// Map a CUDA error to SKV_ECUDA with its text (SKV_OK if e == cudaSuccess).
int cuda_fail(skv_handle *h, cudaError_t e, const char *what);
// True when `stream` is capturing a graph.
bool capturing(cudaStream_t stream);
// Grow-only scratch.  Return SKV_ECAPTURE when growth is needed in capture.
int ensure_workspace(skv_handle *h, size_t bytes, cudaStream_t stream);
int ensure_ring(skv_handle *h, size_t bytes_per_slot, int n_slots, cudaStream_t stream);

int64_t segment_bytes(int type, int D);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) takes effect in the current
// device's context only, so a kernel's opt-in (and the occupancy it gives) is
// recorded per device.  One cache per kernel instance; host threads share it
// under its mutex.
constexpr int kAttrDevices = 64;
struct KernelAttrCache {
    std::mutex mu;
    int smem[kAttrDevices] = {};       // dynamic shared memory opted in on each device
    int occ_smem[kAttrDevices] = {};   // the (smem, threads) the cached occupancy was taken at
    int occ_threads[kAttrDevices] = {};
    int occ_ctas[kAttrDevices] = {};
};
// Opt `func` in to `smem` bytes of dynamic shared memory on the current device
// (once per device and size).  With ctas != NULL, also store the CTAs of
// `threads` threads resident per SM at that size.
cudaError_t kernel_smem_optin(KernelAttrCache &c, const void *func, int smem, int threads, int *ctas);

// How key indices of one launch map to cache rows.
enum RowMode { ROWS_DENSE = 0, ROWS_LIST = 1, ROWS_PAGED = 2 };

struct DecodeArgs {
    const __half *q;            // [S][nq][H][D]
    const uint8_t *k;           // cache base
    const uint8_t *v;
    int64_t k_row_bytes;        // dense / list: byte stride between rows
    int64_t v_row_bytes;
    int row_mode;
    int64_t row0;               // dense: cache row of local key 0
    const int32_t *rows;        // list: row ids; paged: page ids
    int64_t rows_ld;            // entries per list
    int rows_per_head;          // list/paged: lists are [S][Hk][rows_ld]
    int64_t rows_off;           // list: entry of local key 0 inside each list
    int page_rows;              // paged: rows per page (power of two)
    const __half *mask;         // [S][nq][mask_ld] or null; column = logical key index
    int64_t mask_ld;
    const int32_t *q_pos;       // [S][nq] or null
    int64_t key_pos0;           // causal position of logical key 0
    int64_t logical0;           // logical index of local key 0
    int64_t n_local;            // local keys of this launch are [key_lo, n_local)
    int64_t key_lo;             // first local key; splits start here (0 unless a range starts mid-page)
    int S, nq, H, Hk, G;
    float scale_log2;           // scale * log2(e)
    int n_cg;                   // column groups (8 query columns each) per (s, k)
    int n_splits;
    int64_t split_len;
    float *o_split;             // per-split partials [split][R][D] (unused when n_splits == 1)
    float *lse_split;           // [split][R]
    int *counters;              // [S*Hk*n_cg] arrival counters, zero between launches
    float *o_out;               // merged result of this launch [R][D]
    float *lse_out;             // [R]
    int64_t R;                  // S*nq*H
    int *status;                // device status word (kernels with bounded waits)
    // The fused block-cache instance (paged mode, pages of kDecodeTile rows):
    // the cache's resolve state (device memory), the call's selection
    // [S][Hk][rows_ld] of block ids and its lookup count, where every lookup's
    // pool page is recorded, the device-mapped host copy in the pool's page
    // layout, the pool pages' publication stamps, this call's epoch and the
    // counter the work items are taken from (zero before the launch).
    const void *rstate;
    const int32_t *sel;
    int64_t n_look;
    int32_t *page_ids_out;
    const uint8_t *host_k;
    const uint8_t *host_v;
    int32_t *page_ready;
    const uint64_t *epoch;
    unsigned long long *steal;
};

// Splits of one launch merged by the last-arriving CTA of each unit are
// capped so that the merge's weights fit its shared-memory chunking.
constexpr int kMaxSplits = 4096;
// Units (sequence x KV head x column group) per launch: one counter each.
constexpr int kMaxUnits = 65536;

// Launch the split-KV decode kernel (one CTA per (split, unit)).
int launch_decode(skv_handle *h, const DecodeArgs &a, int k_type, int v_type, int D, cudaStream_t st);
int launch_decode_f16(skv_handle *h, const DecodeArgs &a, int D, cudaStream_t st);
// The fused block-cache instance (fp16 pages, a.page_src set): a persistent
// cooperative grid of at most the CTAs resident at once.
int launch_decode_fused(skv_handle *h, const DecodeArgs &a, int D, cudaStream_t st);
int launch_decode_quant(skv_handle *h, const DecodeArgs &a, int k_type, int v_type, int D, cudaStream_t st);
// CTAs of the decode kernel resident per SM for this type/D pairing (0 if unsupported).
int decode_ctas_per_sm(skv_handle *h, int k_type, int v_type, int D);
int decode_ctas_f16(skv_handle *h, int D);
int decode_ctas_quant(skv_handle *h, int k_type, int v_type, int D);
// Keys per pipeline stage of the decode kernel, and the most keys one CTA may
// take in list/paged mode.
constexpr int kDecodeTile = 64;
constexpr int kMaxListSplit = 2048;

// Decode over a dense range of quantised rows (q8_0 / q4_0, D = 128, no
// additive mask, Hk <= 8): one CTA per (sequence, column group, split) for
// all KV heads, whole-row stages by bulk copy; splits merged by a combine.
constexpr int kRowsTile = 32;   // keys per stage
bool decode_rows_eligible(const skv_shape *sh, const void *k, const void *v, const void *mask);
int decode_rows_ctas_per_sm(const skv_shape *sh);
int launch_decode_rows(skv_handle *h, const DecodeArgs &a, int kt, int vt, cudaStream_t st);

int launch_combine(int n_parts, const float *o_parts, const float *lse_parts, int64_t rows, int D, float *o,
                   float *lse, cudaStream_t st);

// One launch of the tensor-core prefill kernel over a dense fp16 region.
struct PrefillLaunch {
    const skv_shape *shape;
    const void *q;
    const void *k;              // region base (row 0 of the tensor map)
    const void *v;
    int64_t n_rows;             // rows of the region (tensor-map extent)
    int64_t row0;               // region row of local key 0
    int64_t n_local;
    int64_t logical0;
    const int32_t *q_pos;
    int64_t key_pos0;
    int n_splits;
    int64_t split_len;
    float *o_split;
    float *lse_split;
    float *o_out;
    float *lse_out;
    const int32_t *rows;        // row lists (entry rows_off = local key 0), or null for a dense range
    int64_t rows_ld;
    int64_t rows_off;
    int rows_per_head;
};
bool prefill_eligible(const skv_shape *sh, const void *mask);
// Whether the two-query-tile instance serves a call: dense q8_0 / q4_0 keys
// with q4_0 values over at least two query tiles (`rows`: the keys come
// through row lists).
bool prefill_pairs(const skv_shape *sh, bool rows);
// CTA units per sequence: (KV head, 128-row query tile), or (KV head, pair of
// query tiles) where the two-query-tile instance serves (dense q8_0 / q4_0
// keys with q4_0 values; `rows`: the keys come through row lists)
int prefill_units(const skv_shape *sh, bool rows);
int launch_prefill(skv_handle *h, const PrefillLaunch &L, cudaStream_t st);
constexpr int kPrefillTile = 128;
// Per-CTA fixed cost of the prefill kernel in 128-key tiles (TMEM allocation,
// barrier set-up, Q staging, pipeline fill, epilogue and split merge): about
// 11 us, which is ~9 fp16 tiles (1.2-1.4 us each) but only ~4 tiles of
// q8_0 / q4_0 rows (2.6 us each, the producers decode the codes).  Fitted to
// 128 query tiles over 32768 keys on 152 SMs, where one split per tile beat
// seven (312 against 331 us over fp16 rows, 363 against 397 us over fp16 row
// lists) and seven beat one over q8_0 / q4_0 rows (667 against 710 us).
// The two-query-tile instance (dense q8_0 / q4_0 keys with q4_0 values)
// takes ~3.6 us a key tile for both query tiles: over the 512-token,
// 32768-row window one wave of two even splits per pair (128 CTAs, 463 us)
// beat seven splits in three waves (492 us), and two heads and a tail per
// pair (192 CTAs, 417 us) beat both; a fixed cost of 10 tiles picks that.
inline int prefill_overhead_tiles(const skv_shape *sh, bool rows)
{
    return (sh->k_type == SKV_F16 || prefill_pairs(sh, rows)) ? 10 : 4;
}

// Merge of a unit's split partials by its last CTA, in tiles, charged to a
// head-and-tail plan (which replaces a single split's direct write).
constexpr int kMergeTiles = 2;
int plan_splits_cost(int64_t n_keys, int64_t n_units, int sm_count, int ctas_per_sm, int tile, int64_t max_split,
                     int overhead_tiles, int64_t *split_len, int32_t *n_splits, bool head_tail = false);

// Paged attention over local keys [key_lo, key_hi) of page lists of
// pages_per_list pages (skv_attn_paged is the whole range).
int attn_paged_range(skv_handle *h, const skv_shape *shape, const void *q, const void *k_pages, const void *v_pages,
                     int32_t page_rows, const int32_t *page_ids, int32_t pages_per_list, int64_t key_lo,
                     int64_t key_hi, float *o, float *lse, cudaStream_t st);
// Pages per split of the fused block-cache attention (its work items).
constexpr int kFusedSplitPages = 8;
// The fused block-cache attention over whole lists of kDecodeTile-row pages
// (`fuse` carries rstate .. steal).  SKV_EUNSUPPORTED for a shape it does
// not take (more than one column group of query rows per KV head).
int attn_paged_fused(skv_handle *h, const skv_shape *shape, const void *q, const void *k_pages, const void *v_pages,
                     const int32_t *page_ids, int32_t pages_per_list, float *o, float *lse, cudaStream_t st,
                     const DecodeArgs &fuse);

int launch_dequant(int type, const void *blocks, int64_t n_values, float *out, cudaStream_t st);
int launch_gather(const void *src, int64_t row_bytes, const int32_t *rows, int64_t n, void *dst,
                  cudaStream_t st);

}  // namespace skv
