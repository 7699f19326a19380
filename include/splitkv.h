/*
 * splitkv.h -- C ABI of libsplitkv.so: split-KV flash attention over a
 * partitioned KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The method.  Attention over a long key list is computed per key partition,
 * each partition giving a normalised partial output O_t and its log-sum-exp
 * lse_t; partials merge exactly by
 *     M = max_t lse_t,  O = sum_t e^{lse_t - M} O_t / sum_t e^{lse_t - M},
 *     lse = M + ln sum_t e^{lse_t - M}
 * ("Rolling KV -- position-windowed KV residency", opencoti patch 0070,
 * fattn.cu key-axis tiling and streaming_combine_kernel).  Partitions are a
 * device-resident position window [0, wc) plus a pinned-host tail [wc, n_kv)
 * (same page, two-region forward), or a per-sequence row list into a shared
 * cache with -1 padding ("llama + CUDA: flash_attn_ext_rows (fix unified kv
 * for multi-seq)", the op's doc comment), or pages of a device block cache
 * over a pinned host copy ("Strata compare", KV streaming).
 *
 * Conventions shared by every entry point.
 *  - Every function returns an int status (SKV_OK = 0) and never exits or
 *    aborts.  skv_last_error(h) gives a message for the last failure on h.
 *  - Pointers named *_host are host memory; every other data pointer is
 *    device memory (cudaMalloc / torch CUDA tensors).  The caller owns all
 *    tensors; the handle owns only its streams, events, workspace, ring and
 *    block-cache state.
 *  - Calls are asynchronous and ordered on the caller's `stream` (a
 *    cudaStream_t passed as void*; NULL is the legacy default stream).
 *    Errors found on the host return at once; nothing waits on the GPU
 *    unless a function says so.
 *  - Calls that share one handle must be ordered with respect to each other
 *    (one stream, or caller-side events): they share the handle's workspace
 *    and ring.
 *  - Scratch (workspace, ring) grows on demand and never shrinks.  Growth
 *    calls cudaMalloc, which is refused with SKV_ECAPTURE while `stream` is
 *    capturing a CUDA graph; call skv_reserve() beforehand.
 *
 * Layouts.
 *  - q:   fp16 [S][nq][H][D] (row-major).
 *  - A cache row holds all Hk KV heads of one position, head after head
 *    ("cell-major"); head k's data starts at byte k * seg, where seg = 2*D
 *    (f16), 34*D/32 (q8_0) or 18*D/32 (q4_0); consecutive rows are
 *    k_row_bytes / v_row_bytes apart.
 *  - q8_0 block (34 B): fp16 scale d, 32 int8 codes q; value = d*q.
 *    q4_0 block (18 B): fp16 scale d, 16 bytes; byte j holds u_j in its low
 *    nibble and u_{j+16} in its high nibble; value = d*(u-8).  (The pages name
 *    these 32-value block types but do not print their bytes; this is the
 *    usual ggml layout.)
 *  - GQA: q head h uses KV head h / (H/Hk).
 *  - Outputs: o fp32 [S][nq][H][D] (normalised), lse fp32 [S][nq][H] in
 *    natural log.  A row that sees no key gets o = 0 and lse = -inf.
 *  - Optional additive mask: fp16 [S][nq][mask_ld], column = logical key
 *    index.  Optional causal positions q_pos int32 [S][nq]: logical key j is
 *    visible to token t iff key_pos0 + j <= q_pos[s][t].
 */
#ifndef SPLITKV_H
#define SPLITKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define SKV_OK 0
#define SKV_EINVAL 1         /* bad argument (null pointer, size, shape)       */
#define SKV_EUNSUPPORTED 2   /* shape/type/alignment this build does not cover */
#define SKV_ENOTPINNED 3     /* a *_host pointer is not page-locked host memory */
#define SKV_ENOMEM 4         /* device or pinned allocation failed             */
#define SKV_ECAPTURE 5       /* scratch must grow while the stream captures    */
#define SKV_ECUDA 6          /* a CUDA runtime call failed                     */
#define SKV_ETIMEOUT 7       /* a device-side wait gave up (bounded spin)      */
#define SKV_EDEVICE 8        /* the device status word reports a violation     */

/* ---- element types of cache rows -------------------------------------- */
#define SKV_F16 0
#define SKV_Q8_0 1
#define SKV_Q4_0 2

typedef struct skv_handle skv_handle;

typedef struct skv_shape {
    int32_t S;           /* sequences                                       */
    int32_t nq;          /* query tokens per sequence                       */
    int32_t H;           /* query heads                                     */
    int32_t Hk;          /* KV heads; H % Hk == 0                           */
    int32_t D;           /* head dim (Dk = Dv): 64 or 128                    */
    float scale;         /* score scale, usually 1/sqrt(D)                  */
    int32_t k_type;      /* SKV_F16 / SKV_Q8_0 / SKV_Q4_0                    */
    int32_t v_type;
    int64_t k_row_bytes; /* byte stride between consecutive cache rows      */
    int64_t v_row_bytes;
} skv_shape;

/* ---- handle ---------------------------------------------------------- */

/* Create a handle on `device` (makes it current): a copy stream, the
 * double-buffer events and an error buffer.  No scratch is allocated yet. */
int skv_create(int device, skv_handle **out);

/* Free the handle's scratch, events and stream.  Synchronises the device. */
int skv_destroy(skv_handle *h);

/* Message of the last failure on h (never NULL; "" after success). */
const char *skv_last_error(const skv_handle *h);

/* Static text for a status code. */
const char *skv_status_string(int status);

/* Grow the workspace (partial outputs) to at least workspace_bytes and the
 * tail ring to n_slots (<= 4) slots of ring_bytes_per_slot each.  Call
 * outside graph capture.  Synchronous with respect to earlier work on h. */
int skv_reserve(skv_handle *h, size_t workspace_bytes, size_t ring_bytes_per_slot, int32_t n_slots);

/* Current scratch sizes (bytes), for inspection. */
int skv_scratch_info(const skv_handle *h, size_t *workspace_bytes, size_t *ring_bytes_per_slot,
                     int32_t *n_slots);

/* Wait for all work on the device, then read and clear the handle's device
 * status word.  SKV_ETIMEOUT: a bounded device-side wait (tensor-core
 * pipeline barriers) gave up; the affected outputs are not valid.  SKV_EDEVICE:
 * another bit is set (bit 1 = an append named a position outside its cache;
 * that row was not written).  The word is stored in *dev_code when dev_code
 * is not NULL. */
int skv_status(skv_handle *h, int32_t *dev_code);

/* Number of SMs of the handle's device. */
int skv_sm_count(const skv_handle *h, int32_t *out);

/* Profiling hook.  When `before`/`after` (cudaEvent_t passed as void*) are
 * non-NULL, every later launch of the attention kernel (the split-KV decode
 * kernel) is bracketed by cudaEventRecord(before) / cudaEventRecord(after) on
 * the stream it is launched on, so a caller can time that kernel alone.
 * With several attention launches in one call, the events end up around the
 * last one.  Pass NULLs to switch the hook off. */
int skv_set_profile_events(skv_handle *h, void *before, void *after);

/* ---- host-side planning (pure host logic; no GPU needed) --------------- */

/* Split a key range of n_keys keys, shared by n_units independent
 * (sequence, KV head, column group) units, into n_splits pieces of split_len
 * keys (a multiple of `tile`, at most max_split keys when max_split > 0) so
 * that units * n_splits CTAs fill whole waves of sm_count * ctas_per_sm.
 * The last piece may be shorter.  The tile-count policy of the Rolling KV
 * patch (coarse key tiles to cut launch overhead, tiles aligned to the
 * kernel's key stride) chose tiles per launch; here one launch covers every
 * split and the policy chooses split sizes instead. */
int skv_plan_splits(int64_t n_keys, int64_t n_units, int32_t sm_count, int32_t ctas_per_sm,
                    int32_t tile, int64_t max_split, int64_t *split_len, int32_t *n_splits);

/* The split plan a call of this shape over n_keys keys gets on the
 * tensor-core prefill path (many query rows per KV head: skv_attn_partial
 * and skv_attn_window_tail's window and tail tiles) on sm_count SMs; rows
 * != 0: the keys come through row lists.  One CTA takes a 128-row query tile
 * of a KV head (dense q8_0 / q4_0 keys with q4_0 values: a pair of query
 * tiles) and one split of 128-key tiles, one CTA per SM, at a fixed cost per
 * CTA of 10 tiles (fp16 rows, query-tile pairs) or 4 (other quantised
 * rows).  Besides the even splits of skv_plan_splits the plan weighs m head
 * splits and a tail split per unit when the units' heads leave some SMs
 * free: long heads for every unit, then a short tail for every unit that the
 * free SMs run while the heads do (n_splits = m + 1, split_len = a head's
 * keys).
 * *n_ctas = units x n_splits.  n_keys = 0 gives *n_splits = 0.  SKV_EINVAL
 * on a NULL pointer, negative n_keys, sm_count below 1 or an invalid shape;
 * SKV_EUNSUPPORTED when the shape does not take the tensor-core path. */
int skv_plan_prefill_splits(const skv_shape *shape, int64_t n_keys, int32_t sm_count, int32_t rows,
                            int64_t *split_len, int32_t *n_splits, int64_t *n_ctas);

/* Resident window size ("Rolling KV" page, position-axis residency sizing).
 * budget = min(free_bytes, target_bytes if > 0) - reserve_bytes (floored at
 * 0).  If per_cell_bytes * kv_size fits the budget the whole cache stays
 * resident: *window_cells = kv_size.  Otherwise *window_cells is the largest
 * cell count whose bytes fit, rounded down to align = max(n_pad (0: 32), 256),
 * at least align, and at most kv_size - align (rounded down) so that a tail
 * of at least one step remains.  per_cell_bytes is the K+V bytes of one
 * position over every layer kept in the cache. */
int skv_plan_window(int64_t per_cell_bytes, int64_t kv_size, int64_t free_bytes, int64_t target_bytes,
                    int64_t reserve_bytes, int32_t n_pad, int64_t *window_cells);

/* Tail tile size (same page, streaming forward's tile sizing): start from
 * ceil(n_keys / target_keys) tiles (the page uses 32768 keys per tile to keep
 * launches few), raise the count until n_slots slots of one tile (per_key_bytes
 * each key) fit slot_cap_bytes (the page: 4 slots within 512 MiB), keep at
 * most one tile per align-key block, and make every tile a whole number of
 * blocks.  *tile_rows = rows per tile, *n_tiles = tiles covering n_keys. */
int skv_plan_tail_tile(int64_t n_keys, int64_t per_key_bytes, int32_t n_slots, int64_t slot_cap_bytes,
                       int64_t target_keys, int32_t align, int64_t *tile_rows, int32_t *n_tiles);

/* ---- attention ------------------------------------------------------- */

/* Attention of every (s, t, h) row over logical keys [kv_begin, kv_end) of a
 * cache (key_offset semantics below), written as one normalised result:
 *   kv_rows == NULL : logical key j reads cache row j.
 *   kv_rows != NULL : logical key j of sequence s reads cache row
 *                     kv_rows[s*kv_rows_ld + j] (kv_rows_per_head == 0) or
 *                     kv_rows[(s*Hk + k)*kv_rows_ld + j] (== 1); a negative
 *                     entry is padding: nothing is read and the key is absent
 *                     (flash_attn_ext_rows semantics).  Key tiles whose rows
 *                     are all padding issue no memory reads.
 * Mask column and causal position of logical key j: column j, position
 * key_pos0 + j.  k, v are device pointers to row 0 of the cache.
 * Internally the range is split across CTAs (skv_plan_splits) and the
 * partials are merged by the log-sum-exp combine; o/lse receive the merged
 * result.  Errors: SKV_EINVAL (shape), SKV_EUNSUPPORTED (D not 64/128, a
 * type pairing or alignment the kernels do not cover), SKV_ECAPTURE. */
int skv_attn_partial(skv_handle *h, const skv_shape *shape,
                     const void *q, const void *k, const void *v,
                     const void *mask, int64_t mask_ld,
                     const int32_t *q_pos, int64_t key_pos0,
                     const int32_t *kv_rows, int64_t kv_rows_ld, int32_t kv_rows_per_head,
                     int64_t kv_begin, int64_t kv_end,
                     float *o, float *lse, void *stream);

/* skv_attn_partial for callers that cannot allocate device memory.  The pages
 * have no counterpart of this entry point; it exists for code that must not
 * call cudaMalloc: an engine that reserves all device memory up front and
 * serves every buffer from its own pool, a latency-critical path that cannot
 * afford the device-wide synchronisation cudaMalloc/cudaFree may cause, or a
 * caller without a library handle (skv_create itself allocates).
 *
 * Same arguments and results as skv_attn_partial, without the handle; it
 * always runs the split-KV decode kernel (never the tensor-core prefill
 * kernel).  It allocates nothing: its scratch (split partials and the
 * in-kernel merge's arrival counters) is one 16 MiB array in device global
 * memory that every GPU loading this library holds until the process exits.
 * The first call on a device, made with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and keeps it for the life of
 * the process; make that first call before any stream capture, and do not call
 * this entry point on a device after cudaDeviceReset (the kept address is then
 * stale).  Maximum: 4096 sequence x KV-head x 8-column units (the arrival
 * counters); a call with more returns SKV_ENOMEM.  When the planned key splits'
 * partials would not fit the rest of the array, the call uses as many splits as
 * fit (one split writes o/lse directly and needs no scratch).  SKV_EINVAL /
 * SKV_EUNSUPPORTED for the same argument errors as skv_attn_partial (there is
 * no handle to carry a message).  All calls share the one array: calls that
 * overlap on the GPU (different streams, or different host threads) race and
 * must be ordered by the caller.  The arrival counters are cleared on `stream`
 * at every call that splits. */
int skv_attn_partial_static(const skv_shape *shape, const void *q, const void *k, const void *v,
                            const void *mask, int64_t mask_ld, const int32_t *q_pos, int64_t key_pos0,
                            const int32_t *kv_rows, int64_t kv_rows_ld, int32_t kv_rows_per_head,
                            int64_t kv_begin, int64_t kv_end, float *o, float *lse, void *stream);

/* Log-sum-exp combine (formula at the top of this file) of n_parts partial
 * results: o_parts fp32 [n_parts][rows][D], lse_parts fp32 [n_parts][rows]
 * -> o [rows][D], lse [rows].  A part with lse = -inf contributes nothing
 * (its o is never read); every part -inf gives o = 0, lse = -inf.
 * n_parts = 0 is allowed (fills o = 0, lse = -inf).  Limits: n_parts <= 4096,
 * D <= 128 and a multiple of 4, o_parts and o 16-byte aligned
 * (SKV_EUNSUPPORTED otherwise). */
int skv_attn_combine(skv_handle *h, int32_t n_parts, const float *o_parts, const float *lse_parts,
                     int64_t rows, int32_t D, float *o, float *lse, void *stream);

/* Window + host-tail attention (Rolling KV patch two-region forward, with
 * the bulk raw-byte lift and persistent scratch ring of opencoti patch 0102).
 * Logical keys [0, n_win) are window rows k_win/v_win (device); logical keys
 * [n_win, n_win + n_tail) are rows of k_tail_host/v_tail_host, which must be
 * page-locked host memory (SKV_ENOTPINNED otherwise).  The tail is cut into
 * tiles of tile_rows rows (<= 0: skv_plan_tail_tile with 32768 target keys,
 * 4 ring slots within 512 MiB, 256-key blocks); each tile's raw bytes (any of the
 * three types) are copied in one cudaMemcpyAsync per K/V into a ring slot on
 * the handle's copy stream, while the window and earlier tiles compute on
 * `stream`; copy_done/compute_done events order slot reuse.  The ring takes
 * one slot per tile, at most 4 (during graph capture: the slots it already
 * has).  All partials merge in one combine into o/lse.  Ring slots hold
 * tile_rows rows and grow only outside capture. */
int skv_attn_window_tail(skv_handle *h, const skv_shape *shape, const void *q,
                         const void *k_win, const void *v_win, int64_t n_win,
                         const void *k_tail_host, const void *v_tail_host, int64_t n_tail,
                         int64_t tile_rows,
                         const void *mask, int64_t mask_ld, const int32_t *q_pos,
                         float *o, float *lse, void *stream);

/* ---- quantised rows and gathers (bit-exact test hooks) ------------------ */

/* Decode n_values (multiple of 32) values of q8_0 / q4_0 blocks into fp32.
 * The product of an fp16 scale and a code of at most 8 bits is exact in
 * fp32, so the output is the exact value d*q (resp. d*(u-8)). */
int skv_kv_dequant_q8_0(skv_handle *h, const void *blocks, int64_t n_values, float *out, void *stream);
int skv_kv_dequant_q4_0(skv_handle *h, const void *blocks, int64_t n_values, float *out, void *stream);

/* dst[i] = src[rows[i]] for i < n, row_bytes bytes per row; rows[i] < 0
 * writes a zero row and reads nothing (the gather through a row list of the
 * flash_attn_ext_rows thread, padding clamped to nothing). */
int skv_gather_rows(skv_handle *h, const void *src, int64_t row_bytes, const int32_t *rows, int64_t n,
                    void *dst, void *stream);

/* Failure-path self-test: one CTA waits, with the same bounded mbarrier wait
 * the tensor-core kernels use for their pipeline barriers, on a barrier that
 * nothing arrives on.  After budget_ns of wall-clock time (1e3 .. 1e9) the
 * wait gives up and sets bit 0 of the handle's device status word, so the
 * next skv_status returns SKV_ETIMEOUT; the context stays usable.  No fault,
 * trap or unbounded wait is involved.  SKV_EINVAL for a budget outside the
 * range. */
int skv_selftest_wait_timeout(skv_handle *h, int64_t budget_ns, void *stream);

/* ---- appending rows (write routing and quantise-on-append) ------------- */

/* Write n new rows of one tensor (K or V) into a cell-major cache of two
 * regions (Rolling KV, "what ships": the K/V copies split between a device
 * window [0, wc) and a pinned host tail [wc, n_kv)).
 *   x          fp32 [n][Hk][D], device, 16-byte aligned; D is 64 or 128.
 *   positions  int32 [n], device: row i goes to cache position positions[i];
 *              position p < n_rows0 is window row p of dst0, otherwise tail
 *              row p - n_rows0 of dst1; a negative position writes nothing;
 *              a position >= n_rows0 + n_rows1 writes nothing and sets bit 1
 *              of the handle's device status word (skv_status).  Two rows
 *              with the same position: either one wins.
 *   dst0/dst1  region bases, each device memory or page-locked device-mapped
 *              host memory (SKV_ENOTPINNED otherwise); row stride row_bytes;
 *              head k's segment sits at byte k*segment(type, D) of a row.
 * type SKV_F16 rounds each value to nearest fp16.  SKV_Q8_0 quantises each
 * 32-value block as on the Strata KV-streaming page (kv_append_q8): in fp32,
 * d = fp16(amax / 127), q = rint(x / d) clamped to [-127, 127]; SKV_Q4_0 uses
 * the same rule with d = fp16(amax / 7) and u = rint(x / d) + 8 clamped to
 * [0, 15] (a reading: the pages give no q4_0 quantiser).  amax = 0 stores d = 0
 * and zero codes.  Byte layouts are those skv_kv_dequant_* decode.  Alignment:
 * bases and row_bytes 4-byte (fp16) or 2-byte (quantised), else
 * SKV_EUNSUPPORTED.  Stream-ordered; allocates nothing. */
int skv_kv_append(skv_handle *h, int32_t type, int32_t Hk, int32_t D, int64_t row_bytes, const float *x,
                  const int32_t *positions, int32_t n, void *dst0, int64_t n_rows0, void *dst1, int64_t n_rows1,
                  void *stream);

/* ---- paged attention and the device block cache --------------------------
 *
 * A page is page_rows consecutive rows of ONE KV head, fp16, D values per
 * row (page_rows * D * 2 bytes); a page pool is an array of such pages.
 */

/* Attention through page lists: logical key j of sequence s, KV head k reads
 * row j % page_rows of pool page page_ids[(s*Hk + k)*pages_per_list +
 * j / page_rows]; a negative page id is padding (its keys are absent).
 * shape->k_type/v_type must be SKV_F16; the row strides are ignored.
 * page_rows must be a power of two <= 2048. */
int skv_attn_paged(skv_handle *h, const skv_shape *shape, const void *q, const void *k_pages, const void *v_pages,
                   int32_t page_rows, const int32_t *page_ids, int32_t pages_per_list, float *o, float *lse,
                   void *stream);

/* Device block cache over a pinned host copy ("Strata compare", KV
 * streaming: a VRAM block cache with CLOCK eviction over a pinned host copy,
 * resolved on the device).  The host copy is paged [n_blocks][Hk][block_rows]
 * [D] fp16 in page-locked, device-mapped memory (SKV_ENOTPINNED otherwise);
 * page (block b, KV head k) = host page b*Hk + k.  The cache holds n_slots
 * resident pages plus an overflow area of max_lookups pages: misses beyond the
 * free capacity are read from the host for that call only. */
typedef struct skv_bcache skv_bcache;

typedef struct skv_bcache_counters {
    uint64_t calls;        /* resolves so far                                 */
    uint64_t lookups;      /* (sequence, KV head, block) lookups              */
    uint64_t hits;         /* lookups that found the page resident            */
    uint64_t misses;       /* distinct missed pages (placed + overflow)       */
    uint64_t overflow;     /* missed pages that found no slot                 */
    int64_t last_misses;   /* of the last resolve                             */
    int64_t last_overflow;
} skv_bcache_counters;

int skv_bcache_create(skv_handle *h, int64_t n_blocks, int32_t block_rows, int32_t Hk, int32_t D, int32_t n_slots,
                      int64_t max_lookups, const void *host_k, const void *host_v, skv_bcache **out);
int skv_bcache_destroy(skv_bcache *c);

/* Evict everything (page table -1, slots free, counters 0); stream-ordered. */
int skv_bcache_reset(skv_bcache *c, void *stream);

/* Make the pages named by sel (int32 block ids [S][Hk][n_sel], device) readable
 * in the pool: hits keep their slot; each missing page, however many lookups
 * name it, takes one slot chosen by second chance (CLOCK) among the slots this
 * call does not read, or -- when none is left -- an overflow page for this call
 * only; then every missed page is copied from the host copy.  page_ids [S][Hk][n_sel] (device; NULL = the
 * cache's own buffer) receives the pool page of each lookup (-1 for a block id
 * out of range).  Runs entirely on `stream`, no host synchronisation. */
int skv_bcache_resolve(skv_bcache *c, const int32_t *sel, int32_t S, int32_t n_sel, int32_t *page_ids, void *stream);

/* Write-through append ("Strata compare", KV streaming: writers write the
 * host copy always and a VRAM page only while its block is resident, so
 * resident pages never go stale).  k_new, v_new: fp32 [n][Hk][D], device,
 * 16-byte aligned; positions int32 [n], device: cache position p is row
 * p % block_rows of block p / block_rows.  Each row is rounded to fp16 and
 * written into the host copy (through its mapped address; the host copy must
 * be 16-byte aligned) and, when page (block, KV head) is resident, into its
 * pool page.  A negative position writes nothing; one >= n_blocks*block_rows
 * writes nothing and sets bit 1 of the handle's device status word.
 * Stream-ordered with resolve and attention on the same stream. */
int skv_bcache_append(skv_bcache *c, const float *k_new, const float *v_new, const int32_t *positions, int32_t n,
                      void *stream);

/* Resolve, copy the missed blocks and attend, for q of shape [S][nq][H][D]
 * ("Strata compare", KV streaming), all on `stream`; residency decisions and
 * counters are those of skv_bcache_resolve.
 * With block_rows = 64 and at most 8 query rows per KV head (nq * H / Hk <=
 * 8), the copy and the attention are one pass: after the lookup, one
 * persistent launch reads each missed page from the host copy in the work
 * item (8 pages of one list) of the page's first lookup, writes it to that
 * lookup's overflow page and attends to it; later lookups of the page read it
 * from there once written; resident pages are read from their slots; the
 * claim / victim / placement pass runs inside the same launch, and the misses
 * it places in slots are moved there afterwards.  The result is bitwise that
 * of the same call on a cache that holds every page (all hits), and the last
 * page ids (skv_bcache_pool) are the slots of resident and placed pages and
 * the overflow page of each other page's first lookup.
 * Otherwise: skv_bcache_resolve, then skv_attn_paged (page_rows = block_rows)
 * through the pool. */
int skv_bcache_attn(skv_bcache *c, const skv_shape *shape, const void *q, const int32_t *sel, int32_t n_sel,
                    float *o, float *lse, void *stream);

/* Cumulative counters (synchronises the device). */
int skv_bcache_stats(skv_bcache *c, skv_bcache_counters *out);

/* Count violations of the residency invariants (every page-table entry is -1
 * or a slot, and the page table and the slot map are inverse maps);
 * synchronises the device. */
int skv_bcache_check(skv_bcache *c, int32_t *violations);

/* Ring layout ("Strata compare", KV streaming: a reader that only ever reads
 * its last cells uses the same host copy with a static table block ->
 * block % n_slots and no resolve, and the ring is refilled from the host copy
 * on a resume).  The cache holds ring_blocks blocks (ring_blocks * Hk pages):
 * page (block b, KV head k) lives in pool page (b % ring_blocks) * Hk + k.
 * skv_bcache_append then writes every row into the host copy and its ring
 * page (a newer block overwrites the block ring_blocks before it);
 * skv_bcache_resolve / skv_bcache_attn return SKV_EUNSUPPORTED.  max_seqs
 * bounds shape->S of skv_bcache_ring_attn.  After creation or a reset the
 * ring's contents are undefined until skv_bcache_ring_restore. */
int skv_bcache_create_ring(skv_handle *h, int64_t n_blocks, int32_t block_rows, int32_t Hk, int32_t D,
                           int32_t ring_blocks, int32_t max_seqs, const void *host_k, const void *host_v,
                           skv_bcache **out);

/* Refill the ring for a cache of n_keys cells: the pages of the last
 * min(ring_blocks, blocks in use) blocks are copied from the host copy into
 * their ring pages (stream-ordered; 0 <= n_keys <= n_blocks * block_rows). */
int skv_bcache_ring_restore(skv_bcache *c, int64_t n_keys, void *stream);

/* Attention of q [S][nq][H][D] over cells [max(0, n_keys - window), n_keys)
 * read through the ring (window <= 0: every cell the ring holds, i.e. from the
 * first cell of block max(0, last - ring_blocks + 1), last = (n_keys-1) /
 * block_rows).  Every query token sees the same cells.  A window reaching
 * past the ring's oldest cell is SKV_EINVAL.  Results are those of attention
 * over the same cells of the host copy, provided the ring was restored and
 * every later append went through skv_bcache_append. */
int skv_bcache_ring_attn(skv_bcache *c, const skv_shape *shape, const void *q, int64_t n_keys, int64_t window,
                         float *o, float *lse, void *stream);

/* Device pointers of the page pool and of the last resolve's page ids. */
int skv_bcache_pool(const skv_bcache *c, const void **k_pages, const void **v_pages, int64_t *n_pool_pages,
                    const int32_t **last_page_ids);

#ifdef __cplusplus
}
#endif

#endif /* SPLITKV_H */
