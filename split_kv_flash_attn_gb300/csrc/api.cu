// api.cu -- the C ABI: handle, scratch, split planning and the host side of
// the attention calls (decode launches, tail streaming, combine).
#include <string.h>

#include <algorithm>

#include "internal.h"

namespace skv {

int fail(skv_handle *h, int code, const char *fmt, ...)
{
    if (h) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(h->err, sizeof(h->err), fmt, ap);
        va_end(ap);
    }
    return code;
}

int cuda_fail(skv_handle *h, cudaError_t e, const char *what)
{
    if (e == cudaSuccess) return SKV_OK;
    return fail(h, SKV_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool capturing(cudaStream_t stream)
{
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &st) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return st != cudaStreamCaptureStatusNone;
}

static size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

int ensure_workspace(skv_handle *h, size_t bytes, cudaStream_t stream)
{
    if (bytes <= h->ws_cap) return SKV_OK;
    if (capturing(stream))
        return fail(h, SKV_ECAPTURE, "workspace must grow to %zu bytes during graph capture; call skv_reserve first",
                    bytes);
    const size_t cap = round_up(bytes, size_t(1) << 20);
    if (h->workspace) {
        cudaError_t e = cudaFree(h->workspace);   // waits for work still using it
        h->workspace = nullptr;
        h->ws_cap = 0;
        if (e != cudaSuccess) return cuda_fail(h, e, "cudaFree(workspace)");
    }
    cudaError_t e = cudaMalloc(&h->workspace, cap);
    if (e != cudaSuccess) {
        cudaGetLastError();
        h->workspace = nullptr;
        return fail(h, SKV_ENOMEM, "cudaMalloc(%zu) for the workspace: %s", cap, cudaGetErrorString(e));
    }
    h->ws_cap = cap;
    return SKV_OK;
}

int ensure_ring(skv_handle *h, size_t bytes_per_slot, int n_slots, cudaStream_t stream)
{
    if (n_slots > SKV_MAX_SLOTS) return fail(h, SKV_EINVAL, "at most %d ring slots", SKV_MAX_SLOTS);
    if (bytes_per_slot <= h->ring_cap && n_slots <= h->n_ring) return SKV_OK;
    if (capturing(stream))
        return fail(h, SKV_ECAPTURE, "tail ring must grow to %d x %zu bytes during graph capture; call skv_reserve",
                    n_slots, bytes_per_slot);
    const size_t cap = round_up(std::max(bytes_per_slot, h->ring_cap), size_t(1) << 20);
    const int n = std::max(n_slots, h->n_ring);
    // Grow-only and persistent: a slot is never handed to another user while a
    // copy into it may be pending (opencoti patch 0102, bug-2121).  cudaFree
    // waits for pending work before the old slots go away.
    for (int s = 0; s < SKV_MAX_SLOTS; ++s) {
        if (h->ring[s] && (cap > h->ring_cap)) {
            cudaFree(h->ring[s]);
            h->ring[s] = nullptr;
        }
    }
    for (int s = 0; s < n; ++s) {
        if (h->ring[s]) continue;
        cudaError_t e = cudaMalloc(&h->ring[s], cap);
        if (e != cudaSuccess) {
            cudaGetLastError();
            h->ring[s] = nullptr;
            return fail(h, SKV_ENOMEM, "cudaMalloc(%zu) for ring slot %d: %s", cap, s, cudaGetErrorString(e));
        }
    }
    h->ring_cap = cap;
    h->n_ring = n;
    return SKV_OK;
}

cudaError_t kernel_smem_optin(KernelAttrCache &c, const void *func, int smem, int threads, int *ctas)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kAttrDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(c.mu);
    if (c.smem[dev] < smem) {
        e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        c.smem[dev] = smem;
    }
    if (ctas) {
        if (c.occ_smem[dev] != smem || c.occ_threads[dev] != threads) {
            int n = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem);
            if (e != cudaSuccess) return e;
            c.occ_smem[dev] = smem;
            c.occ_threads[dev] = threads;
            c.occ_ctas[dev] = n;
        }
        *ctas = c.occ_ctas[dev];
    }
    return cudaSuccess;
}

int64_t segment_bytes(int type, int D)
{
    switch (type) {
    case SKV_F16: return 2 * static_cast<int64_t>(D);
    case SKV_Q8_0: return 34 * static_cast<int64_t>(D / 32);
    case SKV_Q4_0: return 18 * static_cast<int64_t>(D / 32);
    default: return -1;
    }
}

// Split planning with a cost model: a launch of `total` CTAs runs in
// ceil(total / wave) waves, and each CTA costs its key tiles plus a fixed
// overhead (prologue, pipeline fill, epilogue, merge) of `overhead_tiles`.
// The split count minimising waves x (tiles per split + overhead) wins; ties
// go to fewer splits.
int plan_splits_cost(int64_t n_keys, int64_t n_units, int sm_count, int ctas_per_sm, int tile, int64_t max_split,
                     int overhead_tiles, int64_t *split_len, int32_t *n_splits, bool head_tail)
{
    const int64_t tiles = (n_keys + tile - 1) / tile;
    const int64_t wave = static_cast<int64_t>(sm_count) * ctas_per_sm;
    const int64_t max_tps = max_split > 0 ? max_split / tile : tiles;
    const int64_t min_tps = std::min<int64_t>(tiles, 2);   // at least two stages per CTA when possible
    const int64_t s_max = std::min<int64_t>(tiles, std::max<int64_t>(1, 64 * wave / n_units + 1));
    int64_t best_tps = -1;
    double best_cost = 0.0;
    for (int64_t s = 1; s <= s_max; ++s) {
        const int64_t tps = std::max<int64_t>((tiles + s - 1) / s, min_tps);
        if (tps > max_tps) continue;
        const int64_t splits = (tiles + tps - 1) / tps;
        const int64_t waves = (splits * n_units + wave - 1) / wave;
        const double cost = static_cast<double>(waves) * static_cast<double>(tps + overhead_tiles);
        if (best_tps < 0 || cost < best_cost - 1e-9) {
            best_cost = cost;
            best_tps = tps;
        }
    }
    // Heads and a tail: with fewer units than CTA slots, each unit takes m
    // long head splits on the slots the units' heads fill and one short
    // tail split; the launch dispatches every head before any tail (the
    // split index is the slowest grid dimension), so the slots the heads
    // leave free run k = ceil(units / free) tails each while the heads run.
    // Cost: the longer of a head and k tails, plus the merge of the parts.
    // With fixed cost c per CTA, head + c = k (tail + c) and m heads + tail
    // = tiles balance at tail = (tiles - m c (k - 1)) / (1 + m k).
    if (head_tail && best_tps >= 0 && tiles >= 2) {
        const int64_t c = overhead_tiles;
        for (int64_t m = 1; n_units * m < wave && m < tiles; ++m) {
            const int64_t free_slots = wave - n_units * m;
            const int64_t k = (n_units + free_slots - 1) / free_slots;
            const int64_t b0 = (tiles - m * c * (k - 1)) / (1 + m * k);
            for (int64_t b = b0 - 1; b <= b0 + 2; ++b) {
                if (b < 1 || b >= tiles) continue;
                const int64_t head = (tiles - b + m - 1) / m;
                if (head < b || head > max_tps || (tiles + head - 1) / head != m + 1) continue;
                const int64_t tail = tiles - m * head;
                const double cost = static_cast<double>(std::max(head + c, k * (tail + c)) + kMergeTiles);
                if (cost < best_cost - 1e-9) {
                    best_cost = cost;
                    best_tps = head;
                }
            }
        }
    }
    if (best_tps < 0) best_tps = std::max<int64_t>(1, max_tps);
    const int64_t splits = (tiles + best_tps - 1) / best_tps;
    if (splits > 0x7fffffff) return SKV_EUNSUPPORTED;
    *split_len = best_tps * tile;
    *n_splits = static_cast<int32_t>(splits);
    return SKV_OK;
}

int launch_decode(skv_handle *h, const DecodeArgs &a, int kt, int vt, int D, cudaStream_t st)
{
    if (h->prof_before) cudaEventRecord(h->prof_before, st);
    int rc;
    if (kt == SKV_F16 && vt == SKV_F16) rc = launch_decode_f16(h, a, D, st);
    else if (kt != SKV_F16 && vt != SKV_F16) rc = launch_decode_quant(h, a, kt, vt, D, st);
    else rc = fail(h, SKV_EUNSUPPORTED, "mixed fp16 / quantised K and V are not built");
    if (h->prof_after) cudaEventRecord(h->prof_after, st);
    return rc;
}

int decode_ctas_per_sm(skv_handle *h, int kt, int vt, int D)
{
    if (kt == SKV_F16 && vt == SKV_F16) return decode_ctas_f16(h, D);
    if (kt != SKV_F16 && vt != SKV_F16) return decode_ctas_quant(h, kt, vt, D);
    return 0;
}

// Checks shared by every attention call; fills G and the column-group count.
static int check_shape(skv_handle *h, const skv_shape *sh, int *G, int *n_cg)
{
    if (!sh) return fail(h, SKV_EINVAL, "shape is NULL");
    if (sh->S <= 0 || sh->nq <= 0 || sh->H <= 0 || sh->Hk <= 0 || sh->H % sh->Hk != 0)
        return fail(h, SKV_EINVAL, "bad shape S=%d nq=%d H=%d Hk=%d", sh->S, sh->nq, sh->H, sh->Hk);
    if (sh->D != 64 && sh->D != 128) return fail(h, SKV_EUNSUPPORTED, "head dim %d (supported: 64, 128)", sh->D);
    if (segment_bytes(sh->k_type, sh->D) < 0 || segment_bytes(sh->v_type, sh->D) < 0)
        return fail(h, SKV_EINVAL, "unknown element type");
    if ((sh->k_type == SKV_F16) != (sh->v_type == SKV_F16))
        return fail(h, SKV_EUNSUPPORTED, "mixed fp16 / quantised K and V are not built");
    if (sh->k_row_bytes < sh->Hk * segment_bytes(sh->k_type, sh->D) ||
        sh->v_row_bytes < sh->Hk * segment_bytes(sh->v_type, sh->D))
        return fail(h, SKV_EINVAL, "row stride smaller than Hk head segments");
    *G = sh->H / sh->Hk;
    *n_cg = (sh->nq * *G + 7) / 8;
    if (static_cast<int64_t>(sh->S) * sh->Hk * *n_cg > 65535)
        return fail(h, SKV_EUNSUPPORTED, "S*Hk*ceil(nq*G/8) exceeds 65535");
    return SKV_OK;
}

static int chunk_of(int type, int D)
{
    const int64_t seg = segment_bytes(type, D);
    return type == SKV_F16 ? 16 : (seg % 8 == 0 ? 8 : 4);
}

static int check_cache(skv_handle *h, const skv_shape *sh, const void *k, const void *v)
{
    if (!k || !v) return fail(h, SKV_EINVAL, "K/V pointer is NULL");
    const int ck = chunk_of(sh->k_type, sh->D), cv = chunk_of(sh->v_type, sh->D);
    if ((reinterpret_cast<uintptr_t>(k) % ck) || (sh->k_row_bytes % ck) || (reinterpret_cast<uintptr_t>(v) % cv) ||
        (sh->v_row_bytes % cv))
        return fail(h, SKV_EUNSUPPORTED, "K/V base or row stride not %d/%d-byte aligned", ck, cv);
    return SKV_OK;
}

static DecodeArgs base_args(const skv_shape *sh, int G, int n_cg, const void *q, const void *mask, int64_t mask_ld,
                            const int32_t *q_pos, int64_t key_pos0)
{
    DecodeArgs a;
    memset(&a, 0, sizeof(a));
    a.q = static_cast<const __half *>(q);
    a.k_row_bytes = sh->k_row_bytes;
    a.v_row_bytes = sh->v_row_bytes;
    a.mask = static_cast<const __half *>(mask);
    a.mask_ld = mask_ld;
    a.q_pos = q_pos;
    a.key_pos0 = key_pos0;
    a.S = sh->S;
    a.nq = sh->nq;
    a.H = sh->H;
    a.Hk = sh->Hk;
    a.G = G;
    a.scale_log2 = sh->scale * 1.4426950408889634f;
    a.n_cg = n_cg;
    a.R = static_cast<int64_t>(sh->S) * sh->nq * sh->H;
    return a;
}

}  // namespace skv

using namespace skv;

extern "C" {

const char *skv_status_string(int status)
{
    switch (status) {
    case SKV_OK: return "ok";
    case SKV_EINVAL: return "invalid argument";
    case SKV_EUNSUPPORTED: return "unsupported shape, type or alignment";
    case SKV_ENOTPINNED: return "host pointer is not page-locked";
    case SKV_ENOMEM: return "out of memory";
    case SKV_ECAPTURE: return "scratch would grow during graph capture";
    case SKV_ECUDA: return "CUDA runtime error";
    case SKV_ETIMEOUT: return "device-side wait timed out";
    case SKV_EDEVICE: return "device reported a violation";
    default: return "unknown status";
    }
}

int skv_create(int device, skv_handle **out)
{
    if (!out) return SKV_EINVAL;
    *out = nullptr;
    skv_handle *h = new (std::nothrow) skv_handle();
    if (!h) return SKV_ENOMEM;
    cudaError_t e = cudaSetDevice(device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&h->max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->entry, cudaEventDisableTiming);
    for (int s = 0; s < SKV_MAX_SLOTS && e == cudaSuccess; ++s) {
        e = cudaEventCreateWithFlags(&h->copy_done[s], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->compute_done[s], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = cudaMalloc(&h->counters, sizeof(int) * kMaxUnits);
    if (e == cudaSuccess) e = cudaMemset(h->counters, 0, sizeof(int) * kMaxUnits);
    if (e == cudaSuccess) e = cudaMalloc(&h->status, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaGetLastError();
        skv_destroy(h);
        return SKV_ECUDA;
    }
    h->device = device;
    *out = h;
    return SKV_OK;
}

int skv_destroy(skv_handle *h)
{
    if (!h) return SKV_OK;
    if (h->copy_stream) cudaStreamSynchronize(h->copy_stream);
    cudaFree(h->workspace);
    cudaFree(h->counters);
    cudaFree(h->status);
    for (int s = 0; s < SKV_MAX_SLOTS; ++s) cudaFree(h->ring[s]);
    for (int s = 0; s < SKV_MAX_SLOTS; ++s) {
        if (h->copy_done[s]) cudaEventDestroy(h->copy_done[s]);
        if (h->compute_done[s]) cudaEventDestroy(h->compute_done[s]);
    }
    if (h->entry) cudaEventDestroy(h->entry);
    if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
    delete h;
    return SKV_OK;
}

const char *skv_last_error(const skv_handle *h) { return h ? h->err : "null handle"; }

int skv_reserve(skv_handle *h, size_t workspace_bytes, size_t ring_bytes_per_slot, int32_t n_slots)
{
    if (!h) return SKV_EINVAL;
    h->err[0] = 0;
    if (n_slots < 0 || n_slots > SKV_MAX_SLOTS) return fail(h, SKV_EINVAL, "n_slots must be 0..%d", SKV_MAX_SLOTS);
    int rc = ensure_workspace(h, workspace_bytes, nullptr);
    if (rc == SKV_OK && n_slots > 0) rc = ensure_ring(h, ring_bytes_per_slot, n_slots, nullptr);
    return rc;
}

int skv_scratch_info(const skv_handle *h, size_t *ws, size_t *ring, int32_t *n_slots)
{
    if (!h) return SKV_EINVAL;
    if (ws) *ws = h->ws_cap;
    if (ring) *ring = h->ring_cap;
    if (n_slots) *n_slots = h->n_ring;
    return SKV_OK;
}

int skv_sm_count(const skv_handle *h, int32_t *out)
{
    if (!h || !out) return SKV_EINVAL;
    *out = h->sm_count;
    return SKV_OK;
}

int skv_status(skv_handle *h, int32_t *dev_code)
{
    if (!h) return SKV_EINVAL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaDeviceSynchronize");
    int word = 0;
    e = cudaMemcpy(&word, h->status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(h, e, "reading the status word");
    if (dev_code) *dev_code = word;
    if (word & 1) return fail(h, SKV_ETIMEOUT, "a device-side wait gave up (status word 0x%x)", word);
    if (word) return fail(h, SKV_EDEVICE, "device status word 0x%x", word);
    return SKV_OK;
}

int skv_set_profile_events(skv_handle *h, void *before, void *after)
{
    if (!h) return SKV_EINVAL;
    if ((before == nullptr) != (after == nullptr)) return fail(h, SKV_EINVAL, "pass both events or neither");
    h->prof_before = static_cast<cudaEvent_t>(before);
    h->prof_after = static_cast<cudaEvent_t>(after);
    return SKV_OK;
}

int skv_plan_splits(int64_t n_keys, int64_t n_units, int32_t sm_count, int32_t ctas_per_sm, int32_t tile,
                    int64_t max_split, int64_t *split_len, int32_t *n_splits)
{
    if (!split_len || !n_splits || n_keys < 0 || n_units <= 0 || sm_count <= 0 || ctas_per_sm <= 0 || tile <= 0 ||
        max_split < 0)
        return SKV_EINVAL;
    if (max_split > 0 && max_split < tile) return SKV_EINVAL;
    if (n_keys == 0) {
        *split_len = tile;
        *n_splits = 0;
        return SKV_OK;
    }
    return skv::plan_splits_cost(n_keys, n_units, sm_count, ctas_per_sm, tile, max_split, 1, split_len, n_splits);
}

int skv_plan_prefill_splits(const skv_shape *shape, int64_t n_keys, int32_t sm_count, int32_t rows,
                            int64_t *split_len, int32_t *n_splits, int64_t *n_ctas)
{
    if (!shape || !split_len || !n_splits || !n_ctas || n_keys < 0 || sm_count <= 0 || shape->S < 1 ||
        shape->nq < 1 || shape->Hk < 1 || shape->H < shape->Hk || shape->H % shape->Hk)
        return SKV_EINVAL;
    if (!skv::prefill_eligible(shape, nullptr)) return SKV_EUNSUPPORTED;
    const int64_t units = static_cast<int64_t>(shape->S) * skv::prefill_units(shape, rows != 0);
    if (n_keys == 0) {
        *split_len = skv::kPrefillTile;
        *n_splits = 0;
        *n_ctas = 0;
        return SKV_OK;
    }
    const int rc = skv::plan_splits_cost(n_keys, units, sm_count, 1, skv::kPrefillTile, 0,
                                         skv::prefill_overhead_tiles(shape, rows != 0), split_len, n_splits, true);
    if (rc == SKV_OK) *n_ctas = units * *n_splits;
    return rc;
}

int skv_attn_combine(skv_handle *h, int32_t n_parts, const float *o_parts, const float *lse_parts, int64_t rows,
                     int32_t D, float *o, float *lse, void *stream)
{
    if (!h) return SKV_EINVAL;
    h->err[0] = 0;
    if (n_parts < 0 || rows < 0 || D <= 0 || D > 128) return fail(h, SKV_EINVAL, "bad combine sizes");
    if (!o || !lse || (n_parts > 0 && (!o_parts || !lse_parts))) return fail(h, SKV_EINVAL, "NULL pointer");
    if (n_parts > 4096 || D % 4 || (reinterpret_cast<uintptr_t>(o_parts) | reinterpret_cast<uintptr_t>(o)) % 16)
        return fail(h, SKV_EUNSUPPORTED, "combine needs n_parts <= 4096, D a multiple of 4, 16-byte aligned o");
    int rc = launch_combine(n_parts, o_parts, lse_parts, rows, D, o, lse, static_cast<cudaStream_t>(stream));
    return rc == SKV_OK ? rc : cuda_fail(h, cudaGetLastError(), "combine launch");
}

int skv_attn_partial(skv_handle *h, const skv_shape *shape, const void *q, const void *k, const void *v,
                     const void *mask, int64_t mask_ld, const int32_t *q_pos, int64_t key_pos0,
                     const int32_t *kv_rows, int64_t kv_rows_ld, int32_t kv_rows_per_head, int64_t kv_begin,
                     int64_t kv_end, float *o, float *lse, void *stream)
{
    if (!h) return SKV_EINVAL;
    h->err[0] = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int G = 0, n_cg = 0;
    int rc = check_shape(h, shape, &G, &n_cg);
    if (rc) return rc;
    if (!q || !o || !lse) return fail(h, SKV_EINVAL, "q/o/lse pointer is NULL");
    if ((rc = check_cache(h, shape, k, v))) return rc;
    if (kv_begin < 0 || kv_end < kv_begin) return fail(h, SKV_EINVAL, "bad key range [%lld, %lld)",
                                                       (long long)kv_begin, (long long)kv_end);
    if (kv_rows && kv_rows_ld < kv_end) return fail(h, SKV_EINVAL, "kv_rows_ld smaller than kv_end");
    if (mask && mask_ld < kv_end) return fail(h, SKV_EINVAL, "mask_ld smaller than kv_end");
    const int64_t n_local = kv_end - kv_begin;
    const int64_t R = static_cast<int64_t>(shape->S) * shape->nq * shape->H;
    const int D = shape->D;
    if (n_local == 0) {
        rc = launch_combine(0, nullptr, nullptr, R, D, o, lse, st);
        return rc == SKV_OK ? rc : cuda_fail(h, cudaGetLastError(), "fill launch");
    }
    if (prefill_eligible(shape, mask)) {
        // Many query rows per KV head: the tensor-core path (dense fp16 ranges
        // by TMA; row lists and quantised rows by its software producers).
        const int64_t units_p = static_cast<int64_t>(shape->S) * prefill_units(shape, kv_rows != nullptr);
        int64_t split_len = 0;
        int32_t n_splits = 0;
        if ((rc = plan_splits_cost(n_local, units_p, h->sm_count, 1, kPrefillTile, 0,
                                   prefill_overhead_tiles(shape, kv_rows != nullptr), &split_len, &n_splits, true)))
            return fail(h, rc, "split planning failed");
        if (units_p > kMaxUnits) return fail(h, SKV_EUNSUPPORTED, "too many query tiles");
        PrefillLaunch L;
        memset(&L, 0, sizeof(L));
        L.shape = shape;
        L.q = q;
        L.k = k;
        L.v = v;
        L.n_rows = kv_end;
        L.row0 = kv_rows ? 0 : kv_begin;
        L.n_local = n_local;
        L.logical0 = kv_begin;
        L.rows = kv_rows;
        L.rows_ld = kv_rows_ld;
        L.rows_off = kv_begin;
        L.rows_per_head = kv_rows_per_head ? 1 : 0;
        L.q_pos = q_pos;
        L.key_pos0 = key_pos0;
        L.n_splits = n_splits;
        L.split_len = split_len;
        L.o_out = o;
        L.lse_out = lse;
        if (n_splits > 1) {
            const size_t o_bytes = round_up(static_cast<size_t>(n_splits) * R * D * sizeof(float), 256);
            if ((rc = ensure_workspace(h, o_bytes + static_cast<size_t>(n_splits) * R * sizeof(float), st)))
                return rc;
            L.o_split = static_cast<float *>(h->workspace);
            L.lse_split = reinterpret_cast<float *>(static_cast<uint8_t *>(h->workspace) + o_bytes);
        }
        return launch_prefill(h, L, st);
    }
    // Dense quantised ranges: the whole-row kernel (all KV heads per CTA).
    const bool rows_k = !kv_rows && decode_rows_eligible(shape, k, v, mask);
    const int ctas = rows_k ? decode_rows_ctas_per_sm(shape) : decode_ctas_per_sm(h, shape->k_type, shape->v_type, D);
    if (ctas <= 0) return fail(h, SKV_EUNSUPPORTED, "no decode kernel for this type pairing / head dim");
    const int64_t units = static_cast<int64_t>(shape->S) * (rows_k ? 1 : shape->Hk) * n_cg;
    int64_t split_len = 0;
    int32_t n_splits = 0;
    if (rows_k)
        rc = plan_splits_cost(n_local, units, h->sm_count, ctas, kRowsTile, 0, 1, &split_len, &n_splits);
    else
        rc = skv_plan_splits(n_local, units, h->sm_count, ctas, kDecodeTile, 0, &split_len,
                             &n_splits);
    if (rc) return fail(h, rc, "split planning failed");

    if (n_splits > kMaxSplits) return fail(h, SKV_EUNSUPPORTED, "%d splits exceed %d", n_splits, kMaxSplits);
    if (units > kMaxUnits) return fail(h, SKV_EUNSUPPORTED, "%lld units exceed %d", (long long)units, kMaxUnits);

    DecodeArgs a = base_args(shape, G, n_cg, q, mask, mask_ld, q_pos, key_pos0);
    a.k = static_cast<const uint8_t *>(k);
    a.v = static_cast<const uint8_t *>(v);
    if (kv_rows) {
        a.row_mode = ROWS_LIST;
        a.rows = kv_rows;
        a.rows_ld = kv_rows_ld;
        a.rows_per_head = kv_rows_per_head ? 1 : 0;
        a.rows_off = kv_begin;
        a.row0 = 0;
    } else {
        a.row_mode = ROWS_DENSE;
        a.row0 = kv_begin;
    }
    a.logical0 = kv_begin;
    a.n_local = n_local;
    a.n_splits = n_splits;
    a.split_len = split_len;
    a.counters = h->counters;
    a.o_out = o;
    a.lse_out = lse;
    if (n_splits > 1) {
        const size_t o_bytes = round_up(static_cast<size_t>(n_splits) * R * D * sizeof(float), 256);
        const size_t need = o_bytes + static_cast<size_t>(n_splits) * R * sizeof(float);
        if ((rc = ensure_workspace(h, need, st))) return rc;
        a.o_split = static_cast<float *>(h->workspace);
        a.lse_split = reinterpret_cast<float *>(static_cast<uint8_t *>(h->workspace) + o_bytes);
    }
    if (rows_k) return launch_decode_rows(h, a, shape->k_type, shape->v_type, st);
    return launch_decode(h, a, shape->k_type, shape->v_type, D, st);
}

int skv_attn_window_tail(skv_handle *h, const skv_shape *shape, const void *q, const void *k_win, const void *v_win,
                         int64_t n_win, const void *k_tail_host, const void *v_tail_host, int64_t n_tail,
                         int64_t tile_rows, const void *mask, int64_t mask_ld, const int32_t *q_pos, float *o,
                         float *lse, void *stream)
{
    if (!h) return SKV_EINVAL;
    h->err[0] = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int G = 0, n_cg = 0;
    int rc = check_shape(h, shape, &G, &n_cg);
    if (rc) return rc;
    if (!q || !o || !lse) return fail(h, SKV_EINVAL, "q/o/lse pointer is NULL");
    if (n_win < 0 || n_tail < 0) return fail(h, SKV_EINVAL, "negative region size");
    if (n_win > 0 && (rc = check_cache(h, shape, k_win, v_win))) return rc;
    if (mask && mask_ld < n_win + n_tail) return fail(h, SKV_EINVAL, "mask_ld smaller than n_win + n_tail");
    const int D = shape->D;
    const int64_t R = static_cast<int64_t>(shape->S) * shape->nq * shape->H;
    if (n_win + n_tail == 0) {
        rc = launch_combine(0, nullptr, nullptr, R, D, o, lse, st);
        return rc == SKV_OK ? rc : cuda_fail(h, cudaGetLastError(), "fill launch");
    }
    if (tile_rows <= 0 && n_tail > 0) {
        // default: the tail-tile planner (32768-key tiles, the ring's slots
        // within 512 MiB, whole 256-key blocks)
        int32_t nt = 0;
        if ((rc = skv_plan_tail_tile(n_tail, shape->k_row_bytes + shape->v_row_bytes, SKV_MAX_SLOTS,
                                     int64_t(512) << 20, 32768, 256, &tile_rows, &nt)))
            return fail(h, rc, "tail-tile planning failed");
    }
    if (tile_rows <= 0) tile_rows = 32768;
    if (n_tail > 0) {
        if (!k_tail_host || !v_tail_host) return fail(h, SKV_EINVAL, "tail pointer is NULL");
        // The tail must be page-locked so that the copy engine can DMA it
        // (opencoti patch 0102: bulk copies at full DMA rate, never a converter
        // reading host memory word by word).
        for (const void *p : {k_tail_host, v_tail_host}) {
            cudaPointerAttributes at;
            cudaError_t e = cudaPointerGetAttributes(&at, p);
            if (e != cudaSuccess || at.type != cudaMemoryTypeHost) {
                cudaGetLastError();
                return fail(h, SKV_ENOTPINNED, "tail pointer %p is not page-locked host memory", p);
            }
        }
        tile_rows = std::min(tile_rows, n_tail);
    }
    // Many query rows per KV head: the tensor-core prefill kernel; else the
    // split-KV decode kernel.
    const bool use_tc = prefill_eligible(shape, mask);
    // quantised rows: the whole-row decode kernel (ring slots are 256-byte aligned)
    const bool use_rows = !use_tc && decode_rows_eligible(shape, n_win > 0 ? k_win : nullptr,
                                                          n_win > 0 ? v_win : nullptr, mask);
    const int ctas = use_tc ? 1
                     : use_rows ? decode_rows_ctas_per_sm(shape)
                                : decode_ctas_per_sm(h, shape->k_type, shape->v_type, D);
    if (ctas <= 0) return fail(h, SKV_EUNSUPPORTED, "no decode kernel for this type pairing / head dim");
    const int64_t units = use_tc ? static_cast<int64_t>(shape->S) * prefill_units(shape, false)
                          : use_rows ? static_cast<int64_t>(shape->S) * n_cg
                                     : static_cast<int64_t>(shape->S) * shape->Hk * n_cg;
    const int tile = use_tc ? kPrefillTile : use_rows ? kRowsTile : kDecodeTile;

    int64_t w_len = 0, t_len = 0;
    int32_t w_splits = 0, t_splits = 0;
    const int overhead = use_tc ? prefill_overhead_tiles(shape, false) : 1;
    if ((rc = plan_splits_cost(n_win, units, h->sm_count, ctas, tile, 0, overhead, &w_len, &w_splits, use_tc)))
        return fail(h, rc, "split planning failed");
    const int64_t n_tt = n_tail > 0 ? (n_tail + tile_rows - 1) / tile_rows : 0;
    if (n_tt > 0 &&
        (rc = plan_splits_cost(tile_rows, units, h->sm_count, ctas, tile, 0, overhead, &t_len, &t_splits, use_tc)))
        return fail(h, rc, "split planning failed");
    // One merged part per launch (window, then each tail tile); each launch's
    // splits merge inside the decode kernel.
    const int64_t n_parts = (n_win > 0 ? 1 : 0) + n_tt;
    const int max_splits = std::max(w_splits, t_splits);
    if (max_splits > kMaxSplits) return fail(h, SKV_EUNSUPPORTED, "%d splits exceed %d", max_splits, kMaxSplits);
    if (units > kMaxUnits) return fail(h, SKV_EUNSUPPORTED, "%lld units exceed %d", (long long)units, kMaxUnits);

    // Workspace: [split partials: O, lse][merged parts: O, lse].
    const size_t so = round_up(static_cast<size_t>(max_splits) * R * D * sizeof(float), 256);
    const size_t sl = round_up(static_cast<size_t>(max_splits) * R * sizeof(float), 256);
    const size_t po = round_up(static_cast<size_t>(n_parts) * R * D * sizeof(float), 256);
    const size_t pl = static_cast<size_t>(n_parts) * R * sizeof(float);
    if ((rc = ensure_workspace(h, so + sl + po + pl, st))) return rc;
    uint8_t *ws = static_cast<uint8_t *>(h->workspace);
    float *o_parts = reinterpret_cast<float *>(ws + so + sl);
    float *lse_parts = reinterpret_cast<float *>(ws + so + sl + po);

    // The tail ring: K tile then V tile per slot.
    const size_t k_tile_bytes = static_cast<size_t>(tile_rows) * shape->k_row_bytes;
    const size_t v_off = round_up(k_tile_bytes, 256);
    const size_t slot_bytes = v_off + static_cast<size_t>(tile_rows) * shape->v_row_bytes;
    // One slot per tile, up to SKV_MAX_SLOTS (the Rolling KV patch's slot pool
    // holds at most four; two is its default): with compute on `stream`
    // held back by the window, two slots would leave the copy engine idle
    // until the first tile's compute frees its slot.  During graph capture
    // the ring's present slots serve (growth is refused there).
    int n_slots = static_cast<int>(std::min<int64_t>(SKV_MAX_SLOTS, n_tt));
    if (capturing(st) && h->n_ring > 0) n_slots = std::min(n_slots, h->n_ring);
    if (n_tt > 0 && (rc = ensure_ring(h, slot_bytes, n_slots, st))) return rc;

    DecodeArgs a = base_args(shape, G, n_cg, q, mask, mask_ld, q_pos, 0);
    a.row_mode = ROWS_DENSE;
    a.o_split = reinterpret_cast<float *>(ws);
    a.lse_split = reinterpret_cast<float *>(ws + so);
    a.counters = h->counters;

    const uint8_t *kh_ = static_cast<const uint8_t *>(k_tail_host);
    const uint8_t *vh_ = static_cast<const uint8_t *>(v_tail_host);
    auto rows_of = [&](int64_t t) { return std::min(tile_rows, n_tail - t * tile_rows); };
    auto lift = [&](int64_t t) -> int {
        const int slot = static_cast<int>(t % n_slots);
        uint8_t *dst = static_cast<uint8_t *>(h->ring[slot]);
        const int64_t rows = rows_of(t);
        const int64_t r0 = t * tile_rows;
        cudaError_t e = cudaMemcpyAsync(dst, kh_ + r0 * shape->k_row_bytes, rows * shape->k_row_bytes,
                                        cudaMemcpyHostToDevice, h->copy_stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dst + v_off, vh_ + r0 * shape->v_row_bytes, rows * shape->v_row_bytes,
                                cudaMemcpyHostToDevice, h->copy_stream);
        if (e == cudaSuccess) e = cudaEventRecord(h->copy_done[slot], h->copy_stream);
        return cuda_fail(h, e, "tail lift");
    };

    cudaError_t e = cudaSuccess;
    if (n_tt > 0) {
        // The copy stream starts after everything already queued on the
        // caller's stream: a ring slot still read by an earlier call is never
        // overwritten (Rolling KV patch, cross-call WAR guard, bug-255).
        e = cudaEventRecord(h->entry, st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->copy_stream, h->entry, 0);
        if (e != cudaSuccess) return cuda_fail(h, e, "copy-stream entry");
        for (int64_t t = 0; t < std::min<int64_t>(n_slots, n_tt); ++t)
            if ((rc = lift(t))) return rc;
    }
    // One launch over a dense region (window or ring slot) of n_rows rows.
    auto run = [&](int64_t n_rows) -> int {
        if (use_rows) return launch_decode_rows(h, a, shape->k_type, shape->v_type, st);
        if (!use_tc) return launch_decode(h, a, shape->k_type, shape->v_type, D, st);
        PrefillLaunch L;
        memset(&L, 0, sizeof(L));
        L.shape = shape;
        L.q = q;
        L.k = a.k;
        L.v = a.v;
        L.n_rows = n_rows;
        L.row0 = a.row0;
        L.n_local = a.n_local;
        L.logical0 = a.logical0;
        L.q_pos = q_pos;
        L.key_pos0 = 0;
        L.n_splits = a.n_splits;
        L.split_len = a.split_len;
        L.o_split = a.o_split;
        L.lse_split = a.lse_split;
        L.o_out = a.o_out;
        L.lse_out = a.lse_out;
        return launch_prefill(h, L, st);
    };
    int64_t part = 0;
    if (n_win > 0) {
        a.k = static_cast<const uint8_t *>(k_win);
        a.v = static_cast<const uint8_t *>(v_win);
        a.row0 = 0;
        a.logical0 = 0;
        a.n_local = n_win;
        a.n_splits = w_splits;
        a.split_len = w_len;
        a.o_out = o_parts;
        a.lse_out = lse_parts;
        if ((rc = run(n_win))) return rc;
        ++part;
    }
    for (int64_t t = 0; t < n_tt; ++t, ++part) {
        const int slot = static_cast<int>(t % n_slots);
        e = cudaStreamWaitEvent(st, h->copy_done[slot], 0);
        if (e != cudaSuccess) return cuda_fail(h, e, "wait copy_done");
        const uint8_t *base = static_cast<const uint8_t *>(h->ring[slot]);
        a.k = base;
        a.v = base + v_off;
        a.row0 = 0;
        a.logical0 = n_win + t * tile_rows;
        a.n_local = rows_of(t);
        a.n_splits = t_splits;
        a.split_len = t_len;
        a.o_out = o_parts + static_cast<size_t>(part) * R * D;
        a.lse_out = lse_parts + static_cast<size_t>(part) * R;
        if ((rc = run(rows_of(t)))) return rc;
        e = cudaEventRecord(h->compute_done[slot], st);
        if (e != cudaSuccess) return cuda_fail(h, e, "record compute_done");
        if (t + n_slots < n_tt) {
            e = cudaStreamWaitEvent(h->copy_stream, h->compute_done[slot], 0);
            if (e != cudaSuccess) return cuda_fail(h, e, "wait compute_done");
            if ((rc = lift(t + n_slots))) return rc;
        }
    }
    rc = launch_combine(static_cast<int>(n_parts), o_parts, lse_parts, R, D, o, lse, st);
    return rc == SKV_OK ? rc : cuda_fail(h, cudaGetLastError(), "combine launch");
}

int skv_kv_dequant_q8_0(skv_handle *h, const void *blocks, int64_t n_values, float *out, void *stream)
{
    if (!h) return SKV_EINVAL;
    h->err[0] = 0;
    if (n_values < 0 || n_values % 32) return fail(h, SKV_EINVAL, "n_values must be a multiple of 32");
    if (n_values && (!blocks || !out)) return fail(h, SKV_EINVAL, "NULL pointer");
    if ((reinterpret_cast<uintptr_t>(blocks) & 1) || (reinterpret_cast<uintptr_t>(out) & 15))
        return fail(h, SKV_EUNSUPPORTED, "blocks must be 2-byte and out 16-byte aligned");
    int rc = launch_dequant(SKV_Q8_0, blocks, n_values, out, static_cast<cudaStream_t>(stream));
    return rc == SKV_OK ? rc : cuda_fail(h, cudaGetLastError(), "dequant launch");
}

int skv_kv_dequant_q4_0(skv_handle *h, const void *blocks, int64_t n_values, float *out, void *stream)
{
    if (!h) return SKV_EINVAL;
    h->err[0] = 0;
    if (n_values < 0 || n_values % 32) return fail(h, SKV_EINVAL, "n_values must be a multiple of 32");
    if (n_values && (!blocks || !out)) return fail(h, SKV_EINVAL, "NULL pointer");
    if ((reinterpret_cast<uintptr_t>(blocks) & 1) || (reinterpret_cast<uintptr_t>(out) & 15))
        return fail(h, SKV_EUNSUPPORTED, "blocks must be 2-byte and out 16-byte aligned");
    int rc = launch_dequant(SKV_Q4_0, blocks, n_values, out, static_cast<cudaStream_t>(stream));
    return rc == SKV_OK ? rc : cuda_fail(h, cudaGetLastError(), "dequant launch");
}

int skv_gather_rows(skv_handle *h, const void *src, int64_t row_bytes, const int32_t *rows, int64_t n, void *dst,
                    void *stream)
{
    if (!h) return SKV_EINVAL;
    h->err[0] = 0;
    if (n < 0 || row_bytes < 0) return fail(h, SKV_EINVAL, "negative size");
    if (n > 0 && (!src || !rows || !dst)) return fail(h, SKV_EINVAL, "NULL pointer");
    int rc = launch_gather(src, row_bytes, rows, n, dst, static_cast<cudaStream_t>(stream));
    return rc == SKV_OK ? rc : cuda_fail(h, cudaGetLastError(), "gather launch");
}

}  // extern "C"

extern "C" {

int skv_attn_paged(skv_handle *h, const skv_shape *shape, const void *q, const void *k_pages, const void *v_pages,
                   int32_t page_rows, const int32_t *page_ids, int32_t pages_per_list, float *o, float *lse,
                   void *stream)
{
    if (!h) return SKV_EINVAL;
    h->err[0] = 0;
    return attn_paged_range(h, shape, q, k_pages, v_pages, page_rows, page_ids, pages_per_list, 0,
                            static_cast<int64_t>(pages_per_list) * page_rows, o, lse,
                            static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace skv {

int attn_paged_fused(skv_handle *h, const skv_shape *shape, const void *q, const void *k_pages, const void *v_pages,
                     const int32_t *page_ids, int32_t pages_per_list, float *o, float *lse, cudaStream_t st,
                     const DecodeArgs &fuse)
{
    if (!shape) return fail(h, SKV_EINVAL, "shape is NULL");
    if (shape->k_type != SKV_F16 || shape->v_type != SKV_F16)
        return fail(h, SKV_EUNSUPPORTED, "paged attention reads fp16 pages");
    skv_shape sh = *shape;
    sh.k_row_bytes = sh.v_row_bytes = static_cast<int64_t>(sh.Hk) * 2 * sh.D;
    int G = 0, n_cg = 0;
    int rc = check_shape(h, &sh, &G, &n_cg);
    if (rc) return rc;
    if (n_cg != 1) return fail(h, SKV_EUNSUPPORTED, "the fused block-cache attention takes one column group");
    if (!q || !o || !lse || !k_pages || !v_pages || !page_ids || pages_per_list <= 0)
        return fail(h, SKV_EINVAL, "NULL pointer or empty page lists");
    const int D = sh.D;
    const int64_t R = static_cast<int64_t>(sh.S) * sh.nq * sh.H;
    // splits of kFusedSplitPages pages: the work items the persistent grid
    // takes in lookup order, small enough that the host link stays busy to
    // the end
    const int32_t n_splits = (pages_per_list + kFusedSplitPages - 1) / kFusedSplitPages;
    if (n_splits > kMaxSplits) return fail(h, SKV_EUNSUPPORTED, "%d splits exceed %d", n_splits, kMaxSplits);
    if (static_cast<int64_t>(sh.S) * sh.Hk > kMaxUnits) return fail(h, SKV_EUNSUPPORTED, "too many units");
    DecodeArgs a = base_args(&sh, G, n_cg, q, nullptr, 0, nullptr, 0);
    a.k = static_cast<const uint8_t *>(k_pages);
    a.v = static_cast<const uint8_t *>(v_pages);
    a.row_mode = ROWS_PAGED;
    a.rows = page_ids;
    a.rows_ld = pages_per_list;
    a.rows_per_head = 1;
    a.page_rows = kDecodeTile;
    a.n_local = static_cast<int64_t>(pages_per_list) * kDecodeTile;
    a.n_splits = n_splits;
    a.split_len = static_cast<int64_t>(kFusedSplitPages) * kDecodeTile;
    a.counters = h->counters;
    a.o_out = o;
    a.lse_out = lse;
    a.status = h->status;
    a.rstate = fuse.rstate;
    a.sel = fuse.sel;
    a.n_look = fuse.n_look;
    a.page_ids_out = fuse.page_ids_out;
    a.host_k = fuse.host_k;
    a.host_v = fuse.host_v;
    a.page_ready = fuse.page_ready;
    a.epoch = fuse.epoch;
    a.steal = fuse.steal;
    if (n_splits > 1) {
        const size_t o_bytes = round_up(static_cast<size_t>(n_splits) * R * D * sizeof(float), 256);
        if ((rc = ensure_workspace(h, o_bytes + static_cast<size_t>(n_splits) * R * sizeof(float), st))) return rc;
        a.o_split = static_cast<float *>(h->workspace);
        a.lse_split = reinterpret_cast<float *>(static_cast<uint8_t *>(h->workspace) + o_bytes);
    }
    if (h->prof_before) cudaEventRecord(h->prof_before, st);
    rc = launch_decode_fused(h, a, D, st);
    if (h->prof_after) cudaEventRecord(h->prof_after, st);
    return rc;
}

int attn_paged_range(skv_handle *h, const skv_shape *shape, const void *q, const void *k_pages, const void *v_pages,
                     int32_t page_rows, const int32_t *page_ids, int32_t pages_per_list, int64_t key_lo,
                     int64_t key_hi, float *o, float *lse, cudaStream_t st)
{
    if (!shape) return fail(h, SKV_EINVAL, "shape is NULL");
    if (shape->k_type != SKV_F16 || shape->v_type != SKV_F16)
        return fail(h, SKV_EUNSUPPORTED, "paged attention reads fp16 pages");
    skv_shape sh = *shape;
    sh.k_row_bytes = sh.v_row_bytes = static_cast<int64_t>(sh.Hk) * 2 * sh.D;   // not used by the paged rows
    int G = 0, n_cg = 0;
    int rc = check_shape(h, &sh, &G, &n_cg);
    if (rc) return rc;
    if (!q || !o || !lse || !k_pages || !v_pages || !page_ids || pages_per_list < 0)
        return fail(h, SKV_EINVAL, "NULL pointer or negative page count");
    if (page_rows <= 0 || (page_rows & (page_rows - 1)) || page_rows > kMaxListSplit)
        return fail(h, SKV_EINVAL, "page_rows must be a power of two <= %d", kMaxListSplit);
    if ((reinterpret_cast<uintptr_t>(k_pages) | reinterpret_cast<uintptr_t>(v_pages)) & 15)
        return fail(h, SKV_EUNSUPPORTED, "page pools must be 16-byte aligned");
    const int D = sh.D;
    const int64_t R = static_cast<int64_t>(sh.S) * sh.nq * sh.H;
    const int64_t n_local = key_hi;
    if (key_lo < 0 || key_hi < key_lo || key_hi > static_cast<int64_t>(pages_per_list) * page_rows)
        return fail(h, SKV_EINVAL, "key range [%lld, %lld) outside the page lists", (long long)key_lo,
                    (long long)key_hi);
    if (n_local == key_lo) {
        rc = launch_combine(0, nullptr, nullptr, R, D, o, lse, st);
        return rc == SKV_OK ? rc : cuda_fail(h, cudaGetLastError(), "fill launch");
    }
    const int ctas = decode_ctas_per_sm(h, SKV_F16, SKV_F16, D);
    const int64_t units = static_cast<int64_t>(sh.S) * sh.Hk * n_cg;
    if (units > kMaxUnits) return fail(h, SKV_EUNSUPPORTED, "too many units");
    int64_t split_len = 0;
    int32_t n_splits = 0;
    // splits end on page boundaries so that each CTA's page list is whole
    const int64_t max_split = std::max<int64_t>(page_rows, (kMaxListSplit / page_rows) * page_rows);
    rc = skv_plan_splits(n_local - key_lo, units, h->sm_count, ctas, std::max(kDecodeTile, page_rows), max_split,
                         &split_len, &n_splits);
    if (rc) return fail(h, rc, "split planning failed");
    if (n_splits > kMaxSplits) return fail(h, SKV_EUNSUPPORTED, "%d splits exceed %d", n_splits, kMaxSplits);
    DecodeArgs a = base_args(&sh, G, n_cg, q, nullptr, 0, nullptr, 0);
    a.key_lo = key_lo;
    a.k = static_cast<const uint8_t *>(k_pages);
    a.v = static_cast<const uint8_t *>(v_pages);
    a.row_mode = ROWS_PAGED;
    a.rows = page_ids;
    a.rows_ld = pages_per_list;
    a.rows_per_head = 1;
    a.page_rows = page_rows;
    a.logical0 = 0;
    a.n_local = n_local;
    a.n_splits = n_splits;
    a.split_len = split_len;
    a.counters = h->counters;
    a.o_out = o;
    a.lse_out = lse;
    if (n_splits > 1) {
        const size_t o_bytes = round_up(static_cast<size_t>(n_splits) * R * D * sizeof(float), 256);
        if ((rc = ensure_workspace(h, o_bytes + static_cast<size_t>(n_splits) * R * sizeof(float), st))) return rc;
        a.o_split = static_cast<float *>(h->workspace);
        a.lse_split = reinterpret_cast<float *>(static_cast<uint8_t *>(h->workspace) + o_bytes);
    }
    return launch_decode(h, a, SKV_F16, SKV_F16, D, st);
}

}  // namespace skv
