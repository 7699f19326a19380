// bcache.cu -- selection-driven device block cache over a pinned host copy.
//
// The host copy is paged [block][Hk][block_rows][D] fp16 (the identity layout
// of "Strata compare", KV streaming, KvHostPools).  The cache unit is one
// page = one (block, KV head): block_rows rows of K and of V.  The device pool
// holds n_slots resident pages plus a per-call overflow area; page_ids map each
// selected (sequence, KV head, block) to a pool page.
//
// skv_bcache_resolve, on the device (capturable, no host round trip):
//   1. lookups: a resident page gets this call's epoch and its reference bit;
//      a missing page is claimed once (-1 -> -2, atomicCAS) into a miss list;
//   2. victims: a second-chance (CLOCK) sweep from the hand picks one slot per
//      miss, never a slot this call uses (epoch), clearing the reference bits
//      it passes; the table is re-pointed (old page -> -1, new page -> slot);
//   3. misses without a slot (demand above capacity) go to the overflow area
//      for this call only and stay non-resident;
//   4. a copy kernel reads every missed page from the host copy (16-byte
//      loads over the host link) into its pool page.
// This follows the resolve / copy design of the Strata KV-streaming page, with
// two readings of our own: the unit is a (block, KV head) page because the
// selection is per KV head, and an oversubscribed call reads its excess misses
// from the host once instead of failing.
#include <string.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

struct skv_bcache {
    skv_handle *h = nullptr;
    int64_t n_blocks = 0;
    int block_rows = 0;
    int Hk = 0;
    int D = 0;
    int n_slots = 0;
    int64_t max_lookups = 0;
    int64_t page_bytes = 0;
    uint8_t *host_k = nullptr;         // device-accessible addresses of the pinned host copy
    uint8_t *host_v = nullptr;
    int32_t *page_table = nullptr;     // [n_blocks*Hk] slot, -1, or transient markers
    int32_t *slot_page = nullptr;      // [n_slots]
    int32_t *slot_epoch = nullptr;     // [n_slots]
    int32_t *slot_ref = nullptr;       // [n_slots]
    int32_t *miss_page = nullptr;      // [max_lookups]
    int32_t *miss_dest = nullptr;      // [max_lookups]
    int32_t *miss_slot = nullptr;      // [n_slots]
    int32_t *page_ids = nullptr;       // [max_lookups] of the last resolve
    uint64_t *ctl = nullptr;           // kCtlWords, see below
    int32_t *check = nullptr;          // invariant-violation counter
    uint8_t *pool_k = nullptr;         // [(n_slots + max_lookups) pages][page_bytes]; ring: [n_slots]
    uint8_t *pool_v = nullptr;
    int64_t ring_blocks = 0;           // > 0: ring layout, page (b, k) -> slot (b % ring_blocks) * Hk + k
};

namespace skv {

// ctl words (uint64): 0 epoch, 1 hand, 2 calls, 3 lookups, 4 hits, 5 misses,
// 6 overflow, 7 last misses, 8 last overflow, 9 pages to fetch.
constexpr int kCtlWords = 16;
constexpr int kResolveThreads = 1024;

__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int &total)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        warp_sums[lane] = t;
    }
    __syncthreads();
    total = warp_sums[31];
    const int excl = x - v + (w > 0 ? warp_sums[w - 1] : 0);
    __syncthreads();
    return excl;
}

struct ResolveArgs {
    const int32_t *sel;       // [S][Hk][n_sel] block ids
    int S, n_sel, Hk;
    int n_slots;
    int64_t n_pages;          // n_blocks * Hk
    int32_t *page_table, *slot_page, *slot_epoch, *slot_ref, *miss_page, *miss_dest, *miss_slot, *page_ids;
    uint64_t *ctl;
};

__global__ void __launch_bounds__(kResolveThreads) bcache_resolve_kernel(ResolveArgs a)
{
    __shared__ int s_nmiss, s_cut;
    __shared__ int warp_sums[32];
    __shared__ unsigned long long s_lookups, s_hits;
    const int tid = threadIdx.x;
    const int epoch = static_cast<int>(a.ctl[0]) + 1;
    if (tid == 0) {
        s_nmiss = 0;
        s_lookups = 0;
        s_hits = 0;
    }
    __syncthreads();
    const int64_t n_look = static_cast<int64_t>(a.S) * a.Hk * a.n_sel;
    // 1. lookups
    unsigned long long hits = 0, looks = 0;
    for (int64_t e = tid; e < n_look; e += kResolveThreads) {
        const int k = static_cast<int>((e / a.n_sel) % a.Hk);
        const int64_t blk = a.sel[e];
        if (blk < 0 || blk * a.Hk + k >= a.n_pages) continue;    // rejected on the host; never indexes out
        const int64_t p = blk * a.Hk + k;
        ++looks;
        const int v = a.page_table[p];
        if (v >= 0) {
            a.slot_epoch[v] = epoch;
            a.slot_ref[v] = 1;
            ++hits;
        } else if (v == -1 && atomicCAS(a.page_table + p, -1, -2) == -1) {
            a.miss_page[atomicAdd(&s_nmiss, 1)] = static_cast<int32_t>(p);
        }
    }
    atomicAdd(&s_lookups, looks);
    atomicAdd(&s_hits, hits);
    __syncthreads();
    // 2. CLOCK victims: one slot per miss, never a slot used by this call.
    const int need = s_nmiss;
    const int n = a.n_slots;
    int hand = static_cast<int>(a.ctl[1]);
    int got = 0;
    for (int scanned = 0; got < need && scanned < 2 * n + kResolveThreads; scanned += kResolveThreads) {
        const int j = static_cast<int>((static_cast<int64_t>(hand) + tid) % n);
        const bool in_window = tid < n;                          // a window never wraps onto itself
        const bool current = in_window && a.slot_epoch[j] == epoch;
        const bool cand = in_window && !current && (a.slot_page[j] < 0 || a.slot_ref[j] == 0);
        int total = 0;
        const int rank = block_exclusive_scan(cand ? 1 : 0, warp_sums, total);
        const int want = need - got;
        if (tid == 0) s_cut = min(n, kResolveThreads);
        __syncthreads();
        if (cand && rank == want - 1) s_cut = tid + 1;           // the hand stops after the last slot taken
        __syncthreads();
        const int cut = s_cut;
        if (cand && rank < want) {
            a.miss_slot[got + rank] = j;
            a.slot_epoch[j] = epoch;                             // taken: a later window must not take it again
        } else if (in_window && tid < cut && !current) {
            a.slot_ref[j] = 0;                                   // second chance used up
        }
        got += min(total, want);
        hand = static_cast<int>((static_cast<int64_t>(hand) + cut) % n);
        __syncthreads();
    }
    const int placed = min(got, need);
    // 3. re-point the table; overflow misses get a transient marker
    for (int m = tid; m < need; m += kResolveThreads) {
        const int p = a.miss_page[m];
        if (m < placed) {
            const int sl = a.miss_slot[m];
            const int old = a.slot_page[sl];
            if (old >= 0) a.page_table[old] = -1;
            a.slot_page[sl] = p;
            a.slot_ref[sl] = 1;
            a.page_table[p] = sl;
            a.miss_dest[m] = sl;
        } else {
            a.page_table[p] = -3 - (m - placed);
            a.miss_dest[m] = n + (m - placed);
        }
    }
    __syncthreads();
    // 4. page ids of every lookup
    for (int64_t e = tid; e < n_look; e += kResolveThreads) {
        const int k = static_cast<int>((e / a.n_sel) % a.Hk);
        const int64_t blk = a.sel[e];
        if (blk < 0 || blk * a.Hk + k >= a.n_pages) {
            a.page_ids[e] = -1;
            continue;
        }
        const int v = a.page_table[blk * a.Hk + k];
        a.page_ids[e] = v >= 0 ? v : n + (-3 - v);
    }
    __syncthreads();
    // 5. overflow pages are not resident after this call
    for (int m = placed + tid; m < need; m += kResolveThreads) a.page_table[a.miss_page[m]] = -1;
    if (tid == 0) {
        a.ctl[0] = static_cast<uint64_t>(epoch);
        a.ctl[1] = static_cast<uint64_t>(hand);
        a.ctl[2] += 1;
        a.ctl[3] += s_lookups;
        a.ctl[4] += s_hits;
        a.ctl[5] += static_cast<uint64_t>(need);
        a.ctl[6] += static_cast<uint64_t>(need - placed);
        a.ctl[7] = static_cast<uint64_t>(need);
        a.ctl[8] = static_cast<uint64_t>(need - placed);
        a.ctl[9] = static_cast<uint64_t>(need);
    }
}

// Copy every missed page (K and V) from the host copy into its pool page:
// one CTA per page in turn, 16 bytes per thread per load, 4 loads in flight.
__global__ void __launch_bounds__(256) bcache_fetch_kernel(const uint64_t *__restrict__ ctl,
                                                           const int32_t *__restrict__ miss_page,
                                                           const int32_t *__restrict__ miss_dest,
                                                           const uint8_t *__restrict__ host_k,
                                                           const uint8_t *__restrict__ host_v, uint8_t *pool_k,
                                                           uint8_t *pool_v, int64_t page_bytes)
{
    const int n_fetch = static_cast<int>(ctl[9]);
    const int64_t n16 = page_bytes / 16;
    for (int m = blockIdx.x; m < n_fetch; m += gridDim.x) {
        const int64_t src = static_cast<int64_t>(miss_page[m]) * page_bytes;
        const int64_t dst = static_cast<int64_t>(miss_dest[m]) * page_bytes;
        const uint4 *sk = reinterpret_cast<const uint4 *>(host_k + src);
        const uint4 *sv = reinterpret_cast<const uint4 *>(host_v + src);
        uint4 *dk = reinterpret_cast<uint4 *>(pool_k + dst);
        uint4 *dv = reinterpret_cast<uint4 *>(pool_v + dst);
        for (int64_t i = threadIdx.x; i < n16; i += 2 * blockDim.x) {
            const int64_t i2 = i + blockDim.x;
            const uint4 a0 = sk[i], b0 = sv[i];
            uint4 a1 = make_uint4(0, 0, 0, 0), b1 = a1;
            if (i2 < n16) {
                a1 = sk[i2];
                b1 = sv[i2];
            }
            dk[i] = a0;
            dv[i] = b0;
            if (i2 < n16) {
                dk[i2] = a1;
                dv[i2] = b1;
            }
        }
    }
}

// Write-through append (the writers of the Strata KV-streaming page): cache
// position p is row p % block_rows of block p / block_rows; each (position, KV
// head) writes its fp16 K and V row into the host copy always and into the
// pool page only when the page is resident (page_table >= 0), so a resident
// page never differs from the host copy.  One warp per (position, KV head);
// each lane converts 8 values into one 16-byte store.  Positions outside
// [0, n_blocks * block_rows) are skipped and set bit 1 of *status.
__global__ void __launch_bounds__(256) bcache_append_kernel(const float *__restrict__ k_new,
                                                            const float *__restrict__ v_new,
                                                            const int32_t *__restrict__ pos, int n, int Hk, int D,
                                                            int block_rows, int64_t n_blocks,
                                                            const int32_t *__restrict__ page_table, uint8_t *host_k,
                                                            uint8_t *host_v, uint8_t *pool_k, uint8_t *pool_v,
                                                            int64_t page_bytes, int *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t item = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (item >= static_cast<int64_t>(n) * Hk) return;
    const int r = static_cast<int>(item / Hk);
    const int k = static_cast<int>(item % Hk);
    const int64_t p = pos[r];
    if (p < 0) return;
    if (p >= n_blocks * block_rows) {
        if (lane == 0 && k == 0) atomicOr(status, 2);
        return;
    }
    const int64_t page = (p / block_rows) * Hk + k;
    const int slot = page_table[page];
    const int64_t off = (p % block_rows) * D * 2;                 // byte offset of the row inside its page
    const int chunks = D / 8;                                     // 16-byte chunks per row
    for (int c = lane; c < 2 * chunks; c += 32) {
        const bool is_v = c >= chunks;
        const int cc = is_v ? c - chunks : c;
        const float4 *src = reinterpret_cast<const float4 *>((is_v ? v_new : k_new) + item * D) + 2 * cc;
        const float4 a = src[0], b = src[1];
        __half2 h[4] = {__floats2half2_rn(a.x, a.y), __floats2half2_rn(a.z, a.w), __floats2half2_rn(b.x, b.y),
                        __floats2half2_rn(b.z, b.w)};
        const uint4 w = *reinterpret_cast<const uint4 *>(h);
        reinterpret_cast<uint4 *>((is_v ? host_v : host_k) + page * page_bytes + off)[cc] = w;
        if (slot >= 0) reinterpret_cast<uint4 *>((is_v ? pool_v : pool_k) + slot * page_bytes + off)[cc] = w;
    }
}

__global__ void bcache_reset_kernel(int32_t *page_table, int64_t n_pages, int32_t *slot_page, int32_t *slot_epoch,
                                    int32_t *slot_ref, int n_slots, uint64_t *ctl)
{
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = i0; i < n_pages; i += st) page_table[i] = -1;
    for (int64_t i = i0; i < n_slots; i += st) {
        slot_page[i] = -1;
        slot_epoch[i] = 0;
        slot_ref[i] = 0;
    }
    if (i0 < kCtlWords) ctl[i0] = 0;
}

// Count violations of: page_table[p] = s >= 0  <=>  slot_page[s] = p, and no
// page left at a transient marker (< -1).
__global__ void bcache_check_kernel(const int32_t *page_table, int64_t n_pages, const int32_t *slot_page,
                                    int n_slots, int32_t *violations)
{
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t p = i0; p < n_pages; p += st) {
        const int v = page_table[p];
        if (v < -1 || v >= n_slots || (v >= 0 && slot_page[v] != p)) atomicAdd(violations, 1);
    }
    for (int64_t s = i0; s < n_slots; s += st) {
        const int p = slot_page[s];
        if (p < -1 || p >= n_pages || (p >= 0 && page_table[p] != s)) atomicAdd(violations, 1);
    }
}

// Ring layout (the Strata KV-streaming page's ring for a reader of the last
// cells only): a static table, page (block b, head k) -> slot
// (b % ring_blocks) * Hk + k, no resolve.  Appends then write the host copy
// and the ring slot of every row; a newer block overwrites the slot of the
// block ring_blocks before it.
__global__ void ring_init_kernel(int32_t *page_table, int64_t n_pages, int Hk, int64_t ring_blocks,
                                 int32_t *slot_page, int n_slots, uint64_t *ctl)
{
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t p = i0; p < n_pages; p += st)
        page_table[p] = static_cast<int32_t>(((p / Hk) % ring_blocks) * Hk + p % Hk);
    for (int64_t i = i0; i < n_slots; i += st) slot_page[i] = -1;
    if (i0 < kCtlWords) ctl[i0] = 0;
}

// Refill: the pages of blocks [first, first + n_blk) become the fetch list
// (page -> its ring slot); the fetch kernel then copies them from the host.
__global__ void ring_restore_kernel(int64_t first, int n_blk, int Hk, int64_t ring_blocks, int32_t *miss_page,
                                    int32_t *miss_dest, int32_t *slot_page, uint64_t *ctl)
{
    const int n = n_blk * Hk;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int64_t b = first + i / Hk;
        const int k = i % Hk;
        const int32_t slot = static_cast<int32_t>((b % ring_blocks) * Hk + k);
        miss_page[i] = static_cast<int32_t>(b * Hk + k);
        miss_dest[i] = slot;
        slot_page[slot] = static_cast<int32_t>(b * Hk + k);
    }
    if (threadIdx.x == 0) ctl[9] = static_cast<uint64_t>(n);
}

// Page lists [S][Hk][n_blk] of blocks first .. first + n_blk - 1 through the ring.
__global__ void ring_ids_kernel(int64_t first, int n_blk, int S, int Hk, int64_t ring_blocks, int32_t *ids)
{
    const int64_t n = static_cast<int64_t>(S) * Hk * n_blk;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int j = static_cast<int>(i % n_blk);
        const int k = static_cast<int>((i / n_blk) % Hk);
        ids[i] = static_cast<int32_t>(((first + j) % ring_blocks) * Hk + k);
    }
}

// Ring invariant: every page maps to its static slot.
__global__ void ring_check_kernel(const int32_t *page_table, int64_t n_pages, int Hk, int64_t ring_blocks,
                                  int32_t *violations)
{
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t p = i0; p < n_pages; p += st)
        if (page_table[p] != ((p / Hk) % ring_blocks) * Hk + p % Hk) atomicAdd(violations, 1);
}

}  // namespace skv

using namespace skv;

extern "C" {

int skv_bcache_destroy(skv_bcache *c)
{
    if (!c) return SKV_OK;
    cudaFree(c->page_table);
    cudaFree(c->slot_page);
    cudaFree(c->slot_epoch);
    cudaFree(c->slot_ref);
    cudaFree(c->miss_page);
    cudaFree(c->miss_dest);
    cudaFree(c->miss_slot);
    cudaFree(c->page_ids);
    cudaFree(c->ctl);
    cudaFree(c->check);
    cudaFree(c->pool_k);
    cudaFree(c->pool_v);
    delete c;
    return SKV_OK;
}

int skv_bcache_reset(skv_bcache *c, void *stream)
{
    if (!c) return SKV_EINVAL;
    const int64_t n_pages = c->n_blocks * c->Hk;
    if (c->ring_blocks > 0)
        ring_init_kernel<<<256, 256, 0, static_cast<cudaStream_t>(stream)>>>(c->page_table, n_pages, c->Hk,
                                                                            c->ring_blocks, c->slot_page,
                                                                            c->n_slots, c->ctl);
    else
        bcache_reset_kernel<<<256, 256, 0, static_cast<cudaStream_t>(stream)>>>(
            c->page_table, n_pages, c->slot_page, c->slot_epoch, c->slot_ref, c->n_slots, c->ctl);
    return cuda_fail(c->h, cudaGetLastError(), "block-cache reset");
}

static int bcache_create_impl(skv_handle *h, int64_t n_blocks, int32_t block_rows, int32_t Hk, int32_t D,
                              int32_t n_slots, int64_t max_lookups, int64_t ring_blocks, const void *host_k,
                              const void *host_v, skv_bcache **out)
{
    if (!h || !out) return SKV_EINVAL;
    h->err[0] = 0;
    *out = nullptr;
    if (n_blocks <= 0 || Hk <= 0 || n_slots <= 0 || max_lookups <= 0 || (D != 64 && D != 128))
        return fail(h, SKV_EINVAL, "bad block-cache sizes");
    if (block_rows <= 0 || (block_rows & (block_rows - 1)) || block_rows > kMaxListSplit)
        return fail(h, SKV_EINVAL, "block_rows must be a power of two <= %d", kMaxListSplit);
    if (n_blocks * Hk > 0x7fffffffLL || n_slots + max_lookups > 0x7fffffffLL)
        return fail(h, SKV_EUNSUPPORTED, "too many pages");
    if (!host_k || !host_v) return fail(h, SKV_EINVAL, "host copy is NULL");
    const void *dk = nullptr, *dv = nullptr;
    for (int i = 0; i < 2; ++i) {
        const void *p = i ? host_v : host_k;
        cudaPointerAttributes at;
        cudaError_t e = cudaPointerGetAttributes(&at, p);
        if (e != cudaSuccess || at.type != cudaMemoryTypeHost || !at.devicePointer) {
            cudaGetLastError();
            return fail(h, SKV_ENOTPINNED, "host copy %p is not page-locked, device-mapped memory", p);
        }
        (i ? dv : dk) = at.devicePointer;
    }
    skv_bcache *c = new (std::nothrow) skv_bcache();
    if (!c) return SKV_ENOMEM;
    c->h = h;
    c->n_blocks = n_blocks;
    c->block_rows = block_rows;
    c->Hk = Hk;
    c->D = D;
    c->n_slots = n_slots;
    c->max_lookups = max_lookups;
    c->ring_blocks = ring_blocks;
    c->page_bytes = static_cast<int64_t>(block_rows) * D * 2;
    c->host_k = static_cast<uint8_t *>(const_cast<void *>(dk));
    c->host_v = static_cast<uint8_t *>(const_cast<void *>(dv));
    const int64_t n_pages = n_blocks * Hk;
    const size_t pool_pages = static_cast<size_t>(n_slots) + (ring_blocks > 0 ? 0 : static_cast<size_t>(max_lookups));
    cudaError_t e = cudaSuccess;
    auto A = [&](void **p, size_t bytes) {
        if (e == cudaSuccess) e = cudaMalloc(p, bytes);
    };
    A(reinterpret_cast<void **>(&c->page_table), sizeof(int32_t) * n_pages);
    A(reinterpret_cast<void **>(&c->slot_page), sizeof(int32_t) * n_slots);
    A(reinterpret_cast<void **>(&c->slot_epoch), sizeof(int32_t) * n_slots);
    A(reinterpret_cast<void **>(&c->slot_ref), sizeof(int32_t) * n_slots);
    A(reinterpret_cast<void **>(&c->miss_page), sizeof(int32_t) * max_lookups);
    A(reinterpret_cast<void **>(&c->miss_dest), sizeof(int32_t) * max_lookups);
    A(reinterpret_cast<void **>(&c->miss_slot), sizeof(int32_t) * n_slots);
    A(reinterpret_cast<void **>(&c->page_ids), sizeof(int32_t) * max_lookups);
    A(reinterpret_cast<void **>(&c->ctl), sizeof(uint64_t) * kCtlWords);
    A(reinterpret_cast<void **>(&c->check), sizeof(int32_t));
    A(reinterpret_cast<void **>(&c->pool_k), pool_pages * c->page_bytes);
    A(reinterpret_cast<void **>(&c->pool_v), pool_pages * c->page_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        skv_bcache_destroy(c);
        return fail(h, SKV_ENOMEM, "block-cache allocation: %s", cudaGetErrorString(e));
    }
    int rc = skv_bcache_reset(c, nullptr);
    if (rc == SKV_OK) rc = cuda_fail(h, cudaDeviceSynchronize(), "block-cache init");
    if (rc) {
        skv_bcache_destroy(c);
        return rc;
    }
    *out = c;
    return SKV_OK;
}

int skv_bcache_create(skv_handle *h, int64_t n_blocks, int32_t block_rows, int32_t Hk, int32_t D, int32_t n_slots,
                      int64_t max_lookups, const void *host_k, const void *host_v, skv_bcache **out)
{
    return bcache_create_impl(h, n_blocks, block_rows, Hk, D, n_slots, max_lookups, 0, host_k, host_v, out);
}

int skv_bcache_create_ring(skv_handle *h, int64_t n_blocks, int32_t block_rows, int32_t Hk, int32_t D,
                           int32_t ring_blocks, int32_t max_seqs, const void *host_k, const void *host_v,
                           skv_bcache **out)
{
    if (!h || !out) return SKV_EINVAL;
    h->err[0] = 0;
    if (ring_blocks <= 0 || ring_blocks > n_blocks || max_seqs <= 0 || Hk <= 0)
        return fail(h, SKV_EINVAL, "ring of %d blocks over %lld blocks, %d sequences", ring_blocks,
                    (long long)n_blocks, max_seqs);
    const int64_t slots = static_cast<int64_t>(ring_blocks) * Hk;
    if (slots > 0x7fffffffLL || slots * max_seqs > 0x7fffffffLL) return fail(h, SKV_EUNSUPPORTED, "ring too large");
    return bcache_create_impl(h, n_blocks, block_rows, Hk, D, static_cast<int32_t>(slots), slots * max_seqs,
                              ring_blocks, host_k, host_v, out);
}

int skv_bcache_resolve(skv_bcache *c, const int32_t *sel, int32_t S, int32_t n_sel, int32_t *page_ids, void *stream)
{
    if (!c) return SKV_EINVAL;
    skv_handle *h = c->h;
    h->err[0] = 0;
    if (c->ring_blocks > 0) return fail(h, SKV_EUNSUPPORTED, "a ring cache has a static table and no resolve");
    if (!sel || S <= 0 || n_sel <= 0) return fail(h, SKV_EINVAL, "bad selection");
    const int64_t n_look = static_cast<int64_t>(S) * c->Hk * n_sel;
    if (n_look > c->max_lookups) return fail(h, SKV_EINVAL, "%lld lookups exceed max_lookups %lld",
                                             (long long)n_look, (long long)c->max_lookups);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ResolveArgs a;
    a.sel = sel;
    a.S = S;
    a.n_sel = n_sel;
    a.Hk = c->Hk;
    a.n_slots = c->n_slots;
    a.n_pages = c->n_blocks * c->Hk;
    a.page_table = c->page_table;
    a.slot_page = c->slot_page;
    a.slot_epoch = c->slot_epoch;
    a.slot_ref = c->slot_ref;
    a.miss_page = c->miss_page;
    a.miss_dest = c->miss_dest;
    a.miss_slot = c->miss_slot;
    a.page_ids = page_ids ? page_ids : c->page_ids;
    a.ctl = c->ctl;
    bcache_resolve_kernel<<<1, kResolveThreads, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(h, e, "resolve launch");
    bcache_fetch_kernel<<<2 * h->sm_count, 256, 0, st>>>(c->ctl, c->miss_page, c->miss_dest, c->host_k, c->host_v,
                                                         c->pool_k, c->pool_v, c->page_bytes);
    return cuda_fail(h, cudaGetLastError(), "fetch launch");
}

int skv_bcache_append(skv_bcache *c, const float *k_new, const float *v_new, const int32_t *positions, int32_t n,
                      void *stream)
{
    if (!c) return SKV_EINVAL;
    skv_handle *h = c->h;
    h->err[0] = 0;
    if (n < 0) return fail(h, SKV_EINVAL, "negative row count");
    if (n == 0) return SKV_OK;
    if (!k_new || !v_new || !positions) return fail(h, SKV_EINVAL, "NULL pointer");
    if (reinterpret_cast<uintptr_t>(k_new) % 16 || reinterpret_cast<uintptr_t>(v_new) % 16)
        return fail(h, SKV_EUNSUPPORTED, "k_new / v_new must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(c->host_k) % 16 || reinterpret_cast<uintptr_t>(c->host_v) % 16)
        return fail(h, SKV_EUNSUPPORTED, "the host copy must be 16-byte aligned for appends");
    const int64_t items = static_cast<int64_t>(n) * c->Hk;
    if ((items + 7) / 8 > 0x7fffffffLL) return fail(h, SKV_EUNSUPPORTED, "too many rows for one launch");
    bcache_append_kernel<<<static_cast<unsigned>((items + 7) / 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        k_new, v_new, positions, n, c->Hk, c->D, c->block_rows, c->n_blocks, c->page_table, c->host_k, c->host_v,
        c->pool_k, c->pool_v, c->page_bytes, h->status);
    return cuda_fail(h, cudaGetLastError(), "block-cache append");
}

int skv_bcache_stats(skv_bcache *c, skv_bcache_counters *out)
{
    if (!c || !out) return SKV_EINVAL;
    uint64_t w[kCtlWords];
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(w, c->ctl, sizeof(w), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(c->h, e, "reading block-cache counters");
    out->calls = w[2];
    out->lookups = w[3];
    out->hits = w[4];
    out->misses = w[5];
    out->overflow = w[6];
    out->last_misses = static_cast<int64_t>(w[7]);
    out->last_overflow = static_cast<int64_t>(w[8]);
    return SKV_OK;
}

int skv_bcache_check(skv_bcache *c, int32_t *violations)
{
    if (!c || !violations) return SKV_EINVAL;
    cudaError_t e = cudaMemset(c->check, 0, sizeof(int32_t));
    if (e != cudaSuccess) return cuda_fail(c->h, e, "check reset");
    if (c->ring_blocks > 0)
        ring_check_kernel<<<128, 256>>>(c->page_table, c->n_blocks * c->Hk, c->Hk, c->ring_blocks, c->check);
    else
        bcache_check_kernel<<<128, 256>>>(c->page_table, c->n_blocks * c->Hk, c->slot_page, c->n_slots, c->check);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(violations, c->check, sizeof(int32_t), cudaMemcpyDeviceToHost);
    return cuda_fail(c->h, e, "block-cache check");
}

int skv_bcache_pool(const skv_bcache *c, const void **k_pages, const void **v_pages, int64_t *n_pool_pages,
                    const int32_t **last_page_ids)
{
    if (!c) return SKV_EINVAL;
    if (k_pages) *k_pages = c->pool_k;
    if (v_pages) *v_pages = c->pool_v;
    if (n_pool_pages) *n_pool_pages = c->n_slots + (c->ring_blocks > 0 ? 0 : c->max_lookups);
    if (last_page_ids) *last_page_ids = c->page_ids;
    return SKV_OK;
}

}  // extern "C"

extern "C" int skv_bcache_attn(skv_bcache *c, const skv_shape *shape, const void *q, const int32_t *sel,
                               int32_t n_sel, float *o, float *lse, void *stream)
{
    if (!c || !shape) return SKV_EINVAL;
    if (shape->Hk != c->Hk || shape->D != c->D)
        return skv::fail(c->h, SKV_EINVAL, "shape (Hk=%d, D=%d) does not match the cache (Hk=%d, D=%d)", shape->Hk,
                         shape->D, c->Hk, c->D);
    int rc = skv_bcache_resolve(c, sel, shape->S, n_sel, c->page_ids, stream);
    if (rc) return rc;
    return skv_attn_paged(c->h, shape, q, c->pool_k, c->pool_v, c->block_rows, c->page_ids, n_sel, o, lse, stream);
}

extern "C" int skv_bcache_ring_restore(skv_bcache *c, int64_t n_keys, void *stream)
{
    if (!c) return SKV_EINVAL;
    skv_handle *h = c->h;
    h->err[0] = 0;
    if (c->ring_blocks <= 0) return skv::fail(h, SKV_EINVAL, "not a ring cache");
    if (n_keys < 0 || n_keys > c->n_blocks * c->block_rows)
        return skv::fail(h, SKV_EINVAL, "n_keys %lld outside the cache", (long long)n_keys);
    if (n_keys == 0) return SKV_OK;
    const int64_t last = (n_keys - 1) / c->block_rows;
    const int64_t first = std::max<int64_t>(0, last - c->ring_blocks + 1);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ring_restore_kernel<<<1, 256, 0, st>>>(first, static_cast<int>(last - first + 1), c->Hk, c->ring_blocks,
                                          c->miss_page, c->miss_dest, c->slot_page, c->ctl);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return skv::cuda_fail(h, e, "ring restore launch");
    bcache_fetch_kernel<<<2 * h->sm_count, 256, 0, st>>>(c->ctl, c->miss_page, c->miss_dest, c->host_k, c->host_v,
                                                         c->pool_k, c->pool_v, c->page_bytes);
    return skv::cuda_fail(h, cudaGetLastError(), "ring fetch launch");
}

extern "C" int skv_bcache_ring_attn(skv_bcache *c, const skv_shape *shape, const void *q, int64_t n_keys,
                                    int64_t window, float *o, float *lse, void *stream)
{
    if (!c || !shape) return SKV_EINVAL;
    skv_handle *h = c->h;
    h->err[0] = 0;
    if (c->ring_blocks <= 0) return skv::fail(h, SKV_EINVAL, "not a ring cache");
    if (shape->Hk != c->Hk || shape->D != c->D)
        return skv::fail(h, SKV_EINVAL, "shape (Hk=%d, D=%d) does not match the cache (Hk=%d, D=%d)", shape->Hk,
                         shape->D, c->Hk, c->D);
    if (n_keys < 0 || n_keys > c->n_blocks * c->block_rows)
        return skv::fail(h, SKV_EINVAL, "n_keys %lld outside the cache", (long long)n_keys);
    const int64_t br = c->block_rows;
    const int64_t last = n_keys > 0 ? (n_keys - 1) / br : 0;
    const int64_t ring_first = std::max<int64_t>(0, last - c->ring_blocks + 1) * br;   // oldest cell in the ring
    const int64_t lo = window > 0 ? std::max<int64_t>(0, n_keys - window) : ring_first;
    if (lo < ring_first)
        return skv::fail(h, SKV_EINVAL, "window of %lld cells reaches past the ring (oldest cell %lld)",
                         (long long)window, (long long)ring_first);
    const int64_t first_blk = lo / br;
    const int n_blk = n_keys > lo ? static_cast<int>(last - first_blk + 1) : 0;
    if (static_cast<int64_t>(shape->S) * c->Hk * std::max(n_blk, 1) > c->max_lookups)
        return skv::fail(h, SKV_EINVAL, "%d sequences exceed the ring's page-list capacity", shape->S);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n_blk > 0) {
        ring_ids_kernel<<<64, 256, 0, st>>>(first_blk, n_blk, shape->S, c->Hk, c->ring_blocks, c->page_ids);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return skv::cuda_fail(h, e, "ring page-list launch");
    }
    return skv::attn_paged_range(h, shape, q, c->pool_k, c->pool_v, c->block_rows, c->page_ids, std::max(n_blk, 1),
                                 lo - first_blk * br, n_keys - first_blk * br, o, lse, st);
}
