// bcache.cu -- selection-driven device block cache over a pinned host copy.
//
// The host copy is paged [block][Hk][block_rows][D] fp16 (the identity layout
// of "Strata compare", KV streaming, KvHostPools).  The cache unit is one
// page = one (block, KV head): block_rows rows of K and of V.  The device pool
// holds n_slots resident pages plus a per-call overflow area; page ids map each
// selected (sequence, KV head, block) to a pool page.
//
// The page's guarantees for a resolve are kept: a page this call reads is never
// evicted by it, each missing page is claimed once however many lookups name
// it, and victims are chosen by second chance (CLOCK).  The structure is this
// library's own, three stream-ordered launches with no host round trip:
//   lookup  (grid)   a resident page is stamped with the call's epoch and its
//                    reference bit; a missing page records, by one atomic
//                    maximum on its claim word, the first lookup that names it;
//   claim + victims + placement  (1 CTA)  the missed pages are listed in the
//                    order of their first lookups (a block scan over the
//                    lookups), so every decision below is deterministic; every
//                    slot is classed, in hand order, as in use by this call,
//                    cold (free or unreferenced) or warm (referenced), and one
//                    scan of the class counts gives the whole sweep at once --
//                    the first `need` cold slots, then (when the cold ones run
//                    out, after the hand has passed and cleared every warm
//                    slot) warm slots in hand order; misses beyond cold + warm
//                    go to the overflow area, decided here once for the call;
//                    victims are re-pointed (old page -> -1, new page -> slot);
//   fetch + ids  (persistent grid)  every missed page is copied from the host
//                    copy into its pool page over the host link, and every
//                    lookup gets its pool page id.
// Attention then reads the pages through the ids.  skv_bcache_attn on 64-row
// pages copies and attends in one pass instead: the lookup, the fused
// attention (decode_kernel.cuh), whose CTA 0 runs the claim / victim /
// placement pass while the other CTAs stage every missed page from the host
// copy in the overflow page of its first lookup, and a last launch that moves
// the misses placed in slots there (bcache_attn_fused below).  (Attending to
// the pages resident at entry on another stream while the misses stream was
// measured and not kept: on this part a kernel that saturates HBM slows the
// host-link copy beside it by about as much as it takes.)  Two readings of
// our own: the unit is a (block, KV head) page because the selection is per KV
// head, and an oversubscribed call reads its excess misses from the host once
// instead of failing.
#include <string.h>

#include <algorithm>

#include "bcache_resolve.cuh"
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
    int32_t *page_table = nullptr;     // [n_blocks*Hk] slot or -1
    uint64_t *page_claim = nullptr;    // [n_blocks*Hk] epoch << 32 | ~lookup of the call that last missed the page
    int32_t *page_miss = nullptr;      // [n_blocks*Hk] its index in that call's miss list
    int32_t *slot_page = nullptr;      // [n_slots]
    int32_t *slot_epoch = nullptr;     // [n_slots] epoch of the last call that used the slot
    int32_t *slot_ref = nullptr;       // [n_slots] reference bit
    int32_t *victim = nullptr;         // [n_slots] slots chosen for this call's misses, in order
    int32_t *miss_page = nullptr;      // [max_lookups]
    int32_t *miss_dest = nullptr;      // [max_lookups] pool page each miss is fetched into
    int32_t *page_ids = nullptr;       // [max_lookups] of the last resolve
    uint64_t *ctl = nullptr;           // kCtlWords, see below
    int32_t *check = nullptr;          // invariant-violation counter
    uint8_t *pool_k = nullptr;         // [(n_slots + max_lookups) pages][page_bytes]; ring: [n_slots]
    uint8_t *pool_v = nullptr;
    int64_t ring_blocks = 0;           // > 0: ring layout, page (b, k) -> slot (b % ring_blocks) * Hk + k
    void *rstate = nullptr;            // the ResolveState of this cache, in device memory (fused attention)
    int32_t *page_ready = nullptr;     // [pool pages] epoch of the call that last published the page
};

namespace skv {

// Lookup pass (this call's epoch is one past the last resolve's).
__global__ void __launch_bounds__(256) bcache_lookup_kernel(ResolveState r, const int32_t *__restrict__ sel,
                                                            int64_t n_look, int n_sel, int Hk)
{
    const int epoch = static_cast<int>(r.ctl[0]) + 1;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        r.ctl[kCtlEpochNow] = static_cast<uint64_t>(epoch);
        r.ctl[kCtlSteal] = 0;
    }
    unsigned looks = 0, hits = 0;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_look;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t p = lookup_page(sel, e, n_sel, Hk, r.n_pages);
        if (p >= 0) {
            ++looks;
            const int s = r.page_table[p];
            if (s >= 0) {
                r.slot_epoch[s] = epoch;          // in use: no victim this call
                r.slot_ref[s] = 1;
                ++hits;
            } else {
                atomicMax(reinterpret_cast<unsigned long long *>(r.page_claim + p), claim_key(epoch, e));
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        looks += __shfl_xor_sync(0xffffffffu, looks, o);
        hits += __shfl_xor_sync(0xffffffffu, hits, o);
    }
    if ((threadIdx.x & 31) == 0 && looks) {
        atomicAdd(reinterpret_cast<unsigned long long *>(r.ctl + 3), static_cast<unsigned long long>(looks));
        atomicAdd(reinterpret_cast<unsigned long long *>(r.ctl + 4), static_cast<unsigned long long>(hits));
    }
}

// Claim, victim and placement pass as its own launch (one CTA).
__global__ void __launch_bounds__(kVictimThreads) bcache_victim_kernel(ResolveState r, const int32_t *__restrict__ sel,
                                                                       int64_t n_look, int n_sel, int Hk)
{
    victim_pass<kVictimThreads>(r, sel, n_look, n_sel, Hk);
}

// Fetch and ids pass, a persistent grid of one CTA per SM.
//  * With sel != NULL, the pool page id of every lookup: its slot (hits, and
//    misses placed in a slot by this call) or its overflow page.
//  * Every page of the miss list (count entries) is copied from the host copy
//    into its pool page: one warp per page, each lane keeping 8 loads of 16
//    bytes in flight over the host link.  Warps take pages from a counter
//    (ctl word kCtlNext, zero before the launch), so CTAs that start late --
//    the SMs busy with other work -- take fewer pages instead of holding up
//    the copy.
constexpr int kFetchThreads = 256;
__global__ void __launch_bounds__(kFetchThreads, 1) bcache_fetch_kernel(const uint64_t *__restrict__ count,
                                                                        const int32_t *__restrict__ miss_page,
                                                                        const int32_t *__restrict__ miss_dest,
                                                                        const uint8_t *__restrict__ host_k,
                                                                        const uint8_t *__restrict__ host_v,
                                                                        uint8_t *pool_k, uint8_t *pool_v,
                                                                        int64_t page_bytes, ResolveState r,
                                                                        const int32_t *__restrict__ sel, int64_t n_look,
                                                                        int n_sel, int Hk, int32_t *__restrict__ ids)
{
    if (sel) {
        const uint32_t epoch = static_cast<uint32_t>(r.ctl[0]);
        for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_look;
             e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const int64_t p = lookup_page(sel, e, n_sel, Hk, r.n_pages);
            int32_t id = -1;
            if (p >= 0)
                id = (r.page_claim[p] >> 32) == epoch ? r.miss_dest[r.page_miss[p]]   // missed by this call
                                                      : r.page_table[p];
            ids[e] = id;
        }
    }
    constexpr int kU = 4;
    const int64_t n = static_cast<int64_t>(*count);
    const int lane = threadIdx.x & 31;
    const int64_t n16 = page_bytes / 16;
    unsigned long long *next = reinterpret_cast<unsigned long long *>(r.ctl + kCtlNext);
    for (;;) {
        unsigned long long i = 0;
        if (lane == 0) i = atomicAdd(next, 1ull);
        const int64_t m = static_cast<int64_t>(__shfl_sync(0xffffffffu, i, 0));
        if (m >= n) break;
        const int64_t src = static_cast<int64_t>(miss_page[m]) * page_bytes;
        const int64_t dst = static_cast<int64_t>(miss_dest[m]) * page_bytes;
        const uint4 *sk = reinterpret_cast<const uint4 *>(host_k + src);
        const uint4 *sv = reinterpret_cast<const uint4 *>(host_v + src);
        uint4 *dk = reinterpret_cast<uint4 *>(pool_k + dst);
        uint4 *dv = reinterpret_cast<uint4 *>(pool_v + dst);
        for (int64_t base = 0; base < n16; base += 32 * kU) {
            uint4 a[kU], b[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t i = base + u * 32 + lane;
                if (i < n16) {
                    a[u] = sk[i];
                    b[u] = sv[i];
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t i = base + u * 32 + lane;
                if (i < n16) {
                    dk[i] = a[u];
                    dv[i] = b[u];
                }
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

__global__ void bcache_reset_kernel(int32_t *page_table, uint64_t *page_claim, int64_t n_pages, int32_t *slot_page,
                                    int32_t *slot_epoch, int32_t *slot_ref, int n_slots, uint64_t *ctl,
                                    int32_t *page_ready, int64_t n_pool)
{
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t st = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = i0; i < n_pages; i += st) {
        page_table[i] = -1;
        page_claim[i] = 0;
    }
    for (int64_t i = i0; i < n_pool; i += st) page_ready[i] = 0;   // the stamps restart with the epochs
    for (int64_t i = i0; i < n_slots; i += st) {
        slot_page[i] = -1;
        slot_epoch[i] = 0;
        slot_ref[i] = 0;
    }
    if (i0 < kCtlWords) ctl[i0] = 0;
}

// Count violations of: page_table[p] = s >= 0  <=>  slot_page[s] = p, and
// every entry either -1 or a slot.
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
    if (threadIdx.x == 0) {
        ctl[9] = static_cast<uint64_t>(n);
        ctl[kCtlNext] = 0;                       // the fetch's page counter
    }
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

namespace skv {

// Resolve one selection on `st`: lookup, claim + victims + placement, then
// fetch + ids (page ids into `ids`).
static int bcache_resolve_launch(skv_bcache *c, const int32_t *sel, int32_t S, int32_t n_sel, int32_t *ids,
                                 cudaStream_t st)
{
    skv_handle *h = c->h;
    if (c->ring_blocks > 0) return fail(h, SKV_EUNSUPPORTED, "a ring cache has a static table and no resolve");
    if (!sel || S <= 0 || n_sel <= 0) return fail(h, SKV_EINVAL, "bad selection");
    const int64_t n_look = static_cast<int64_t>(S) * c->Hk * n_sel;
    if (n_look > c->max_lookups)
        return fail(h, SKV_EINVAL, "%lld lookups exceed max_lookups %lld", (long long)n_look,
                    (long long)c->max_lookups);
    ResolveState r;
    r.page_table = c->page_table;
    r.page_claim = c->page_claim;
    r.page_miss = c->page_miss;
    r.slot_page = c->slot_page;
    r.slot_epoch = c->slot_epoch;
    r.slot_ref = c->slot_ref;
    r.victim = c->victim;
    r.miss_page = c->miss_page;
    r.miss_dest = c->miss_dest;
    r.ctl = c->ctl;
    r.n_slots = c->n_slots;
    r.n_pages = c->n_blocks * c->Hk;
    const unsigned g_look = static_cast<unsigned>(std::min<int64_t>((n_look + 255) / 256, 4 * h->sm_count));
    bcache_lookup_kernel<<<g_look, 256, 0, st>>>(r, sel, n_look, n_sel, c->Hk);
    bcache_victim_kernel<<<1, kVictimThreads, 0, st>>>(r, sel, n_look, n_sel, c->Hk);
    bcache_fetch_kernel<<<h->sm_count, kFetchThreads, 0, st>>>(c->ctl + 12, c->miss_page, c->miss_dest, c->host_k,
                                                               c->host_v, c->pool_k, c->pool_v, c->page_bytes, r, sel,
                                                               n_look, n_sel, c->Hk, ids);
    return cuda_fail(h, cudaGetLastError(), "resolve launch");
}

// The cache's resolve state.
static ResolveState resolve_state_of(const skv_bcache *c)
{
    ResolveState r;
    r.page_table = c->page_table;
    r.page_claim = c->page_claim;
    r.page_miss = c->page_miss;
    r.slot_page = c->slot_page;
    r.slot_epoch = c->slot_epoch;
    r.slot_ref = c->slot_ref;
    r.victim = c->victim;
    r.miss_page = c->miss_page;
    r.miss_dest = c->miss_dest;
    r.ctl = c->ctl;
    r.n_slots = c->n_slots;
    r.n_pages = c->n_blocks * c->Hk;
    return r;
}

// After the fused attention: the misses the claim pass placed in slots are
// moved from their overflow pages (that of each page's first lookup) into
// their slots, and their lookups' page ids become the slots.
__global__ void __launch_bounds__(256) bcache_place_kernel(ResolveState r, const int32_t *__restrict__ sel,
                                                           int64_t n_look, int n_sel, int Hk, uint8_t *pool_k,
                                                           uint8_t *pool_v, int64_t page_bytes,
                                                           int32_t *__restrict__ ids)
{
    const int64_t placed = static_cast<int64_t>(r.ctl[11]);
    const uint32_t epoch = static_cast<uint32_t>(r.ctl[0]);
    const int64_t n16 = page_bytes / 16;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t m = warp; m < placed; m += n_warps) {
        const int32_t p = r.miss_page[m];
        const int64_t first = 0xffffffffll - static_cast<int64_t>(r.page_claim[p] & 0xffffffffull);
        const int64_t src = (r.n_slots + first) * page_bytes, dst = static_cast<int64_t>(r.miss_dest[m]) * page_bytes;
        const uint4 *sk = reinterpret_cast<const uint4 *>(pool_k + src);
        const uint4 *sv = reinterpret_cast<const uint4 *>(pool_v + src);
        uint4 *dk = reinterpret_cast<uint4 *>(pool_k + dst);
        uint4 *dv = reinterpret_cast<uint4 *>(pool_v + dst);
        for (int64_t i = lane; i < n16; i += 32) {
            dk[i] = sk[i];
            dv[i] = sv[i];
        }
    }
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_look;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t p = lookup_page(sel, e, n_sel, Hk, r.n_pages);
        if (p >= 0 && (r.page_claim[p] >> 32) == epoch && r.page_miss[p] < placed) ids[e] = r.miss_dest[r.page_miss[p]];
    }
}

// Resolve and attention as one pass over the host link ("Strata compare", KV
// streaming: resolve, copy, attend): the lookup pass, then the fused
// attention (splitkv_decode_kernel with FUSE), which stages each missed page
// from the host copy while one of its CTAs runs the claim / victim /
// placement pass, then the move of the placed misses into their slots.
// Taken for whole lists of kDecodeTile-row pages and one column group of
// query rows per KV head; *taken says whether it was.  The pool page ids
// recorded for the call are the slots of resident and placed pages and, for
// the rest, the overflow page of each page's first lookup.
static int bcache_attn_fused(skv_bcache *c, const skv_shape *shape, const void *q, const int32_t *sel, int32_t n_sel,
                             float *o, float *lse, cudaStream_t st, bool *taken)
{
    *taken = false;
    skv_handle *h = c->h;
    if (c->ring_blocks > 0 || c->block_rows != kDecodeTile || !c->rstate || !c->page_ready) return SKV_OK;
    if (shape->k_type != SKV_F16 || shape->v_type != SKV_F16 || shape->Hk <= 0 || shape->H % shape->Hk != 0 ||
        shape->nq <= 0 || shape->nq * (shape->H / shape->Hk) > 8 || n_sel <= 0 || !q || !o || !lse)
        return SKV_OK;
    if (!sel || shape->S <= 0) return fail(h, SKV_EINVAL, "bad selection");
    const int64_t n_look = static_cast<int64_t>(shape->S) * c->Hk * n_sel;
    if (n_look > c->max_lookups)
        return fail(h, SKV_EINVAL, "%lld lookups exceed max_lookups %lld", (long long)n_look,
                    (long long)c->max_lookups);
    *taken = true;
    const ResolveState r = resolve_state_of(c);
    const unsigned g_look = static_cast<unsigned>(std::min<int64_t>((n_look + 255) / 256, 4 * h->sm_count));
    bcache_lookup_kernel<<<g_look, 256, 0, st>>>(r, sel, n_look, n_sel, c->Hk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(h, e, "block-cache lookup");
    DecodeArgs f;
    memset(&f, 0, sizeof(f));
    f.rstate = c->rstate;
    f.sel = sel;
    f.n_look = n_look;
    f.page_ids_out = c->page_ids;
    f.host_k = c->host_k;
    f.host_v = c->host_v;
    f.page_ready = c->page_ready;
    f.epoch = c->ctl + kCtlEpochNow;
    f.steal = reinterpret_cast<unsigned long long *>(c->ctl + kCtlSteal);
    int rc = attn_paged_fused(h, shape, q, c->pool_k, c->pool_v, sel, n_sel, o, lse, st, f);
    if (rc) return rc;
    bcache_place_kernel<<<h->sm_count, 256, 0, st>>>(r, sel, n_look, n_sel, c->Hk, c->pool_k, c->pool_v,
                                                     c->page_bytes, c->page_ids);
    return cuda_fail(h, cudaGetLastError(), "block-cache placement");
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
    cudaFree(c->page_claim);
    cudaFree(c->page_miss);
    cudaFree(c->victim);
    cudaFree(c->page_ids);
    cudaFree(c->ctl);
    cudaFree(c->check);
    cudaFree(c->pool_k);
    cudaFree(c->pool_v);
    cudaFree(c->rstate);
    cudaFree(c->page_ready);
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
            c->page_table, c->page_claim, n_pages, c->slot_page, c->slot_epoch, c->slot_ref, c->n_slots, c->ctl,
            c->page_ready, static_cast<int64_t>(c->n_slots) + c->max_lookups);
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
    A(reinterpret_cast<void **>(&c->page_claim), sizeof(uint64_t) * n_pages);
    A(reinterpret_cast<void **>(&c->page_miss), sizeof(int32_t) * n_pages);
    A(reinterpret_cast<void **>(&c->slot_page), sizeof(int32_t) * n_slots);
    A(reinterpret_cast<void **>(&c->slot_epoch), sizeof(int32_t) * n_slots);
    A(reinterpret_cast<void **>(&c->slot_ref), sizeof(int32_t) * n_slots);
    A(reinterpret_cast<void **>(&c->miss_page), sizeof(int32_t) * max_lookups);
    A(reinterpret_cast<void **>(&c->miss_dest), sizeof(int32_t) * max_lookups);
    A(reinterpret_cast<void **>(&c->victim), sizeof(int32_t) * n_slots);
    A(reinterpret_cast<void **>(&c->page_ids), sizeof(int32_t) * max_lookups);
    A(reinterpret_cast<void **>(&c->ctl), sizeof(uint64_t) * kCtlWords);
    A(reinterpret_cast<void **>(&c->check), sizeof(int32_t));
    A(reinterpret_cast<void **>(&c->pool_k), pool_pages * c->page_bytes);
    A(reinterpret_cast<void **>(&c->pool_v), pool_pages * c->page_bytes);
    if (ring_blocks == 0) {
        A(&c->rstate, sizeof(ResolveState));
        A(reinterpret_cast<void **>(&c->page_ready), sizeof(int32_t) * pool_pages);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        skv_bcache_destroy(c);
        return fail(h, SKV_ENOMEM, "block-cache allocation: %s", cudaGetErrorString(e));
    }
    if (c->rstate) {
        const ResolveState r = resolve_state_of(c);
        e = cudaMemcpy(c->rstate, &r, sizeof(r), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            cudaGetLastError();
            skv_bcache_destroy(c);
            return fail(h, SKV_ECUDA, "block-cache state: %s", cudaGetErrorString(e));
        }
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
    c->h->err[0] = 0;
    return bcache_resolve_launch(c, sel, S, n_sel, page_ids ? page_ids : c->page_ids,
                                 static_cast<cudaStream_t>(stream));
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
    c->h->err[0] = 0;
    bool taken = false;
    int rc = skv::bcache_attn_fused(c, shape, q, sel, n_sel, o, lse, static_cast<cudaStream_t>(stream), &taken);
    if (taken || rc) return rc;
    rc = skv_bcache_resolve(c, sel, shape->S, n_sel, c->page_ids, stream);
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
    ResolveState none;
    memset(&none, 0, sizeof(none));
    none.ctl = c->ctl;                           // the fetch's page counter
    bcache_fetch_kernel<<<h->sm_count, kFetchThreads, 0, st>>>(c->ctl + 9, c->miss_page, c->miss_dest, c->host_k,
                                                               c->host_v, c->pool_k, c->pool_v, c->page_bytes, none,
                                                               nullptr, 0, 0, 0, nullptr);
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
