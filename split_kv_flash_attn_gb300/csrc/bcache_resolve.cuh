// bcache_resolve.cuh -- the block cache's resolve state and its claim /
// victim / placement pass, shared by the resolve launches (bcache.cu) and the
// fused block-cache attention (decode_kernel.cuh), which runs the pass in one
// of its CTAs.
#pragma once

#include <cub/block/block_scan.cuh>

#include "internal.h"

namespace skv {

// ctl words (uint64): 0 epoch of the last resolve, 1 hand, 2 calls, 3 lookups,
// 4 hits, 5 misses, 6 overflow, 7 last misses, 8 last overflow, 9 pages a ring
// restore fetches, 11 misses placed in slots by the last resolve, 12 misses of
// the last resolve, 13 pages the running fetch has handed out, 14 and 15 below.
constexpr int kCtlWords = 16;
constexpr int kCtlNext = 13;
constexpr int kCtlEpochNow = 14;   // epoch of the call in progress (written by the lookup pass)
constexpr int kCtlSteal = 15;      // work items the fused attention has handed out (zeroed by the lookup pass)
constexpr int kVictimThreads = 512;

struct ResolveState {
    int32_t *page_table;
    uint64_t *page_claim;
    int32_t *page_miss;
    int32_t *slot_page, *slot_epoch, *slot_ref, *victim;
    int32_t *miss_page, *miss_dest;
    uint64_t *ctl;
    int n_slots;
    int64_t n_pages;
};

__device__ __forceinline__ int64_t lookup_page(const int32_t *sel, int64_t e, int n_sel, int Hk, int64_t n_pages)
{
    const int64_t b = sel[e];
    const int64_t p = b * Hk + (e / n_sel) % Hk;
    return (b < 0 || p >= n_pages) ? -1 : p;     // out-of-range ids are rejected here; never indexed
}

// Claim key of lookup e in call `epoch`: a later call, then an earlier lookup,
// compares larger.
__device__ __forceinline__ unsigned long long claim_key(int epoch, int64_t e)
{
    return (static_cast<unsigned long long>(static_cast<uint32_t>(epoch)) << 32) |
           static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(e));
}

// Claim, victim and placement pass, one CTA of NT threads.
//  1. Miss list: lookup e owns page p when p's claim word holds e's key (the
//     first lookup of this call naming a missing p); owners are numbered in
//     lookup order by a block scan, tile by tile.
//  2. Victims: thread t owns hand-relative positions [t*per, (t+1)*per);
//     position i is slot (hand + i) % n_slots.
//  3. Placement (below).
constexpr int kClaimItems = 16;   // lookups per thread and tile of step 1
constexpr int kSlotItems = 16;    // slots per thread whose classes stay in registers in step 2
constexpr int kPlaceBatch = 16;   // misses per thread and round of step 3
template <int NT>
__device__ __forceinline__ void victim_pass(const ResolveState &r, const int32_t *__restrict__ sel, int64_t n_look,
                                            int n_sel, int Hk)
{
    using Scan = cub::BlockScan<unsigned long long, NT>;
    __shared__ typename Scan::TempStorage scan_tmp;
    __shared__ int s_stop;
    const int epoch = static_cast<int>(r.ctl[0]) + 1;
    if (threadIdx.x == 0) r.ctl[kCtlNext] = 0;      // the fetch's page counter
    // 1. the miss list in lookup order
    int64_t need = 0;
    for (int64_t t0 = 0; t0 < n_look; t0 += static_cast<int64_t>(NT) * kClaimItems) {
        const int64_t e0 = t0 + static_cast<int64_t>(threadIdx.x) * kClaimItems;
        // lookups are [S][Hk][n_sel]: the KV head of e0, stepped item by item
        const int64_t row = e0 / n_sel;
        int col = static_cast<int>(e0 - row * n_sel);
        int kh = static_cast<int>(row % Hk);
        int32_t pg[kClaimItems];
#pragma unroll
        for (int u = 0; u < kClaimItems; ++u) {
            const int64_t e = e0 + u;
            int32_t p = -1;
            if (e < n_look) {
                const int64_t blk = sel[e];
                const int64_t pp = blk * Hk + kh;
                if (blk >= 0 && pp < r.n_pages) p = static_cast<int32_t>(pp);   // out-of-range ids: no page
            }
            pg[u] = p;
            if (++col == n_sel) {
                col = 0;
                if (++kh == Hk) kh = 0;
            }
        }
        unsigned own = 0;                            // bit u: lookup e0 + u owns its page
#pragma unroll
        for (int u = 0; u < kClaimItems; ++u)
            if (pg[u] >= 0 && r.page_claim[pg[u]] == claim_key(epoch, e0 + u)) own |= 1u << u;
        unsigned long long before = 0, total = 0;
        Scan(scan_tmp).ExclusiveSum(static_cast<unsigned long long>(__popc(own)), before, total);
        int64_t m = need + static_cast<int64_t>(before);
#pragma unroll
        for (int u = 0; u < kClaimItems; ++u) {
            if (own & (1u << u)) {
                r.miss_page[m] = pg[u];
                r.page_miss[pg[u]] = static_cast<int32_t>(m);
                ++m;
            }
        }
        need += static_cast<int64_t>(total);
        __syncthreads();                             // scan_tmp is reused
    }
    // 2. victims
    const int n = r.n_slots;
    const int hand = static_cast<int>(r.ctl[1] % static_cast<uint64_t>(n));
    const int per = (n + NT - 1) / NT;
    const int i0 = min(n, static_cast<int>(threadIdx.x) * per), i1 = min(n, i0 + per);
    const int cnt = i1 - i0;
    // slot of hand-relative position i0 + k (k < per <= n)
    auto slot_k = [&](int k) {
        int j = hand + i0 + k;
        j -= j >= n ? n : 0;
        j -= j >= n ? n : 0;
        return j;
    };
    // 0: in use by this call, 1: cold (free or unreferenced), 2: warm (referenced)
    auto class_of = [&](int32_t ep, int32_t pgid, int32_t ref) { return ep == epoch ? 0 : (pgid < 0 || ref == 0) ? 1 : 2; };
    uint32_t cls = 0;                                // classes of positions k < kSlotItems, 2 bits each
    {
        int32_t ep[kSlotItems], sp[kSlotItems], rf[kSlotItems];
#pragma unroll
        for (int k = 0; k < kSlotItems; ++k) {       // every load in flight at once
            const int j = slot_k(k);
            const bool in = k < cnt;
            ep[k] = in ? r.slot_epoch[j] : 0;
            sp[k] = in ? r.slot_page[j] : 0;
            rf[k] = in ? r.slot_ref[j] : 0;
        }
#pragma unroll
        for (int k = 0; k < kSlotItems; ++k) cls |= static_cast<uint32_t>(class_of(ep[k], sp[k], rf[k])) << (2 * k);
    }
    auto class_at = [&](int k) {
        if (k < kSlotItems) return static_cast<int>((cls >> (2 * k)) & 3u);
        const int j = slot_k(k);
        return class_of(r.slot_epoch[j], r.slot_page[j], r.slot_ref[j]);
    };
    unsigned long long mine = 0;                 // cold count | warm count << 32
    for (int k = 0; k < cnt; ++k) {
        const int c = class_at(k);
        mine += c == 1 ? 1ull : (c == 2 ? (1ull << 32) : 0ull);
    }
    unsigned long long before = 0, total = 0;
    Scan(scan_tmp).ExclusiveSum(mine, before, total);
    const int64_t n_cold = static_cast<int64_t>(total & 0xffffffffull), n_warm = static_cast<int64_t>(total >> 32);
    const int64_t placed = min(need, n_cold + n_warm);
    // The sweep wraps once the cold slots run out: the hand has then passed --
    // and cleared -- every warm slot, and takes warm slots on its second round.
    const bool wraps = need > n_cold;
    const int64_t warm_taken = wraps ? placed - n_cold : 0;
    if (threadIdx.x == 0) s_stop = -1;
    __syncthreads();
    int64_t rc = static_cast<int64_t>(before & 0xffffffffull), rw = static_cast<int64_t>(before >> 32);
    for (int k = 0; k < cnt; ++k) {
        const int c = class_at(k);
        const int j = slot_k(k);
        if (c == 1) {
            if (rc < need) {
                r.victim[rc] = j;
                if (rc == (wraps ? (warm_taken == 0 ? n_cold - 1 : -1) : need - 1)) s_stop = i0 + k;
            }
            ++rc;
        } else if (c == 2) {
            if (wraps) {
                r.slot_ref[j] = 0;
                if (rw < warm_taken) {
                    r.victim[n_cold + rw] = j;
                    if (rw == warm_taken - 1) s_stop = i0 + k;
                }
            }
            ++rw;
        }
    }
    __syncthreads();
    const int stop = s_stop;
    if (!wraps && stop >= 0) {
        // one partial round: the warm slots before the stop lose their reference bit
        for (int k = 0; k < min(cnt, stop - i0); ++k)
            if (class_at(k) == 2) r.slot_ref[slot_k(k)] = 0;
    }
    __syncthreads();                                 // victim[] complete
    // 3. placement: miss m < placed takes victim[m]; the rest go to the
    //    overflow area (pool page n_slots + m - placed), for this call only.
    //    Each thread places kPlaceBatch misses at a time, all their loads
    //    issued before any store.
    for (int64_t m0 = threadIdx.x; m0 < need; m0 += static_cast<int64_t>(NT) * kPlaceBatch) {
        int pg[kPlaceBatch], vj[kPlaceBatch], old[kPlaceBatch];
#pragma unroll
        for (int u = 0; u < kPlaceBatch; ++u) {
            const int64_t m = m0 + static_cast<int64_t>(u) * NT;
            pg[u] = m < need ? r.miss_page[m] : -1;
            vj[u] = m < placed ? r.victim[m] : -1;
        }
#pragma unroll
        for (int u = 0; u < kPlaceBatch; ++u) old[u] = vj[u] >= 0 ? r.slot_page[vj[u]] : -1;
#pragma unroll
        for (int u = 0; u < kPlaceBatch; ++u) {
            const int64_t m = m0 + static_cast<int64_t>(u) * NT;
            if (m >= need) continue;
            if (vj[u] >= 0) {
                const int j = vj[u];
                if (old[u] >= 0) r.page_table[old[u]] = -1;   // a resident page no lookup of this call named
                r.slot_page[j] = pg[u];
                r.slot_ref[j] = 1;
                r.slot_epoch[j] = epoch;
                r.page_table[pg[u]] = j;
                r.miss_dest[m] = j;
            } else {
                r.miss_dest[m] = static_cast<int32_t>(n + (m - placed));
            }
        }
    }
    if (threadIdx.x == 0) {
        if (stop >= 0) r.ctl[1] = static_cast<uint64_t>((static_cast<int64_t>(hand) + stop + 1) % n);
        r.ctl[0] = static_cast<uint64_t>(epoch);
        r.ctl[2] += 1;
        r.ctl[5] += static_cast<uint64_t>(need);
        r.ctl[6] += static_cast<uint64_t>(need - placed);
        r.ctl[7] = static_cast<uint64_t>(need);
        r.ctl[8] = static_cast<uint64_t>(need - placed);
        r.ctl[11] = static_cast<uint64_t>(placed);
        r.ctl[12] = static_cast<uint64_t>(need);
    }
}

}  // namespace skv
