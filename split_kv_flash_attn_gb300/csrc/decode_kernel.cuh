// decode_kernel.cuh -- split-KV decode attention kernel (template; instantiated
// in decode_f16.cu and decode_quant.cu).
//
// One CTA owns one (sequence s, KV head k, column group) unit and one split
// [j_lo, j_hi) of its key list.  The unit's "columns" are up to 8 query rows
// (token t, q head k*G + g) that share the KV head -- GQA grouping as in the
// Rolling KV patch's streaming_lse_kernel head mapping (h / gqa_ratio), so
// every K/V byte is read once for all G heads.
//
// Per 64-key tile (one pipeline stage):
//   * each of the 4 warps owns 16 keys of the tile and stages their K and V
//     head segments itself with cp.async (16 B for fp16 rows, 8/4 B for
//     q8_0/q4_0 segments), STAGES-1 tiles ahead, so a warp waits only for its
//     own copies and the warps never meet at a block barrier inside the loop.
//     Rows come from a dense range, from a row list (padding rows read
//     nothing: zero-filled), or from pages of a block cache.  Row-list
//     entries stream through a small per-warp ring, fetched in the copy group
//     that completes before the tile that needs them is issued, so a split
//     may be any length.
//   * each warp computes on its 16 keys: S^T = K Q^T with mma.sync m16n8k16
//     (keys = M, query columns = N, head dim = K), fp16 in / fp32 accumulate.
//     q8_0 / q4_0 codes are exact in fp16; the per-32-value scale of K is
//     applied to each block's partial dot product in fp32, the scale of V is
//     folded into the probabilities of that block.
//   * online softmax in log2 units (running max m, running sum l per
//     column), then O^T += V^T P^T with the probability fragment transposed by
//     movmatrix into the B operand.
// The 4 warps' (m, l, O) merge through shared memory; the CTA writes its
// normalised partial O and lse = ln2 * (m + log2 l), or O = 0, lse = -inf when
// no key was visible (the empty-row convention of the patch's tail-partial
// conversion kernel).
#pragma once

#include <algorithm>

#include "bcache_resolve.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace skv {

template <int T, int D>
struct Seg {
    static constexpr int bytes = T == SKV_F16 ? 2 * D : (T == SKV_Q8_0 ? 34 * D / 32 : 18 * D / 32);
    // cp.async granule: the largest of 16/8/4 bytes that divides the segment.
    static constexpr int chunk = T == SKV_F16 ? 16 : (bytes % 8 == 0 ? 8 : 4);
    static constexpr bool quant = T != SKV_F16;
};

template <int D, int KT, int VT>
struct DecodeCfg {
    static constexpr int kTile = kDecodeTile;
    static constexpr int kWarps = 4;
    static constexpr int kThreads = 128;
#ifndef SKV_DECODE_STAGES_F16
#define SKV_DECODE_STAGES_F16 2     // 3 CTAs (12 warps) per SM beat a third stage at 2 CTAs
#endif
#ifndef SKV_DECODE_STAGES_QUANT
#define SKV_DECODE_STAGES_QUANT 2   // 3 CTAs per SM: the code conversion needs the warps more than depth
#endif
    static constexpr int STAGES = (KT == SKV_F16 && VT == SKV_F16) ? SKV_DECODE_STAGES_F16 : SKV_DECODE_STAGES_QUANT;
    static constexpr int SEGK = Seg<KT, D>::bytes;
    static constexpr int SEGV = Seg<VT, D>::bytes;
    static constexpr int stage_k = ((kTile * SEGK + 127) / 128) * 128;
    static constexpr int stage_v = ((kTile * SEGV + 127) / 128) * 128;
    static constexpr int stage_bytes = stage_k + stage_v;
    // Row indices: the page table of a paged split (kMaxListSplit entries at
    // most), or in list mode each warp's ring of kIdxRing tiles x 16 entries.
    static constexpr int kIdxRing = 8;
    static_assert(kIdxRing >= 2 * STAGES - 1, "the index ring must hold 2*STAGES-1 tiles");
    static_assert(kWarps * kIdxRing * 16 <= kMaxListSplit, "index rings must fit the index buffer");
    static constexpr int idx_off = STAGES * stage_bytes;
    static constexpr int code_off = idx_off + kMaxListSplit * 4;
    static constexpr int code_k = Seg<KT, D>::quant ? 32 * D : 0;   // 16 keys x D halfs per warp
    static constexpr int code_v = Seg<VT, D>::quant ? 32 * D : 0;
    static constexpr int scale_off = code_off + kWarps * (code_k + code_v);
    static constexpr int scale_k = Seg<KT, D>::quant ? 16 * (D / 32) * 4 : 0;
    static constexpr int scale_v = Seg<VT, D>::quant ? 16 * (D / 32) * 4 : 0;
    static constexpr int smem = scale_off + kWarps * (scale_k + scale_v);
    static constexpr int merge_bytes = kWarps * 8 * (D + 2) * 4;
    static_assert(merge_bytes <= STAGES * stage_bytes, "merge buffer must fit in the stage ring");
    static_assert(8 * 256 * 4 <= STAGES * stage_bytes, "split-merge weights must fit in the stage ring");
};

// Byte offset of 16-byte chunk `ch` of row `r` in a swizzled fp16 tile whose
// rows are D halfs: chunk index XOR (r mod 8) keeps ldmatrix conflict-free.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int ch)
{
    return static_cast<uint32_t>(r * (2 * D) + ((ch ^ (r & 7)) << 4));
}

// Two codes -> one half2, exactly.  The byte c (0..255) placed under the
// exponent byte 0x64 reads as the fp16 value 1024 + c (the spacing of fp16
// numbers in [1024, 2048) is 1), so one byte permute and one half2 subtract
// turn two codes into two fp16 values without a conversion instruction.
__device__ __forceinline__ uint32_t bytes_to_half2(uint32_t two_bytes, uint32_t bias_h2)
{
    const uint32_t h = __byte_perm(two_bytes, 0x64646464u, 0x4140);   // [b0, 0x64, b1, 0x64]
    __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&h), *reinterpret_cast<const __half2 *>(&bias_h2));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t ld_u16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

// Convert 16 keys of q8_0 / q4_0 head segments (raw stage rows) into an fp16
// code tile (swizzled, 16 x D) and per-(key, block) fp32 scales.
//  q8_0: int8 q  -> byte q ^ 0x80 = q + 128, minus 1152 (= 1024 + 128) gives q.
//  q4_0: nibble u -> byte u, minus 1032 (= 1024 + 8) gives u - 8.
template <int T, int D>
__device__ __forceinline__ void convert_codes(const uint8_t *raw, __half *code, float *scale, int lane)
{
    constexpr int SEG = Seg<T, D>::bytes;
    constexpr int NB = D / 32;
    uint8_t *cb = reinterpret_cast<uint8_t *>(code);
    if constexpr (T == SKV_Q8_0) {
        constexpr uint32_t kBias = 0x64806480u;   // half2(1152, 1152)
        constexpr int ITEMS = 16 * NB * 4;        // (key, block, 8-value part)
#pragma unroll 2
        for (int idx = lane; idx < ITEMS; idx += 32) {
            const int kk = idx / (NB * 4);
            const int rem = idx % (NB * 4);
            const int b = rem >> 2;
            const int part = rem & 3;
            const uint8_t *blk = raw + kk * SEG + b * 34;
            const uint8_t *src = blk + 2 + part * 8;
            uint4 out;
            out.x = bytes_to_half2(ld_u16(src) ^ 0x8080u, kBias);
            out.y = bytes_to_half2(ld_u16(src + 2) ^ 0x8080u, kBias);
            out.z = bytes_to_half2(ld_u16(src + 4) ^ 0x8080u, kBias);
            out.w = bytes_to_half2(ld_u16(src + 6) ^ 0x8080u, kBias);
            *reinterpret_cast<uint4 *>(cb + swz<D>(kk, b * 4 + part)) = out;
            if (part == 0) scale[kk * NB + b] = __half2float(*reinterpret_cast<const __half *>(blk));
        }
    } else {
        constexpr uint32_t kBias = 0x64086408u;   // half2(1032, 1032)
        constexpr int ITEMS = 16 * NB * 2;        // (key, block, 8-byte half of the codes)
#pragma unroll 2
        for (int idx = lane; idx < ITEMS; idx += 32) {
            const int kk = idx / (NB * 2);
            const int rem = idx % (NB * 2);
            const int b = rem >> 1;
            const int hb = rem & 1;
            const uint8_t *blk = raw + kk * SEG + b * 18;
            const uint8_t *src = blk + 2 + hb * 8;
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) w[i] = ld_u16(src + 2 * i);
            uint4 lo, hi;
            lo.x = bytes_to_half2(w[0] & 0x0F0Fu, kBias);
            lo.y = bytes_to_half2(w[1] & 0x0F0Fu, kBias);
            lo.z = bytes_to_half2(w[2] & 0x0F0Fu, kBias);
            lo.w = bytes_to_half2(w[3] & 0x0F0Fu, kBias);
            hi.x = bytes_to_half2((w[0] >> 4) & 0x0F0Fu, kBias);
            hi.y = bytes_to_half2((w[1] >> 4) & 0x0F0Fu, kBias);
            hi.z = bytes_to_half2((w[2] >> 4) & 0x0F0Fu, kBias);
            hi.w = bytes_to_half2((w[3] >> 4) & 0x0F0Fu, kBias);
            // byte j holds value j (low nibble) and value j + 16 (high nibble)
            *reinterpret_cast<uint4 *>(cb + swz<D>(kk, b * 4 + hb)) = lo;
            *reinterpret_cast<uint4 *>(cb + swz<D>(kk, b * 4 + 2 + hb)) = hi;
            if (hb == 0) scale[kk * NB + b] = __half2float(*reinterpret_cast<const __half *>(blk));
        }
    }
}

// One split of one unit: the CTA's whole job in an ordinary launch, one work
// item of the fused block-cache instance (FUSE, below the kernel).
template <int D, int KT, int VT, bool FUSE>
__device__ __forceinline__ void decode_split(const DecodeArgs &a, const int cg, const int kh, const int split,
                                             const int s, uint8_t *smem)
{
    using C = DecodeCfg<D, KT, VT>;
    constexpr int kTile = C::kTile;
    constexpr int STAGES = C::STAGES;
    constexpr int SEGK = C::SEGK;
    constexpr int SEGV = C::SEGV;
    constexpr int CHK = Seg<KT, D>::chunk;
    constexpr int CHV = Seg<VT, D>::chunk;
    constexpr bool QK = Seg<KT, D>::quant;
    constexpr bool QV = Seg<VT, D>::quant;
    constexpr int NB = D / 32;   // 32-value blocks per head

    int32_t *idx_s = reinterpret_cast<int32_t *>(smem + C::idx_off);
    static_assert(!FUSE || (KT == SKV_F16 && VT == SKV_F16), "the fused instance reads fp16 pages");
    constexpr int kPubTiles = FUSE ? kMaxListSplit / C::kTile : 1;
    int32_t *src_s = idx_s + kMaxListSplit / 2;      // fused: each page's source (tables of at most 33 pages)
    __shared__ int s_pub[kPubTiles];                 // fused: warps that have written tile t's rows to its pool page

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ---- unit and split -------------------------------------------------
    const int unit = (s * a.Hk + kh) * a.n_cg + cg;
    const int64_t j_lo = a.key_lo + static_cast<int64_t>(split) * a.split_len;
    const int64_t j_hi = min(a.n_local, j_lo + a.split_len);
    const int64_t list = a.rows_per_head ? (static_cast<int64_t>(s) * a.Hk + kh) : s;
    const int lg_pr = a.row_mode == ROWS_PAGED ? (31 - __clz(a.page_rows)) : 0;
    const int64_t page_lo = j_lo >> lg_pr;

    const int wrow = warp * 16;                  // this warp's 16 keys of every tile

    // ---- page table of this split (paged mode) ----------------------------
    // Asynchronous 4-byte copies: every request is in flight at once, so the
    // split starts after one memory round trip, not one per entry.
    if (a.row_mode == ROWS_PAGED) {
        const int32_t *src = a.rows + list * a.rows_ld + page_lo;
        const int n = j_hi > j_lo ? static_cast<int>(((j_hi - 1) >> lg_pr) - page_lo + 1) : 0;
        if constexpr (FUSE) {
            // Each page's pool page and source, from the lookup pass's claims:
            // a page this call missed is staged in the overflow page of its
            // first lookup (n_slots + that lookup), read from the host by the
            // first lookup and from the pool by later ones; any other page is
            // resident at entry, and its table entry stays put for the call.
            const ResolveState &r = *static_cast<const ResolveState *>(a.rstate);
            const uint32_t ep = static_cast<uint32_t>(*a.epoch);
            for (int i = tid; i < n; i += C::kThreads) {
                const int64_t e = list * a.rows_ld + page_lo + i;
                const int64_t blk = a.sel[e];
                const int64_t p = blk * a.Hk + kh;
                int32_t id = -1, from = -1;
                if (blk >= 0 && p < r.n_pages) {
                    const unsigned long long claim = r.page_claim[p];
                    if ((claim >> 32) == ep) {
                        const int64_t first = 0xffffffffll - static_cast<int64_t>(claim & 0xffffffffull);
                        id = static_cast<int32_t>(r.n_slots + first);
                        from = first == e ? static_cast<int32_t>(p) : -2;
                    } else {
                        id = r.page_table[p];
                    }
                }
                idx_s[i] = id;
                src_s[i] = from;
                a.page_ids_out[e] = id;
            }
            for (int i = tid; i < kPubTiles; i += C::kThreads) s_pub[i] = 0;
        } else {
            for (int i = tid; i < n; i += C::kThreads) cp_async4(smem_addr(idx_s + i), src + i, 4);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
    }
    // List mode: entries of tile t for this warp's keys sit in slot t % kIdxRing.
    int32_t *ring = idx_s + warp * C::kIdxRing * 16;
    const int32_t *list_src = a.row_mode == ROWS_LIST ? a.rows + list * a.rows_ld + a.rows_off : nullptr;
    auto load_idx = [&](int t) {
        if (a.row_mode != ROWS_LIST || lane >= 16) return;
        const int64_t j = j_lo + static_cast<int64_t>(t) * kTile + wrow + lane;
        if (j < j_hi) cp_async4(smem_addr(ring + (t & (C::kIdxRing - 1)) * 16 + lane), list_src + j, 4);
    };

    // Cache row (dense / list mode) or pool row (paged mode) of key wrow + rr
    // of tile t, or -1 when the key is absent (past the split, or a padding
    // entry).
    auto key_row = [&](int t, int rr) -> int64_t {
        const int64_t j = j_lo + static_cast<int64_t>(t) * kTile + wrow + rr;
        if (j >= j_hi) return -1;
        if (a.row_mode == ROWS_DENSE) return a.row0 + j;
        if (a.row_mode == ROWS_LIST) return ring[(t & (C::kIdxRing - 1)) * 16 + rr];
        const int32_t pg = idx_s[(j >> lg_pr) - page_lo];
        return pg < 0 ? -1 : (static_cast<int64_t>(pg) << lg_pr) + (j & (a.page_rows - 1));
    };
    // A row holds all Hk heads, except in paged mode where a page holds one.
    const bool paged = a.row_mode == ROWS_PAGED;
    const int64_t head_k = paged ? 0 : static_cast<int64_t>(kh) * SEGK;
    const int64_t head_v = paged ? 0 : static_cast<int64_t>(kh) * SEGV;
    const int64_t stride_k = paged ? SEGK : a.k_row_bytes;
    const int64_t stride_v = paged ? SEGV : a.v_row_bytes;

    // Fused: wait (bounded) until pool page pg carries this call's stamp.
    const int epoch = FUSE ? static_cast<int>(*a.epoch) : 0;
    auto wait_published = [&](int32_t pg) {
        if (lane == 0) {
            uint64_t t0 = 0;
            for (uint32_t it = 0;; ++it) {
                int v;
                asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.page_ready + pg) : "memory");
                if (v == epoch) break;
                if ((it & 63) == 0) {
                    uint64_t t;
                    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
                    if (it == 0) t0 = t;
                    else if (t - t0 > 2000000000ull) {
                        atomicOr(a.status, 1);
                        break;
                    }
                }
                __nanosleep(128);
            }
        }
        __syncwarp();
    };
    // Stage this warp's 16 keys of tile t into stage st.
    auto load_tile = [&](int t, int st) {
        uint8_t *sk_ = smem + st * C::stage_bytes;
        uint8_t *sv_ = sk_ + C::stage_k;
        if constexpr (!QK && !QV) {
            // fp16: each lane owns one 16-byte column chunk of rows rr,
            // rr+RPW, ...; one row lookup serves K and V.
            constexpr int CPR = D / 8;
            constexpr int RPW = 32 / CPR;
            const int ch = lane % CPR;
            const uint32_t dk = smem_addr(sk_), dv = smem_addr(sv_);
            // fused: tile t is page t of the split; a host source moves the
            // rows from pool page pg to host page sr
            const uint8_t *kb = a.k, *vb = a.v;
            int64_t shift = 0;
            if constexpr (FUSE) {
                const int32_t sr = src_s[t], pg = idx_s[t];
                if (pg >= 0 && sr >= 0) {
                    kb = a.host_k;
                    vb = a.host_v;
                    shift = static_cast<int64_t>(sr - pg) << lg_pr;
                } else if (pg >= 0 && sr == -2) {
                    wait_published(pg);
                }
            }
#pragma unroll
            for (int it = 0; it < 16 / RPW; ++it) {
                const int rr = lane / CPR + RPW * it;
                const int r = wrow + rr;
                const uint8_t *src_k, *src_v;
                bool ok;
                if constexpr (FUSE) {
                    const int64_t row = key_row(t, rr) + shift;
                    ok = row >= shift;
                    src_k = kb + (ok ? row * stride_k + head_k + ch * 16 : 0);
                    src_v = vb + (ok ? row * stride_v + head_v + ch * 16 : 0);
                } else {                                 // the same with no shift, written out: cheaper code
                    const int64_t row = key_row(t, rr);
                    ok = row >= 0;
                    src_k = a.k + (ok ? row * stride_k + head_k + ch * 16 : 0);
                    src_v = a.v + (ok ? row * stride_v + head_v + ch * 16 : 0);
                }
                cp_async16(dk + swz<D>(r, ch), src_k, ok ? 16 : 0);
                cp_async16(dv + swz<D>(r, ch), src_v, ok ? 16 : 0);
            }
        } else {
            {
                constexpr int CPR = SEGK / CHK;
                constexpr int TOT = 16 * CPR;
                const uint32_t dk = smem_addr(sk_);
#pragma unroll
                for (int it = 0; it < (TOT + 31) / 32; ++it) {
                    const int c = lane + it * 32;
                    if (TOT % 32 != 0 && c >= TOT) break;
                    const int rr = c / CPR;
                    const int r = wrow + rr;
                    const int ch = c - rr * CPR;
                    const int64_t row = key_row(t, rr);
                    const bool ok = row >= 0;
                    cp_async<CHK>(dk + static_cast<uint32_t>(r * SEGK + ch * CHK),
                                  a.k + (ok ? row * stride_k + head_k + ch * CHK : 0), ok);
                }
            }
            {
                constexpr int CPR = SEGV / CHV;
                constexpr int TOT = 16 * CPR;
                const uint32_t dv = smem_addr(sv_);
#pragma unroll
                for (int it = 0; it < (TOT + 31) / 32; ++it) {
                    const int c = lane + it * 32;
                    if (TOT % 32 != 0 && c >= TOT) break;
                    const int rr = c / CPR;
                    const int r = wrow + rr;
                    const int ch = c - rr * CPR;
                    const int64_t row = key_row(t, rr);
                    const bool ok = row >= 0;
                    cp_async<CHV>(dv + static_cast<uint32_t>(r * SEGV + ch * CHV),
                                  a.v + (ok ? row * stride_v + head_v + ch * CHV : 0), ok);
                }
            }
        }
    };

    // ---- query fragments (B operand: K = head dim, N = 8 columns) -------
    uint32_t qb[D / 16][2];
    {
        const int n = lane >> 2;
        const int c = cg * 8 + n;
        const int t = c / a.G;
        const int g = c % a.G;
        const bool ok = t < a.nq;
        const __half *qp = a.q + ((static_cast<int64_t>(s) * a.nq + (ok ? t : 0)) * a.H + kh * a.G + g) * D;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const int d0 = ks * 16 + 2 * (lane & 3);
            qb[ks][0] = ok ? *reinterpret_cast<const uint32_t *>(qp + d0) : 0u;
            qb[ks][1] = ok ? *reinterpret_cast<const uint32_t *>(qp + d0 + 8) : 0u;
        }
    }
    // This thread's two accumulator columns: c0 = 2*(lane%4), c1 = c0 + 1.
    bool col_ok[2];
    int col_t[2];
    int32_t col_pos[2];
    const __half *col_mask[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int c = cg * 8 + 2 * (lane & 3) + e;
        const int t = c / a.G;
        col_ok[e] = t < a.nq;
        col_t[e] = col_ok[e] ? t : 0;
        col_pos[e] = a.q_pos ? a.q_pos[static_cast<int64_t>(s) * a.nq + col_t[e]] : 0;
        col_mask[e] = a.mask ? a.mask + (static_cast<int64_t>(s) * a.nq + col_t[e]) * a.mask_ld : nullptr;
    }

    float o[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};

    __half *codek = reinterpret_cast<__half *>(smem + C::code_off + warp * C::code_k);
    __half *codev = reinterpret_cast<__half *>(smem + C::code_off + C::kWarps * C::code_k + warp * C::code_v);
    float *scalek = reinterpret_cast<float *>(smem + C::scale_off + warp * C::scale_k);
    float *scalev = reinterpret_cast<float *>(smem + C::scale_off + C::kWarps * C::scale_k + warp * C::scale_v);

    const int n_tiles = static_cast<int>((j_hi - j_lo + kTile - 1) / kTile);
    constexpr float kLog2e = 1.4426950408889634f;

    // ---- pipeline (per warp) ---------------------------------------------
    // Copy groups, in commit order: the list entries of tiles 0..STAGES-2;
    // then for p < STAGES-1 tile p with the entries of tile p+STAGES-1; then
    // at iteration i tile i+STAGES-1 with the entries of tile i+2*STAGES-2.
    // Waiting at iteration i for all but the STAGES-2 newest groups completes
    // tile i and the entries of every tile issued at iteration i, and the ring
    // then holds tiles i .. i+2*STAGES-2 (2*STAGES-1 <= kIdxRing slots).
    for (int p = 0; p < STAGES - 1; ++p) if (p < n_tiles) load_idx(p);
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
#pragma unroll
    for (int p = 0; p < STAGES - 1; ++p) {
        if (p < n_tiles) load_tile(p, p);
        if (p + STAGES - 1 < n_tiles) load_idx(p + STAGES - 1);
        cp_async_commit();
    }
    for (int i = 0; i < n_tiles; ++i) {
        cp_async_wait<STAGES - 2>();
        __syncwarp();
        if constexpr (FUSE) {
            // tile i = page i: a page read from the host is written to its
            // pool page (this warp's 16 rows), then published by the last warp
            const int32_t sr = src_s[i], pg = idx_s[i];
            if (sr >= 0 && pg >= 0) {
                const uint8_t *skp = smem + (i % STAGES) * C::stage_bytes;
                const uint8_t *svp = skp + C::stage_k;
                uint8_t *dk = const_cast<uint8_t *>(a.k) + (static_cast<int64_t>(pg) << lg_pr) * stride_k;
                uint8_t *dv = const_cast<uint8_t *>(a.v) + (static_cast<int64_t>(pg) << lg_pr) * stride_v;
                constexpr int CPR = D / 8;
#pragma unroll 4
                for (int c = lane; c < 16 * CPR; c += 32) {
                    const int r = wrow + c / CPR, ch = c % CPR;
                    *reinterpret_cast<uint4 *>(dk + r * stride_k + ch * 16) =
                        *reinterpret_cast<const uint4 *>(skp + swz<D>(r, ch));
                    *reinterpret_cast<uint4 *>(dv + r * stride_v + ch * 16) =
                        *reinterpret_cast<const uint4 *>(svp + swz<D>(r, ch));
                }
                __threadfence();
                __syncwarp();
                if (lane == 0 && atomicAdd(&s_pub[i], 1) == C::kWarps - 1) {
                    __threadfence();
                    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(a.page_ready + pg), "r"(epoch) : "memory");
                }
            }
        }
        {
            const int nt = i + STAGES - 1;
            if (nt < n_tiles) load_tile(nt, nt % STAGES);
            if (i + 2 * STAGES - 2 < n_tiles) load_idx(i + 2 * STAGES - 2);
            cp_async_commit();
        }
        const int st = i % STAGES;
        const uint8_t *sk_ = smem + st * C::stage_bytes;
        const uint8_t *sv_ = sk_ + C::stage_k;
        const int64_t jw = j_lo + static_cast<int64_t>(i) * kTile + wrow;   // first key of this warp
        const int r0 = lane >> 2;
        const bool v0 = key_row(i, r0) >= 0;
        const bool v1 = key_row(i, r0 + 8) >= 0;
        if (!__any_sync(0xffffffffu, v0 || v1)) continue;   // all 16 keys absent: nothing to do

        // S^T = K Q^T  (16 keys x 8 columns)
        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (!QK) {
            const uint32_t base = smem_addr(sk_);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int key = wrow + ((lane >> 3) & 1) * 8 + (lane & 7);
                const int ch = 2 * ks + (lane >> 4);
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4(base + swz<D>(key, ch), a0, a1, a2, a3);
                mma_16816(sacc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
            }
        } else {
            __syncwarp();
            convert_codes<KT, D>(sk_ + wrow * SEGK, codek, scalek, lane);
            __syncwarp();
            const uint32_t base = smem_addr(codek);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int ks = 2 * b + kk;
                    const int key = ((lane >> 3) & 1) * 8 + (lane & 7);
                    const int ch = 2 * ks + (lane >> 4);
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(base + swz<D>(key, ch), a0, a1, a2, a3);
                    mma_16816(t, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                }
                const float d0 = scalek[r0 * NB + b];
                const float d1 = scalek[(r0 + 8) * NB + b];
                sacc[0] = fmaf(d0, t[0], sacc[0]);
                sacc[1] = fmaf(d0, t[1], sacc[1]);
                sacc[2] = fmaf(d1, t[2], sacc[2]);
                sacc[3] = fmaf(d1, t[3], sacc[3]);
            }
        }

        // scores in log2 units with masking
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int rr = r0 + ((e >> 1) << 3);
            const int ce = e & 1;
            const bool kv_ok = (e >> 1) ? v1 : v0;
            float val = sacc[e] * a.scale_log2;
            const int64_t jl = jw + rr;                      // local key index
            const int64_t logical = a.logical0 + jl;
            if (!kv_ok) val = -INFINITY;
            if (a.q_pos && a.key_pos0 + logical > col_pos[ce]) val = -INFINITY;
            if (col_mask[ce] && kv_ok) val += __half2float(col_mask[ce][logical]) * kLog2e;
            x[e] = val;
        }
        // online softmax per column
        float mx0 = fmaxf(x[0], x[2]);
        float mx1 = fmaxf(x[1], x[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m_run[0], mx0);
        const float mn1 = fmaxf(m_run[1], mx1);
        const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
        const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = fast_exp2(m_run[0] - ref0);
        const float al1 = fast_exp2(m_run[1] - ref1);
        float p[4];
        p[0] = fast_exp2(x[0] - ref0);
        p[1] = fast_exp2(x[1] - ref1);
        p[2] = fast_exp2(x[2] - ref0);
        p[3] = fast_exp2(x[3] - ref1);
        l_run[0] = l_run[0] * al0 + p[0] + p[2];
        l_run[1] = l_run[1] * al1 + p[1] + p[3];
        m_run[0] = mn0;
        m_run[1] = mn1;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
        }

        // O^T += V^T P^T
        if constexpr (!QV) {
            const uint32_t pb0 = movmatrix_trans(pack_half2(p[0], p[1]));
            const uint32_t pb1 = movmatrix_trans(pack_half2(p[2], p[3]));
            const uint32_t base = smem_addr(sv_);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int key = wrow + (lane >> 4) * 8 + (lane & 7);
                const int ch = 2 * mt + ((lane >> 3) & 1);
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4_trans(base + swz<D>(key, ch), a0, a1, a2, a3);
                mma_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
            }
        } else {
            __syncwarp();
            convert_codes<VT, D>(sv_ + wrow * SEGV, codev, scalev, lane);
            __syncwarp();
            const uint32_t base = smem_addr(codev);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float d0 = scalev[r0 * NB + b];
                const float d1 = scalev[(r0 + 8) * NB + b];
                const uint32_t pb0 = movmatrix_trans(pack_half2(p[0] * d0, p[1] * d0));
                const uint32_t pb1 = movmatrix_trans(pack_half2(p[2] * d1, p[3] * d1));
#pragma unroll
                for (int mm = 0; mm < 2; ++mm) {
                    const int mt = 2 * b + mm;
                    const int key = (lane >> 4) * 8 + (lane & 7);
                    const int ch = 2 * mt + ((lane >> 3) & 1);
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4_trans(base + swz<D>(key, ch), a0, a1, a2, a3);
                    mma_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
                }
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- merge the 4 warps -------------------------------------------------
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
    }
    float *mg_o = reinterpret_cast<float *>(smem);             // [warp][8][D]
    float *mg_m = mg_o + C::kWarps * 8 * D;                     // [warp][8]
    float *mg_l = mg_m + C::kWarps * 8;                         // [warp][8]
    {
        const int c0 = 2 * (lane & 3);
        if (lane < 4) {
            mg_m[warp * 8 + c0] = m_run[0];
            mg_m[warp * 8 + c0 + 1] = m_run[1];
            mg_l[warp * 8 + c0] = l_run[0];
            mg_l[warp * 8 + c0 + 1] = l_run[1];
        }
        const int d = lane >> 2;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            float *w = mg_o + warp * 8 * D;
            w[c0 * D + mt * 16 + d] = o[mt][0];
            w[(c0 + 1) * D + mt * 16 + d] = o[mt][1];
            w[c0 * D + mt * 16 + d + 8] = o[mt][2];
            w[(c0 + 1) * D + mt * 16 + d + 8] = o[mt][3];
        }
    }
    __syncthreads();
    // This CTA's result per column: written straight to the output when the
    // launch has one split, else to the split scratch for the merge below.
    const int col = tid >> 4;
    const int sub = tid & 15;
    const int ccol = cg * 8 + col;
    const int t_c = ccol / a.G;
    const int64_t r_c = (static_cast<int64_t>(s) * a.nq + (t_c < a.nq ? t_c : 0)) * a.H + kh * a.G + ccol % a.G;
    const bool col_valid = t_c < a.nq;
    const bool direct = a.n_splits == 1;
    if (col_valid) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, mg_m[w * 8 + col]);
        float *op = direct ? a.o_out + r_c * D : a.o_split + (static_cast<int64_t>(split) * a.R + r_c) * D;
        float *lp = direct ? a.lse_out + r_c : a.lse_split + static_cast<int64_t>(split) * a.R + r_c;
        if (M == -INFINITY) {
            for (int d = sub; d < D; d += 16) op[d] = 0.f;
            if (sub == 0) *lp = -INFINITY;
        } else {
            float sc[C::kWarps];
            float L = 0.f;
#pragma unroll
            for (int w = 0; w < C::kWarps; ++w) {
                const float mw = mg_m[w * 8 + col];
                sc[w] = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
                L += sc[w] * mg_l[w * 8 + col];
            }
            const float inv = 1.f / L;
            for (int d = sub; d < D; d += 16) {
                float acc = 0.f;
#pragma unroll
                for (int w = 0; w < C::kWarps; ++w) acc += sc[w] * mg_o[(w * 8 + col) * D + d];
                op[d] = acc * inv;
            }
            if (sub == 0) *lp = (M + __log2f(L)) * 0.6931471805599453f;
        }
    }
    if (direct) return;

    // ---- last CTA of the unit merges all splits (log-sum-exp combine) ------
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(a.counters + unit, 1);
        s_last = prev == a.n_splits - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    constexpr int CH = 256;                          // splits per weight chunk
    float *wsm = reinterpret_cast<float *>(smem) + col * CH;
    float M = -INFINITY;
    if (col_valid)
        for (int sp = sub; sp < a.n_splits; sp += 16)
            M = fmaxf(M, __ldcg(a.lse_split + static_cast<int64_t>(sp) * a.R + r_c));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float acc[D / 16];
#pragma unroll
    for (int e = 0; e < D / 16; ++e) acc[e] = 0.f;
    float W = 0.f;
    const unsigned gmask = 0xFFFFu << (lane & 16);   // the 16 lanes of this column
    if (col_valid && M != -INFINITY) {
        for (int base = 0; base < a.n_splits; base += CH) {
            const int n = min(CH, a.n_splits - base);
            __syncwarp(gmask);
            for (int i = sub; i < n; i += 16) {
                const float l = __ldcg(a.lse_split + static_cast<int64_t>(base + i) * a.R + r_c);
                const float w = l == -INFINITY ? 0.f : fast_exp2((l - M) * 1.4426950408889634f);
                wsm[i] = w;
                W += w;
            }
            __syncwarp(gmask);
            // Every split wrote finite values (0 for an empty split), so a zero
            // weight needs no branch; 4 splits' loads are issued together.
            const float *op0 = a.o_split + (static_cast<int64_t>(base) * a.R + r_c) * D + sub;
            const int64_t pstride = a.R * D;
            int i = 0;
            for (; i + 4 <= n; i += 4) {
                float x[4][D / 16];
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int e = 0; e < D / 16; ++e) x[u][e] = __ldcg(op0 + (i + u) * pstride + 16 * e);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float w = wsm[i + u];
#pragma unroll
                    for (int e = 0; e < D / 16; ++e) acc[e] = fmaf(w, x[u][e], acc[e]);
                }
            }
            for (; i < n; ++i) {
                const float w = wsm[i];
#pragma unroll
                for (int e = 0; e < D / 16; ++e) acc[e] = fmaf(w, __ldcg(op0 + i * pstride + 16 * e), acc[e]);
            }
        }
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
    if (col_valid) {
        float *op = a.o_out + r_c * D;
        if (M == -INFINITY) {
#pragma unroll
            for (int e = 0; e < D / 16; ++e) op[sub + 16 * e] = 0.f;
            if (sub == 0) a.lse_out[r_c] = -INFINITY;
        } else {
            const float inv = 1.f / W;
#pragma unroll
            for (int e = 0; e < D / 16; ++e) op[sub + 16 * e] = acc[e] * inv;
            if (sub == 0) a.lse_out[r_c] = M + __logf(W);
        }
    }
    if (tid == 0) a.counters[unit] = 0;              // ready for the next launch
}

// An ordinary launch: one CTA per (unit, split) -- grid x = (KV head, column
// group) fastest, y = split, z = sequence, so CTAs that run side by side read
// the other heads' segments of the same cache rows.
//
// FUSE: the block-cache attention that also fetches (fp16 pages of kTile
// rows, whole lists, one column group), launched right after the lookup pass.
// CTA 0 first runs the claim / victim / placement pass (NT = 128), which only
// decides where the missed pages will live; the pages themselves are staged
// meanwhile.  A persistent grid takes (unit, split) work items from a counter
// in lookup order (sequence, KV head, split).  A page this call missed is read
// from the host copy by its first lookup and, once the CTA's four warps have
// it in shared memory, written to the overflow page of that lookup and
// published (its stamp set to this call's epoch); a later lookup of the page
// reads it there once published -- its publisher's item was taken earlier and
// waits only for items taken before it, so every wait ends (and each is
// bounded).  Resident pages are read from their slots.  Pages and arithmetic
// are those of an ordinary launch with the same splits over the pool.
template <int D, int KT, int VT, bool FUSE = false>
__global__ void __launch_bounds__(128) splitkv_decode_kernel(const DecodeArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    if constexpr (!FUSE) {
        decode_split<D, KT, VT, false>(a, blockIdx.x % a.n_cg, blockIdx.x / a.n_cg, blockIdx.y, blockIdx.z, smem);
    } else {
        __shared__ unsigned long long s_item;
        const unsigned long long items =
            static_cast<unsigned long long>(a.S) * a.Hk * a.n_cg * static_cast<unsigned long long>(a.n_splits);
        if (blockIdx.x == 0) {
            victim_pass<DecodeCfg<D, KT, VT>::kThreads>(*static_cast<const ResolveState *>(a.rstate), a.sel, a.n_look,
                                     static_cast<int>(a.rows_ld), a.Hk);
            __syncthreads();
        }
        for (;;) {
            if (threadIdx.x == 0) s_item = atomicAdd(a.steal, 1ull);
            __syncthreads();
            const unsigned long long w = s_item;
            __syncthreads();                         // s_item is read before it is taken again
            if (w >= items) break;
            const int split = static_cast<int>(w % a.n_splits);
            const unsigned long long u = w / a.n_splits;   // (s * Hk + kh) * n_cg + cg
            decode_split<D, KT, VT, true>(a, static_cast<int>(u % a.n_cg), static_cast<int>((u / a.n_cg) % a.Hk),
                                          split, static_cast<int>(u / (static_cast<unsigned long long>(a.n_cg) * a.Hk)),
                                          smem);
            __syncthreads();                         // shared memory is reused by the next item
        }
    }
}

namespace {
// One cache per instance and translation unit (internal linkage: a static in
// an external template would be merged across every copy of the library a
// process loads).
template <int D, int KT, int VT, bool FUSE = false>
KernelAttrCache &decode_attr_cache()
{
    static KernelAttrCache c;
    return c;
}
}  // namespace

template <int D, int KT, int VT>
int launch_decode_t(skv_handle *h, const DecodeArgs &a, cudaStream_t st)
{
    using C = DecodeCfg<D, KT, VT>;
    cudaError_t e = kernel_smem_optin(decode_attr_cache<D, KT, VT>(),
                                      reinterpret_cast<const void *>(splitkv_decode_kernel<D, KT, VT>), C::smem,
                                      C::kThreads, nullptr);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute(decode)");
    if (a.Hk * a.n_cg > 65535 || a.n_splits > 65535 || a.S > 65535)
        return fail(h, SKV_EUNSUPPORTED, "grid too large: Hk*n_cg=%d splits=%d S=%d", a.Hk * a.n_cg, a.n_splits, a.S);
    if (a.n_splits > kMaxSplits) return fail(h, SKV_EUNSUPPORTED, "%d splits exceed %d", a.n_splits, kMaxSplits);
    dim3 grid(static_cast<unsigned>(a.Hk * a.n_cg), static_cast<unsigned>(a.n_splits), static_cast<unsigned>(a.S));
    splitkv_decode_kernel<D, KT, VT><<<grid, C::kThreads, C::smem, st>>>(a);
    return cuda_fail(h, cudaGetLastError(), "decode kernel launch");
}

// The fused block-cache instance: a persistent grid of at most the CTAs
// resident at once, launched cooperatively since its CTAs wait for pages
// others publish.
template <int D>
int launch_decode_fused_t(skv_handle *h, const DecodeArgs &a, cudaStream_t st)
{
    using C = DecodeCfg<D, SKV_F16, SKV_F16>;
    const void *fn = reinterpret_cast<const void *>(splitkv_decode_kernel<D, SKV_F16, SKV_F16, true>);
    int per_sm = 0;
    cudaError_t e = kernel_smem_optin(decode_attr_cache<D, SKV_F16, SKV_F16, true>(), fn, C::smem, C::kThreads, &per_sm);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute(fused decode)");
    if (per_sm <= 0) return fail(h, SKV_EUNSUPPORTED, "the fused decode kernel cannot be resident");
    const int64_t items = static_cast<int64_t>(a.S) * a.Hk * a.n_cg * a.n_splits;
    const int64_t ctas = std::min<int64_t>(items, static_cast<int64_t>(per_sm) * h->sm_count);
    if (ctas <= 0) return SKV_OK;
    DecodeArgs arg = a;
    void *args[] = {&arg};
    e = cudaLaunchCooperativeKernel(fn, dim3(static_cast<unsigned>(ctas)), dim3(C::kThreads), args,
                                    static_cast<size_t>(C::smem), st);
    return cuda_fail(h, e, "fused decode launch");
}

template <int D, int KT, int VT>
int decode_ctas_per_sm_t(skv_handle *h)
{
    using C = DecodeCfg<D, KT, VT>;
    int n = 0;
    if (kernel_smem_optin(decode_attr_cache<D, KT, VT>(), reinterpret_cast<const void *>(splitkv_decode_kernel<D, KT, VT>),
                          C::smem, C::kThreads, &n) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    (void)h;
    return n;
}

}  // namespace skv
