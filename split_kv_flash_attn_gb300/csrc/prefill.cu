// prefill.cu -- prefill-chunk attention on the 5th-generation tensor cores.
//
// The only place in the path where the work is a dense contraction: nq new
// tokens x G heads of one KV head against a range of keys.  One CTA owns a
// 128-row query tile (128/G tokens x G heads of KV head k, the GQA packing) and
// one split of the key range, and walks it in 128-key tiles:
//
//   TMA (warp 4)  : K_j, V_j tiles (128 keys x 128 d, fp16, 128-byte swizzle)
//                   into a 2-deep K ring and a 2-deep V ring.
//   MMA (warp 5)  : S_j = Q K_j^T        tcgen05.mma kind::f16, M=N=128, into
//                                        one of two TMEM S buffers (fp32);
//                   O  += P_j V_j        into the TMEM O accumulator; V is the
//                                        B operand in MN-major layout.
//   softmax (0-3) : thread = query row = TMEM lane: tcgen05.ld S_j, causal
//                   mask, online softmax in log2 units, P_j (fp16) to shared
//                   memory.  O is rescaled in TMEM only when a row maximum
//                   grows by more than 2^8 (the stale maximum stays the
//                   reference otherwise, exactly as in the plain online
//                   softmax with a different shift).
//
// The per-split result (O normalised, lse) is merged across splits by the
// last CTA of each (sequence, KV head, query tile), as in the decode kernel.
// Every mbarrier wait is bounded; a wait that gives up sets the handle's
// device status word and the CTA stops issuing work, drains what it issued
// and frees its TMEM.
#include <string.h>

#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace skv {

namespace {

constexpr int kPM = 128;        // query rows per tile (TMEM lanes)
constexpr int kPN = 128;        // keys per tile
constexpr int kPD = 128;        // head dim
constexpr int kSoftmaxWarps = 8;   // two warps per query-row group (one per column half)
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kPThreads = kSoftmaxThreads + 64;  // + TMA warp + MMA warp
constexpr int kTileBytes = kPN * kPD * 2;       // 32 KiB per K or V tile
constexpr int kHalfTile = kTileBytes / 2;       // one 64-column swizzle block
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;       // 2 stages
constexpr int kOffV = kOffK + 2 * kTileBytes;   // 2 stages
constexpr int kOffP = kOffV + 2 * kTileBytes;
constexpr int kOffBar = kOffP + kTileBytes;
constexpr int kSmem = kOffBar + 256 + 1024;     // + barriers + alignment slack
constexpr uint32_t kIdescS = tc::idesc_f16(kPM, kPN, false);
constexpr uint32_t kIdescPV = tc::idesc_f16(kPM, kPD, true);
constexpr float kRescaleLog2 = 8.0f;            // rescale O only when the max grows by > 2^8

// barrier slots (8 bytes each) inside the barrier area
enum { B_KFULL = 0, B_KEMPTY = 2, B_VFULL = 4, B_VEMPTY = 6, B_QFULL = 8, B_SFULL = 9, B_SFREE = 11, B_PFULL = 13,
       B_PVDONE = 14, B_COUNT = 15 };

}  // namespace

struct PrefillArgs {
    const __half *q;          // [S][nq][H][D]
    int S, nq, H, Hk, G;
    float scale_log2;
    const int32_t *q_pos;     // [S][nq] or null
    int64_t key_pos0;
    int64_t logical0;
    int64_t row0;             // tensor-map row of local key 0
    int64_t n_local;
    int m_tiles;
    int n_splits;
    int64_t split_len;
    float *o_split;
    float *lse_split;
    int *counters;
    float *o_out;
    float *lse_out;
    int64_t R;
    int *status;
};

__global__ void __launch_bounds__(kPThreads, 1)
    splitkv_prefill_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                           const PrefillArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(sm);
    const uint32_t bar0 = sbase + kOffBar;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ int s_maxpos;
    __shared__ int s_last;
    // [slot][column half][row]: partial row maxima by tile parity (slots 0, 1),
    // then the halves' row sums (slot 2, so that no partner read is pending)
    __shared__ float s_pair[3][2][kPM];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int mt = blockIdx.x % a.m_tiles;
    const int kh = blockIdx.x / a.m_tiles;
    const int split = blockIdx.y;
    const int s = blockIdx.z;
    const int unit = (s * a.Hk + kh) * a.m_tiles + mt;
    const int tpt = kPM / a.G;                       // tokens per query tile

    const int64_t j_lo = static_cast<int64_t>(split) * a.split_len;
    const int64_t j_hi = min(a.n_local, j_lo + a.split_len);

    // Softmax threads: query row m = TMEM lane (warp % 4) * 32 + lane, and the
    // column half hf (key columns hf*64 .. hf*64+63 of each 128-key tile).
    const bool softmax = warp < kSoftmaxWarps;
    const int m = (warp & 3) * 32 + lane;
    const int hf = warp >> 2;
    const int t_row = mt * tpt + m / a.G;
    const bool row_ok = softmax && t_row < a.nq;
    const int32_t pos_row = (row_ok && a.q_pos) ? a.q_pos[static_cast<int64_t>(s) * a.nq + t_row] : INT32_MAX;

    if (tid == 0) {
        s_abort = 0;
        s_maxpos = INT32_MIN;
    }
    __syncthreads();
    if (a.q_pos && row_ok && hf == 0) atomicMax(&s_maxpos, pos_row);
    if (warp == 0) {
        tc::tmem_alloc<512>(smem_addr(&s_tmem));
        tc::tmem_relinquish();
    }
    if (tid == kSoftmaxThreads) {
        tc::mbar_init(bar(B_KFULL), 1);
        tc::mbar_init(bar(B_KFULL + 1), 1);
        tc::mbar_init(bar(B_KEMPTY), 1);
        tc::mbar_init(bar(B_KEMPTY + 1), 1);
        tc::mbar_init(bar(B_VFULL), 1);
        tc::mbar_init(bar(B_VFULL + 1), 1);
        tc::mbar_init(bar(B_VEMPTY), 1);
        tc::mbar_init(bar(B_VEMPTY + 1), 1);
        tc::mbar_init(bar(B_QFULL), kSoftmaxThreads);
        tc::mbar_init(bar(B_SFULL), 1);
        tc::mbar_init(bar(B_SFULL + 1), 1);
        tc::mbar_init(bar(B_SFREE), kSoftmaxThreads);
        tc::mbar_init(bar(B_SFREE + 1), kSoftmaxThreads);
        tc::mbar_init(bar(B_PFULL), kSoftmaxThreads);
        tc::mbar_init(bar(B_PVDONE), 1);
        tc::fence_barrier_init();
        tc::prefetch_tmap(&tmap_k);
        tc::prefetch_tmap(&tmap_v);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = s_tmem;

    // Keys past the largest query position of the tile are invisible to all
    // its rows: the tile walk stops there.
    int64_t j_end = j_hi;
    if (a.q_pos) {
        const int64_t last_visible = static_cast<int64_t>(s_maxpos) - a.key_pos0 - a.logical0;   // local index
        j_end = min(j_end, last_visible + 1);
    }
    const int n_tiles = j_end > j_lo ? static_cast<int>((j_end - j_lo + kPN - 1) / kPN) : 0;

    auto fail_wait = [&]() {
        s_abort = 1;
        if (a.status) atomicOr(a.status, 1);
    };
    auto wait = [&](int b, uint32_t parity) -> bool {
        if (*reinterpret_cast<volatile int *>(&s_abort)) return false;
        if (tc::mbar_wait(bar(b), parity, a.status)) return true;
        fail_wait();
        return false;
    };
    // The two warps that share rows (w and w + 4) meet on named barrier 1 + w%4.
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;\n" ::"r"(1 + (warp & 3)) : "memory"); };

    float m_ref = -INFINITY, l_run = 0.f;

    if (warp == kSoftmaxWarps) {
        // ---------------- TMA producer ------------------------------------
        if (lane == 0) {
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int b = j & 1;
                const int y = static_cast<int>(a.row0 + j_lo + static_cast<int64_t>(j) * kPN);
                const int x = kh * kPD;
                if (j >= 2 && !wait(B_KEMPTY + b, ((j >> 1) - 1) & 1)) break;
                tc::mbar_expect_tx(bar(B_KFULL + b), kTileBytes);
                tc::tma_load_2d(sbase + kOffK + b * kTileBytes, &tmap_k, x, y, bar(B_KFULL + b));
                tc::tma_load_2d(sbase + kOffK + b * kTileBytes + kHalfTile, &tmap_k, x + 64, y, bar(B_KFULL + b));
                ++k_issued;
                if (j >= 2 && !wait(B_VEMPTY + b, ((j >> 1) - 1) & 1)) break;
                tc::mbar_expect_tx(bar(B_VFULL + b), kTileBytes);
                tc::tma_load_2d(sbase + kOffV + b * kTileBytes, &tmap_v, x, y, bar(B_VFULL + b));
                tc::tma_load_2d(sbase + kOffV + b * kTileBytes + kHalfTile, &tmap_v, x + 64, y, bar(B_VFULL + b));
                ++v_issued;
            }
            if (*reinterpret_cast<volatile int *>(&s_abort)) {
                // drain: every issued load must land before the CTA exits
                for (int j = (k_issued > 2 ? k_issued - 2 : 0); j < k_issued; ++j)
                    tc::mbar_wait(bar(B_KFULL + (j & 1)), (j >> 1) & 1, nullptr, 100000000ull);
                for (int j = (v_issued > 2 ? v_issued - 2 : 0); j < v_issued; ++j)
                    tc::mbar_wait(bar(B_VFULL + (j & 1)), (j >> 1) & 1, nullptr, 100000000ull);
            }
        }
    } else if (warp == kSoftmaxWarps + 1) {
        // ---------------- MMA issuer ----------------------------------------
        if (lane == 0 && n_tiles > 0) {
            bool ok = wait(B_QFULL, 0);
            tc::tc_fence_after();
            int committed_pv = 0;
            for (int jj = 0; ok && jj <= n_tiles; ++jj) {
                if (jj < n_tiles) {
                    const int b = jj & 1;
                    if (!wait(B_KFULL + b, (jj >> 1) & 1)) break;
                    if (jj >= 2 && !wait(B_SFREE + b, ((jj >> 1) - 1) & 1)) break;
                    tc::tc_fence_after();
                    const uint32_t d_s = tmem + static_cast<uint32_t>(b * kPN);
#pragma unroll
                    for (int kk = 0; kk < kPD / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kHalfTile + (kk & 3) * 32;
                        const uint64_t ad = tc::smem_desc(sbase + kOffQ + off, 16, 1024);
                        const uint64_t bd = tc::smem_desc(sbase + kOffK + b * kTileBytes + off, 16, 1024);
                        tc::mma_f16(d_s, ad, bd, kIdescS, kk > 0);
                    }
                    tc::mma_commit(bar(B_SFULL + b));
                    tc::mma_commit(bar(B_KEMPTY + b));
                }
                if (jj >= 1) {
                    const int j = jj - 1;
                    const int b = j & 1;
                    if (!wait(B_PFULL, j & 1)) break;
                    if (!wait(B_VFULL + b, (j >> 1) & 1)) break;
                    tc::tc_fence_after();
                    const uint32_t d_o = tmem + 2 * kPN;
#pragma unroll
                    for (int kk = 0; kk < kPN / 16; ++kk) {
                        const uint32_t poff = (kk >> 2) * kHalfTile + (kk & 3) * 32;
                        const uint64_t ad = tc::smem_desc(sbase + kOffP + poff, 16, 1024);
                        // V tile as B in MN-major layout: 16 keys = 2048 bytes per k-step;
                        // the second 64-wide d block is kHalfTile away (leading offset),
                        // 8-key row groups are 1024 bytes apart (stride offset).
                        const uint64_t bd = tc::smem_desc(sbase + kOffV + b * kTileBytes + kk * 2048, kHalfTile, 1024);
                        tc::mma_f16(d_o, ad, bd, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(bar(B_PVDONE));
                    tc::mma_commit(bar(B_VEMPTY + b));
                    ++committed_pv;
                }
            }
            if (*reinterpret_cast<volatile int *>(&s_abort) && committed_pv > 0)
                tc::mbar_wait(bar(B_PVDONE), (committed_pv - 1) & 1, nullptr, 100000000ull);   // drain issued MMAs
        }
    } else {
        // ---------------- softmax warps (two threads per query row) -----------
        // Q: this thread's half of its row -> the 128-byte-swizzled K-major layout.
        {
            const __half *qp = a.q + ((static_cast<int64_t>(s) * a.nq + (row_ok ? t_row : 0)) * a.H + kh * a.G +
                                      (m % a.G)) * kPD + hf * 64;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                uint4 v = row_ok ? *reinterpret_cast<const uint4 *>(qp + cc * 8) : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(sm + kOffQ + hf * kHalfTile + m * 128 + ((cc ^ (m & 7)) << 4)) = v;
            }
            tc::fence_proxy_async_smem();
            tc::mbar_arrive(bar(B_QFULL));
        }
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        constexpr int NC = kPN / 2;                 // columns per thread
        // No early exit from this loop: the two warps of a row pair meet on a
        // named barrier every tile, so both must run every iteration.  After
        // a wait gives up, every later wait returns at once and the CTA runs
        // through to its exit (its outputs are then invalid and the status
        // word says so).
        for (int j = 0; j < n_tiles; ++j) {
            const int b = j & 1;
            __all_sync(0xffffffffu, wait(B_SFULL + b, (j >> 1) & 1));
            tc::tc_fence_after();
            uint32_t sr[NC / 32][32];
#pragma unroll
            for (int c = 0; c < NC / 32; ++c) tc::tmem_ld32(lane_base + b * kPN + hf * NC + c * 32, sr[c]);
#pragma unroll
            for (int c = 0; c < NC / 32; ++c) tc::tmem_wait_ld(sr[c]);
            float x[NC];
#pragma unroll
            for (int c = 0; c < NC / 32; ++c)
#pragma unroll
                for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(sr[c][i]);
            tc::tc_fence_before();
            tc::mbar_arrive(bar(B_SFREE + b));

            const int64_t key0 = j_lo + static_cast<int64_t>(j) * kPN + hf * NC;   // local index of column 0
            const int64_t pos0 = a.key_pos0 + a.logical0 + key0;
            const int64_t lim_pos = static_cast<int64_t>(pos_row) - pos0;   // columns > lim_pos are masked
            const int64_t lim_end = j_hi - key0;                            // columns >= lim_end are outside the split
            // Masking only where a tile reaches past a row's position or the
            // split's end (warp-uniform test; most tiles skip it).
            if (__any_sync(0xffffffffu, lim_pos < NC - 1 || lim_end < NC)) {
#pragma unroll
                for (int i = 0; i < NC; ++i)
                    if (i > lim_pos || i >= lim_end) x[i] = -INFINITY;
            }
            // Row maximum on the raw scores (the scale is positive): this
            // half's four chains, then the partner half's value.
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < NC; i += 4) {
                mq[0] = fmaxf(mq[0], x[i]);
                mq[1] = fmaxf(mq[1], x[i + 1]);
                mq[2] = fmaxf(mq[2], x[i + 2]);
                mq[3] = fmaxf(mq[3], x[i + 3]);
            }
            const float mh = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            s_pair[b][hf][m] = mh;
            pair_sync();
            const float mx = fmaxf(mh, s_pair[b][hf ^ 1][m]) * a.scale_log2;
            const float m_new = fmaxf(m_ref, mx);
            const bool resc = m_new > m_ref + kRescaleLog2;   // true on the first finite maximum
            const float ref = resc ? m_new : m_ref;
            const float alpha = resc ? fast_exp2(m_ref - ref) : 1.f;
            const float neg_ref = ref == -INFINITY ? 0.f : -ref;
            // p = 2^(s * scale_log2 - ref): one FMA and one exp2 per score.
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t ph[NC / 2];
#pragma unroll
            for (int i = 0; i < NC; i += 2) {
                const float p0 = fast_exp2(fmaf(x[i], a.scale_log2, neg_ref));
                const float p1 = fast_exp2(fmaf(x[i + 1], a.scale_log2, neg_ref));
                ls[(i >> 1) & 3] += p0 + p1;
                ph[i / 2] = pack_half2(p0, p1);
            }
            l_run = l_run * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));   // this half's columns
            m_ref = ref;
            // P buffer and O are free once PV of the previous tile is done.
            if (j > 0) {
                __all_sync(0xffffffffu, wait(B_PVDONE, (j - 1) & 1));
                tc::tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int c = 0; c < NC / 32; ++c) {
                        uint32_t r[32];
                        tc::tmem_ld32(lane_base + 2 * kPN + hf * NC + c * 32, r);
                        tc::tmem_wait_ld(r);
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * alpha;
                        tc::tmem_st32(lane_base + 2 * kPN + hf * NC + c * 32, v);
                    }
                    tc::tmem_wait_st();
                }
            }
            // this half's 64 keys are exactly one 64-key swizzle block of P
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
                *reinterpret_cast<uint4 *>(sm + kOffP + hf * kHalfTile + m * 128 + ((cc ^ (m & 7)) << 4)) =
                    make_uint4(ph[cc * 4], ph[cc * 4 + 1], ph[cc * 4 + 2], ph[cc * 4 + 3]);
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            tc::mbar_arrive(bar(B_PFULL));
        }
        // ---------------- epilogue: O / l, lse -------------------------------
        float ov[NC];
        bool have = n_tiles > 0 && !*reinterpret_cast<volatile int *>(&s_abort);
        if (have) have = wait(B_PVDONE, (n_tiles - 1) & 1);
        have = __all_sync(0xffffffffu, have);
        if (have) {
            tc::tc_fence_after();
            uint32_t orr[NC / 32][32];
#pragma unroll
            for (int c = 0; c < NC / 32; ++c) tc::tmem_ld32(lane_base + 2 * kPN + hf * NC + c * 32, orr[c]);
#pragma unroll
            for (int c = 0; c < NC / 32; ++c) tc::tmem_wait_ld(orr[c]);
#pragma unroll
            for (int c = 0; c < NC / 32; ++c)
#pragma unroll
                for (int i = 0; i < 32; ++i) ov[c * 32 + i] = __uint_as_float(orr[c][i]);
        }
        // the row's sum is the two halves' sums
        s_pair[2][hf][m] = l_run;
        pair_sync();
        const float l_row = l_run + s_pair[2][hf ^ 1][m];
        if (row_ok) {
            const int64_t r = (static_cast<int64_t>(s) * a.nq + t_row) * a.H + kh * a.G + (m % a.G);
            const bool direct = a.n_splits == 1;
            float *op = (direct ? a.o_out + r * kPD : a.o_split + (static_cast<int64_t>(split) * a.R + r) * kPD) +
                        hf * NC;
            float *lp = direct ? a.lse_out + r : a.lse_split + static_cast<int64_t>(split) * a.R + r;
            if (!have || m_ref == -INFINITY || l_row <= 0.f) {
#pragma unroll
                for (int i = 0; i < NC; i += 4) *reinterpret_cast<float4 *>(op + i) = make_float4(0.f, 0.f, 0.f, 0.f);
                if (hf == 0) *lp = -INFINITY;
            } else {
                const float inv = 1.f / l_row;
#pragma unroll
                for (int i = 0; i < NC; i += 4)
                    *reinterpret_cast<float4 *>(op + i) =
                        make_float4(ov[i] * inv, ov[i + 1] * inv, ov[i + 2] * inv, ov[i + 3] * inv);
                if (hf == 0) *lp = (m_ref + __log2f(l_row)) * 0.6931471805599453f;
            }
        }
    }

    // ---------------- teardown, then the cross-split merge --------------------
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc<512>(tmem);
    }
    if (a.n_splits == 1) return;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(a.counters + unit, 1) == a.n_splits - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (row_ok) {
        // thread (row, half) merges its 64 columns over the splits
        const int64_t r = (static_cast<int64_t>(s) * a.nq + t_row) * a.H + kh * a.G + (m % a.G);
        float M = -INFINITY;
        for (int sp = 0; sp < a.n_splits; ++sp) M = fmaxf(M, __ldcg(a.lse_split + static_cast<int64_t>(sp) * a.R + r));
        float *op = a.o_out + r * kPD + hf * 64;
        if (M == -INFINITY) {
            for (int i = 0; i < 64; i += 4) *reinterpret_cast<float4 *>(op + i) = make_float4(0.f, 0.f, 0.f, 0.f);
            if (hf == 0) a.lse_out[r] = -INFINITY;
        } else {
            float acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) acc[i] = 0.f;
            float W = 0.f;
            for (int sp = 0; sp < a.n_splits; ++sp) {
                const float l = __ldcg(a.lse_split + static_cast<int64_t>(sp) * a.R + r);
                if (l == -INFINITY) continue;
                const float w = fast_exp2((l - M) * 1.4426950408889634f);
                W += w;
                const float4 *src = reinterpret_cast<const float4 *>(
                    a.o_split + (static_cast<int64_t>(sp) * a.R + r) * kPD + hf * 64);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float4 v = __ldcg(src + i);
                    acc[4 * i] = fmaf(w, v.x, acc[4 * i]);
                    acc[4 * i + 1] = fmaf(w, v.y, acc[4 * i + 1]);
                    acc[4 * i + 2] = fmaf(w, v.z, acc[4 * i + 2]);
                    acc[4 * i + 3] = fmaf(w, v.w, acc[4 * i + 3]);
                }
            }
            const float inv = 1.f / W;
            for (int i = 0; i < 64; i += 4)
                *reinterpret_cast<float4 *>(op + i) = make_float4(acc[i] * inv, acc[i + 1] * inv, acc[i + 2] * inv,
                                                                  acc[i + 3] * inv);
            if (hf == 0) a.lse_out[r] = M + __logf(W);
        }
    }
    if (tid == 0) a.counters[unit] = 0;
}

// ---- host side ------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// 2-D map over a cell-major fp16 cache region: x = element within the row
// (Hk*D wide), y = row; box 64 x 128 with the 128-byte swizzle.
static int make_map(skv_handle *h, CUtensorMap *map, const void *base, int64_t n_rows, int Hk, int64_t row_bytes)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(h, SKV_ECUDA, "cuTensorMapEncodeTiled is not available");
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(Hk) * kPD, static_cast<cuuint64_t>(n_rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {64, kPN};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(h, SKV_EUNSUPPORTED, "tensor map encoding failed (%d)", static_cast<int>(r));
    return SKV_OK;
}

bool prefill_eligible(const skv_shape *sh, const void *mask)
{
    return sh->k_type == SKV_F16 && sh->v_type == SKV_F16 && sh->D == kPD && mask == nullptr &&
           (kPM % (sh->H / sh->Hk)) == 0 && static_cast<int64_t>(sh->nq) * (sh->H / sh->Hk) >= 64 &&
           sh->k_row_bytes % 16 == 0 && sh->v_row_bytes % 16 == 0;
}

int prefill_units(const skv_shape *sh) { return sh->Hk * ((sh->nq * (sh->H / sh->Hk) + kPM - 1) / kPM); }

int launch_prefill(skv_handle *h, const PrefillLaunch &L, cudaStream_t st)
{
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(splitkv_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute(prefill)");
        attr_done = true;
    }
    const skv_shape *sh = L.shape;
    const int G = sh->H / sh->Hk;
    CUtensorMap mk, mv;
    int rc = make_map(h, &mk, L.k, L.n_rows, sh->Hk, sh->k_row_bytes);
    if (rc == SKV_OK) rc = make_map(h, &mv, L.v, L.n_rows, sh->Hk, sh->v_row_bytes);
    if (rc) return rc;
    PrefillArgs a;
    memset(&a, 0, sizeof(a));
    a.q = static_cast<const __half *>(L.q);
    a.S = sh->S;
    a.nq = sh->nq;
    a.H = sh->H;
    a.Hk = sh->Hk;
    a.G = G;
    a.scale_log2 = sh->scale * 1.4426950408889634f;
    a.q_pos = L.q_pos;
    a.key_pos0 = L.key_pos0;
    a.logical0 = L.logical0;
    a.row0 = L.row0;
    a.n_local = L.n_local;
    a.m_tiles = (sh->nq * G + kPM - 1) / kPM;
    a.n_splits = L.n_splits;
    a.split_len = L.split_len;
    a.o_split = L.o_split;
    a.lse_split = L.lse_split;
    a.counters = h->counters;
    a.o_out = L.o_out;
    a.lse_out = L.lse_out;
    a.R = static_cast<int64_t>(sh->S) * sh->nq * sh->H;
    a.status = h->status;
    if (a.split_len % kPN) return fail(h, SKV_EINVAL, "prefill split length must be a multiple of %d", kPN);
    if (sh->Hk * a.m_tiles > 65535 || a.n_splits > 65535 || sh->S > 65535)
        return fail(h, SKV_EUNSUPPORTED, "prefill grid too large");
    if (L.row0 + L.n_local > 0x7fffffff) return fail(h, SKV_EUNSUPPORTED, "region too long for the tensor map");
    dim3 grid(static_cast<unsigned>(sh->Hk * a.m_tiles), static_cast<unsigned>(a.n_splits),
              static_cast<unsigned>(sh->S));
    if (h->prof_before) cudaEventRecord(h->prof_before, st);
    splitkv_prefill_kernel<<<grid, kPThreads, kSmem, st>>>(mk, mv, a);
    if (h->prof_after) cudaEventRecord(h->prof_after, st);
    return cuda_fail(h, cudaGetLastError(), "prefill kernel launch");
}

}  // namespace skv
