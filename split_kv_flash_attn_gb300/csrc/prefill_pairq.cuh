// prefill_pairq.cuh -- prefill attention over a dense range of q8_0 / q4_0
// keys and q4_0 values with two 128-row query tiles per CTA (tcgen05).
//
// Over quantised rows the single-tile kernel (prefill_kernel.cuh, MODE 1) is
// bound by its producer warps: every key tile is decoded into an exact
// (hi, lo) pair of fp16 tiles, every value tile into one fp16 tile, and that
// work is paid once per query tile.  Here a CTA owns two query tiles of one
// KV head (the same GQA packing) and one split of the key range, so each
// decoded K and V tile serves both:
//
//   producers  : four warps, one key row a thread: the row's raw K and V
//                segments are staged by cp.async (one slot each; the next
//                tile's K segment is requested as soon as this tile's keys
//                are decoded, its V segment once its values are), then
//                decoded into the K stage (hi and lo, both K slots) and a
//                2-deep V ring.
//   MMA thread : for tile g = 0, 1 in turn, O_g += P_g(j-1) V(j-1), then,
//                once that PV is done, S_g(j) = Q_g hi(j)^T + Q_g lo(j)^T
//                into the same tensor-memory columns (P_g, fp16 pairs, is
//                written over the first half of S_g); Q_g is the A operand
//                in shared memory.  The K stage is free after S_1(j).
//   softmax g  : four warps, one thread per query row of tile g, 64 keys
//                at a time: the half's maximum, its exponentials against the
//                row's reference maximum (which, like O_g, moves only when
//                the maximum grows by more than 2^8), and its P stored over
//                columns whose scores are already consumed.
//
// Tensor memory: S_0/P_0 in columns 0-127, S_1/P_1 128-255, O_0 256-383,
// O_1 384-511.  Shared memory: Q_0, Q_1, the K stage (hi, lo), two V stages,
// barriers, then the raw K and V segments (223 KB with q8_0 keys).  The
// split's result (O normalised, lse) is merged across splits by the last CTA
// of the pair.  Every mbarrier wait is bounded; a wait that gives up sets the
// handle's device status word and the CTA stops issuing work, drains what it
// issued and frees its tensor memory.
#pragma once

#include "prefill_kernel.cuh"

namespace skv {
namespace pf {

constexpr int kQpSoftmaxWarps = 8;              // warps 0-3: tile 0, warps 4-7: tile 1
constexpr int kQpProducerWarps = 4;             // warps 8-11
constexpr int kQpMmaWarp = kQpSoftmaxWarps + kQpProducerWarps;
constexpr int kQpThreads = (kQpMmaWarp + 1) * 32;
constexpr int kQpProducers = kQpProducerWarps * 32;
static_assert(kQpProducers == kPN, "one key row a producer thread");
constexpr int kQpOffQ = 0;                      // Q_0, Q_1 (A operands, K-major, 128-byte swizzle)
constexpr int kQpOffK = kQpOffQ + 2 * kTileBytes;   // hi, lo
constexpr int kQpOffV = kQpOffK + 2 * kTileBytes;   // two stages
constexpr int kQpOffBar = kQpOffV + 2 * kTileBytes;
constexpr int kQpOffRaw = kQpOffBar + 256;
template <int KT>
__host__ __device__ constexpr int qp_smem_bytes()
{
    return kQpOffRaw + kPN * (seg_bytes_of(KT) + seg_bytes_of(SKV_Q4_0)) + 1024;   // + alignment slack
}
static_assert(qp_smem_bytes<SKV_Q8_0>() <= 227 * 1024, "shared memory per CTA");
constexpr int kQpOCol = 2 * kPN;                // O_g in columns kQpOCol + g * kPD
static_assert(kQpOCol + 2 * kPD <= 512, "tensor memory columns");
// Barriers.  K full: the 128 producer threads; K empty: the commit after
// S_1 (or S_0 alone) of the tile.  V full / V empty per V stage (tile j in
// stage j % 2).  Per query tile g (+g): Q full (its 128 softmax threads), S
// full and PV done (MMA commits), P full (its softmax threads).  Tile j is
// phase j of K full / K empty, S full, P full and PV done, and phase j / 2 of
// its V stage's barriers; no waiter is ever two phases behind, because each
// side needs the other's next step before it can complete another phase.
enum { QB_KFULL = 0, QB_KEMPTY = 1, QB_VFULL = 2, QB_VEMPTY = 4, QB_QFULL = 6, QB_SFULL = 8, QB_PFULL = 10,
       QB_PDONE = 12, QB_COUNT = 14 };
static_assert(QB_COUNT * 8 <= 256, "barrier area");

template <int KT>
__global__ void __launch_bounds__(kQpThreads, 1)
    splitkv_prefill_pairq_kernel(const PrefillArgs a)
{
    constexpr int VT = SKV_Q4_0;
    constexpr int SEGK = seg_bytes_of(KT), SEGV = seg_bytes_of(VT);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(sm);
    const uint32_t bar0 = sbase + kQpOffBar;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ int s_maxpos;
    __shared__ int s_last;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int n_pairs = (a.m_tiles + 1) / 2;
    const int pr = blockIdx.x % n_pairs;
    const int kh = blockIdx.x / n_pairs;
    const int split = blockIdx.z;
    const int s = blockIdx.y;
    const int unit = (s * a.Hk + kh) * n_pairs + pr;
    const bool two = 2 * pr + 1 < a.m_tiles;     // the pair's second query tile exists
    const int tpt = kPM / a.G;                   // tokens per query tile
    const int64_t j_lo = static_cast<int64_t>(split) * a.split_len;
    const int64_t j_hi = min(a.n_local, j_lo + a.split_len);

    // Softmax threads: tile g, query row m = TMEM lane (warp % 4) * 32 + lane.
    const bool softmax = warp < kQpSoftmaxWarps;
    const int g = (warp >> 2) & 1;
    const bool tile_on = softmax && (g == 0 || two);
    const int m = (warp & 3) * 32 + lane;
    const int t_row = (2 * pr + g) * tpt + m / a.G;
    const bool row_ok = tile_on && t_row < a.nq;
    const int32_t pos_row = (row_ok && a.q_pos) ? a.q_pos[static_cast<int64_t>(s) * a.nq + t_row] : INT32_MAX;

    if (tid == 0) {
        s_abort = 0;
        s_maxpos = INT32_MIN;
    }
    __syncthreads();
    if (a.q_pos && row_ok) atomicMax(&s_maxpos, pos_row);
    if (warp == 0) {
        tc::tmem_alloc<512>(smem_addr(&s_tmem));
        tc::tmem_relinquish();
    }
    if (tid == kQpSoftmaxWarps * 32) {
        tc::mbar_init(bar(QB_KFULL), kQpProducers);
        tc::mbar_init(bar(QB_KEMPTY), 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(QB_VFULL + i), kQpProducers);
            tc::mbar_init(bar(QB_VEMPTY + i), 1);
            tc::mbar_init(bar(QB_QFULL + i), kPM);
            tc::mbar_init(bar(QB_SFULL + i), 1);
            tc::mbar_init(bar(QB_PFULL + i), kPM);
            tc::mbar_init(bar(QB_PDONE + i), 1);
        }
        tc::fence_barrier_init();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = s_tmem;

    // Keys past the largest query position of the pair are invisible to all
    // its rows: the tile walk stops there.
    int64_t j_end = j_hi;
    if (a.q_pos) {
        const int64_t last_visible = static_cast<int64_t>(s_maxpos) - a.key_pos0 - a.logical0;   // local index
        j_end = min(j_end, last_visible + 1);
    }
    const int n_tiles = j_end > j_lo ? static_cast<int>((j_end - j_lo + kPN - 1) / kPN) : 0;

    // A phase already complete is taken at once; the abort flag is read only
    // when the barrier is not ready.
    auto wait = [&](int b, uint32_t parity) -> bool {
        if (tc::mbar_try_wait(bar(b), parity)) return true;
        if (*reinterpret_cast<volatile int *>(&s_abort)) return false;
        if (tc::mbar_wait(bar(b), parity, a.status)) return true;
        s_abort = 1;
        if (a.status) atomicOr(a.status, 1);
        return false;
    };

    float m_ref = -INFINITY, l_run = 0.f;

    if (warp >= kQpSoftmaxWarps && warp < kQpMmaWarp) {
        // ---------------- producers: one key row of every tile a thread --------
        const int r0 = tid - kQpSoftmaxWarps * 32;
        auto tile_row = [&](int j) -> int64_t {
            const int64_t key = j_lo + static_cast<int64_t>(j) * kPN + r0;
            return key < j_hi ? a.row0 + key : -1;
        };
        uint8_t *raw_k = sm + kQpOffRaw + r0 * SEGK;
        uint8_t *raw_v = sm + kQpOffRaw + kPN * SEGK + r0 * SEGV;
        auto issue = [&](uint8_t *dst, const uint8_t *base, int64_t row_bytes, int seg, int64_t row) {
            const uint8_t *src = row >= 0 ? base + row * row_bytes + static_cast<int64_t>(kh) * seg : nullptr;
            for (int i = 0; i < seg / 8; ++i)
                cp_async8(smem_addr(dst + 8 * i), src ? src + 8 * i : base, src ? 8 : 0);
            cp_async_commit();
        };
        int64_t e0 = n_tiles > 0 ? tile_row(0) : -1;
        int64_t e1 = n_tiles > 1 ? tile_row(1) : -1;
        if (n_tiles > 0) {
            issue(raw_k, a.k, a.k_row_bytes, SEGK, e0);
            issue(raw_v, a.v, a.v_row_bytes, SEGV, e0);
        }
        for (int j = 0; j < n_tiles; ++j) {
            const int b = j & 1;
            const bool more = j + 1 < n_tiles;
            // keys: this thread's K segment of tile j has landed (its V
            // segment may not have), and S_1 of tile j-1 has read the K stage
            cp_async_wait<1>();
            if (!__all_sync(0xffffffffu, j < 1 || wait(QB_KEMPTY, (j - 1) & 1))) break;
            {
                uint32_t w[QSeg<KT>::NW];
#pragma unroll
                for (int i = 0; i < QSeg<KT>::NW; ++i) w[i] = *reinterpret_cast<const uint32_t *>(raw_k + 4 * i);
                store_row<KT, true>(w, e0 >= 0, sm + kQpOffK, r0, sm + kQpOffK + kTileBytes);
            }
            tc::fence_proxy_async_smem();
            tc::mbar_arrive(bar(QB_KFULL));
            if (more) issue(raw_k, a.k, a.k_row_bytes, SEGK, e1);
            // values: tile j's V segment, once PV of tile j-2 has read the stage
            if (more) cp_async_wait<1>();
            else cp_async_wait<0>();
            if (!__all_sync(0xffffffffu, j < 2 || wait(QB_VEMPTY + b, ((j >> 1) - 1) & 1))) break;
            {
                uint32_t w[QSeg<VT>::NW];
#pragma unroll
                for (int i = 0; i < QSeg<VT>::NW; ++i) w[i] = *reinterpret_cast<const uint32_t *>(raw_v + 4 * i);
                store_row<VT>(w, e0 >= 0, sm + kQpOffV + b * kTileBytes, r0);
            }
            tc::fence_proxy_async_smem();
            tc::mbar_arrive(bar(QB_VFULL + b));
            if (more) issue(raw_v, a.v, a.v_row_bytes, SEGV, e1);
            e0 = e1;
            e1 = j + 2 < n_tiles ? tile_row(j + 2) : -1;
        }
        cp_async_wait<0>();
    } else if (warp == kQpMmaWarp) {
        // ---------------- MMA issuer ----------------------------------------
        if (lane == 0 && n_tiles > 0) {
            const int ng = two ? 2 : 1;
            bool ok = wait(QB_QFULL, 0) && (!two || wait(QB_QFULL + 1, 0));
            tc::tc_fence_after();
            int last_bar = -1;                      // barrier and phase of the last commit
            uint32_t last_par = 0;
            // operand descriptors of the first Q, K and V buffers; the rest are offsets
            const uint64_t dq0 = tc::smem_desc(sbase + kQpOffQ, 16, 1024);
            const uint64_t dk0 = tc::smem_desc(sbase + kQpOffK, 16, 1024);
            const uint64_t dv0 = tc::smem_desc(sbase + kQpOffV, kHalfTile, 1024);
            for (int jj = 0; ok && jj <= n_tiles; ++jj) {
                for (int gg = 0; gg < ng; ++gg) {
                    const uint32_t d_s = tmem + static_cast<uint32_t>(gg * kPN);
                    if (jj >= 1) {
                        // O_g += P_g(j) V(j), P_g in the first 64 columns of S_g
                        const int j = jj - 1, b = j & 1;
                        if (!wait(QB_PFULL + gg, j & 1)) { ok = false; break; }
                        if (gg == 0 && !wait(QB_VFULL + b, (j >> 1) & 1)) { ok = false; break; }
                        tc::tc_fence_after();
                        const uint32_t d_o = tmem + static_cast<uint32_t>(kQpOCol + gg * kPD);
#pragma unroll
                        for (int kk = 0; kk < kPN / 16; ++kk) {
                            // V tile as B in MN-major layout: 16 keys = 2048 bytes per
                            // k-step; the second 64-wide d block is kHalfTile away.
                            const uint64_t bd = tc::desc_add(dv0, b * kTileBytes + kk * 2048);
                            tc::mma_f16_ts(d_o, d_s + static_cast<uint32_t>(kk * 8), bd, kIdescPV,
                                           (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc::mma_commit(bar(QB_PDONE + gg));
                        last_bar = QB_PDONE + gg;
                        last_par = j & 1;
                        if (gg == ng - 1) tc::mma_commit(bar(QB_VEMPTY + b));
                    }
                    if (jj < n_tiles) {
                        // S_g(jj) = Q_g hi^T + Q_g lo^T, once PV_g(jj-1) has read P_g
                        if (gg == 0 && !wait(QB_KFULL, jj & 1)) { ok = false; break; }
                        if (jj >= 1 && !wait(QB_PDONE + gg, (jj - 1) & 1)) { ok = false; break; }
                        tc::tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < 2 * (kPD / 16); ++ks) {
                            const int kk = ks % (kPD / 16);
                            const uint32_t off = (kk >> 2) * kHalfTile + (kk & 3) * 32;
                            const uint64_t ad = tc::desc_add(dq0, gg * kTileBytes + off);
                            const uint64_t bd = tc::desc_add(dk0, (ks / (kPD / 16)) * kTileBytes + off);
                            tc::mma_f16_ss(d_s, ad, bd, kIdescS, ks > 0 ? 1u : 0u);
                        }
                        tc::mma_commit(bar(QB_SFULL + gg));
                        last_bar = QB_SFULL + gg;
                        last_par = jj & 1;
                        if (gg == ng - 1) tc::mma_commit(bar(QB_KEMPTY));
                    }
                }
            }
            if (*reinterpret_cast<volatile int *>(&s_abort)) {
                // drain issued MMAs: the last commit covers every MMA issued before it
                if (last_bar >= 0) tc::mbar_wait(bar(last_bar), last_par, nullptr, 100000000ull);
            } else {
                // no producer waits for the last commits on the stages' free
                // barriers; they are awaited here, so that none is in flight at exit
                wait(QB_KEMPTY, (n_tiles - 1) & 1);
                for (int j = max(0, n_tiles - 2); j < n_tiles; ++j) wait(QB_VEMPTY + (j & 1), (j >> 1) & 1);
            }
        }
    } else if (tile_on) {
        // ---------------- softmax warps: one thread per query row -------------
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t s_col = lane_base + static_cast<uint32_t>(g * kPN);
        const uint32_t o_col = lane_base + static_cast<uint32_t>(kQpOCol + g * kPD);
        {
            // Q row m of tile g into shared memory (the MMA's A operand)
            const __half *qp = a.q + ((static_cast<int64_t>(s) * a.nq + (row_ok ? t_row : 0)) * a.H + kh * a.G +
                                      (m % a.G)) * kPD;
            uint8_t *qt = sm + kQpOffQ + g * kTileBytes;
#pragma unroll
            for (int c = 0; c < kPD / 8; ++c) {
                const uint4 v = row_ok ? *reinterpret_cast<const uint4 *>(qp + c * 8) : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(qt + tile_off(m, c)) = v;
            }
            tc::fence_proxy_async_smem();
            tc::mbar_arrive(bar(QB_QFULL + g));
        }
        constexpr int NH = kPN / 2;                 // columns per half
        // No early exit from this loop: after a wait gives up, every later
        // wait returns at once and the warp runs through to the epilogue (the
        // outputs are then invalid and the status word says so).
        for (int j = 0; j < n_tiles; ++j) {
            const int64_t key0 = j_lo + static_cast<int64_t>(j) * kPN;   // local index of column 0
            __all_sync(0xffffffffu, wait(QB_SFULL + g, j & 1));
            tc::tc_fence_after();
            const int64_t pos0 = a.key_pos0 + a.logical0 + key0;
            const int64_t lim_pos = static_cast<int64_t>(pos_row) - pos0;   // columns > lim_pos are masked
            const int64_t lim_end = j_hi - key0;                            // columns >= lim_end are outside the split
            const bool masked = __any_sync(0xffffffffu, lim_pos < kPN - 1 || lim_end < kPN);
            float x[NH];
            auto load_half = [&](int h) {
                uint32_t sr[NH / 32][32];
#pragma unroll
                for (int c = 0; c < NH / 32; ++c) tc::tmem_ld32(s_col + h * NH + c * 32, sr[c]);
#pragma unroll
                for (int c = 0; c < NH / 32; ++c) tc::tmem_wait_ld(sr[c]);
#pragma unroll
                for (int c = 0; c < NH / 32; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(sr[c][i]);
                if (masked) {
#pragma unroll
                    for (int i = 0; i < NH; ++i)
                        if (h * NH + i > lim_pos || h * NH + i >= lim_end) x[i] = -INFINITY;
                }
            };
            // One pass, a half (64 keys) at a time: a half's exponentials are
            // taken against the reference maximum as it stands after that
            // half (it moves only when the maximum grows by more than 2^8),
            // and P (keys h*64 + 2c, +1 as fp16 pairs in column h*32 + c of
            // S_g) is stored over scores already consumed.  When the second
            // half moves the reference, the first half's stored P is scaled
            // down to it (by at most 2^-8: no fp16 overflow or loss).
            float ref = m_ref, ls0 = 0.f, ls1 = 0.f;
            float beta = 1.f;                         // the first half's factor to the final reference
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                load_half(h);
                float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < NH; i += 4) {
                    mq[0] = fmaxf(mq[0], x[i]);
                    mq[1] = fmaxf(mq[1], x[i + 1]);
                    mq[2] = fmaxf(mq[2], x[i + 2]);
                    mq[3] = fmaxf(mq[3], x[i + 3]);
                }
                const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * a.scale_log2;
                const float prev = ref;
                if (mx > ref + kRescaleLog2) ref = mx;          // true on the first finite maximum
                const float neg_ref = ref == -INFINITY ? 0.f : -ref;
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t ph[NH / 2];
#pragma unroll
                for (int i = 0; i < NH; i += 2) {
                    const float p0 = fast_exp2(fmaf(x[i], a.scale_log2, neg_ref));
                    const float p1 = fast_exp2(fmaf(x[i + 1], a.scale_log2, neg_ref));
                    ls[(i >> 1) & 3] += p0 + p1;
                    ph[i / 2] = pack_half2(p0, p1);
                }
                const float lh = (ls[0] + ls[1]) + (ls[2] + ls[3]);
                if (h == 0) {
                    ls0 = lh;
                } else {
                    ls1 = lh;
                    if (ref != prev) beta = prev == -INFINITY ? 0.f : fast_exp2(prev - ref);
                    if (__any_sync(0xffffffffu, beta != 1.f)) {
                        // the first half's P, stored above, to the moved reference
                        tc::tmem_wait_st();
                        uint32_t pr[32];
                        tc::tmem_ld32(s_col, pr);
                        tc::tmem_wait_ld(pr);
                        const __half2 bb = __float2half2_rn(beta);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&pr[i]), bb);
                            pr[i] = *reinterpret_cast<const uint32_t *>(&v);
                        }
                        tc::tmem_st32u(s_col, pr);
                    }
                }
                tc::tmem_st32u(s_col + h * (NH / 2), ph);
            }
            const float alpha = ref == m_ref ? 1.f : (m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - ref));
            // O_g holds every PV up to tile j-1 (S_g(j) was issued after the
            // last of them was done) and no PV of tile j before P_g is full:
            // the rare rescale needs no further wait.
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int c = 0; c < kPD / 32; ++c) {
                    uint32_t rr[32];
                    tc::tmem_ld32(o_col + c * 32, rr);
                    tc::tmem_wait_ld(rr);
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(rr[i]) * alpha;
                    tc::tmem_st32(o_col + c * 32, v);
                }
            }
            l_run = l_run * alpha + (ls0 * beta + ls1);
            m_ref = ref;
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(bar(QB_PFULL + g));
        }
        // ---------------- epilogue: O / l, lse -------------------------------
        bool have = n_tiles > 0 && !*reinterpret_cast<volatile int *>(&s_abort);
        if (have) have = wait(QB_PDONE + g, (n_tiles - 1) & 1);   // the last PV
        have = __all_sync(0xffffffffu, have);
        if (have) tc::tc_fence_after();
        const int64_t r = (static_cast<int64_t>(s) * a.nq + t_row) * a.H + kh * a.G + (m % a.G);
        const bool direct = a.n_splits == 1;
        float *op = direct ? a.o_out + r * kPD : a.o_split + (static_cast<int64_t>(split) * a.R + r) * kPD;
        float *lp = direct ? a.lse_out + r : a.lse_split + static_cast<int64_t>(split) * a.R + r;
        const bool empty = !have || m_ref == -INFINITY || l_run <= 0.f;
        const float inv = empty ? 0.f : 1.f / l_run;
#pragma unroll
        for (int c = 0; c < kPD / 32; ++c) {
            uint32_t orr[32];
            if (have) {
                tc::tmem_ld32(o_col + c * 32, orr);          // warp-wide: every lane takes part
                tc::tmem_wait_ld(orr);
            }
            if (row_ok) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4 *>(op + c * 32 + i) =
                        empty ? make_float4(0.f, 0.f, 0.f, 0.f)
                              : make_float4(__uint_as_float(orr[i]) * inv, __uint_as_float(orr[i + 1]) * inv,
                                            __uint_as_float(orr[i + 2]) * inv, __uint_as_float(orr[i + 3]) * inv);
            }
        }
        if (row_ok) *lp = empty ? -INFINITY : (m_ref + __log2f(l_run)) * 0.6931471805599453f;
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
        // thread (row) merges its 128 columns over the splits, 64 at a time
        const int64_t r = (static_cast<int64_t>(s) * a.nq + t_row) * a.H + kh * a.G + (m % a.G);
        float M = -INFINITY;
        for (int sp = 0; sp < a.n_splits; ++sp) M = fmaxf(M, __ldcg(a.lse_split + static_cast<int64_t>(sp) * a.R + r));
        float *op = a.o_out + r * kPD;
        if (M == -INFINITY) {
            for (int i = 0; i < kPD; i += 4) *reinterpret_cast<float4 *>(op + i) = make_float4(0.f, 0.f, 0.f, 0.f);
            a.lse_out[r] = -INFINITY;
        } else {
            float W = 0.f;
            for (int hf = 0; hf < 2; ++hf) {
                float acc[64];
#pragma unroll
                for (int i = 0; i < 64; ++i) acc[i] = 0.f;
                W = 0.f;
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
                    *reinterpret_cast<float4 *>(op + hf * 64 + i) =
                        make_float4(acc[i] * inv, acc[i + 1] * inv, acc[i + 2] * inv, acc[i + 3] * inv);
            }
            a.lse_out[r] = M + __logf(W);
        }
    }
    if (tid == 0) a.counters[unit] = 0;
}

namespace {
template <int KT>
KernelAttrCache &prefill_pairq_attr_cache()
{
    static KernelAttrCache c;
    return c;
}
}  // namespace

// Launch the pair instance: grid x = (KV head, query-tile pair), y =
// sequence, z = split.
template <int KT>
int launch_prefill_pairq_t(skv_handle *h, const PrefillArgs &a, dim3 grid, cudaStream_t st)
{
    cudaError_t e = kernel_smem_optin(prefill_pairq_attr_cache<KT>(),
                                      reinterpret_cast<const void *>(splitkv_prefill_pairq_kernel<KT>),
                                      qp_smem_bytes<KT>(), kQpThreads, nullptr);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute(prefill pair)");
    if (h->prof_before) cudaEventRecord(h->prof_before, st);
    splitkv_prefill_pairq_kernel<KT><<<grid, kQpThreads, qp_smem_bytes<KT>(), st>>>(a);
    if (h->prof_after) cudaEventRecord(h->prof_after, st);
    return cuda_fail(h, cudaGetLastError(), "prefill pair kernel launch");
}

}  // namespace pf
}  // namespace skv
