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
//   * cp.async (16 B for fp16 rows, 8/4 B for q8_0/q4_0 segments) stages the
//     tile's K and V head segments into shared memory, STAGES-1 tiles ahead.
//     Rows come from a dense range, from a row list (padding rows read
//     nothing: zero-filled), or from pages of a block cache.
//   * each of the 4 warps takes 16 keys: S^T = K Q^T with mma.sync m16n8k16
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
    static constexpr int STAGES = (KT == SKV_F16 && VT == SKV_F16) ? 3 : 4;
    static constexpr int SEGK = Seg<KT, D>::bytes;
    static constexpr int SEGV = Seg<VT, D>::bytes;
    static constexpr int stage_k = ((kTile * SEGK + 127) / 128) * 128;
    static constexpr int stage_v = ((kTile * SEGV + 127) / 128) * 128;
    static constexpr int stage_bytes = stage_k + stage_v;
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
};

// Byte offset of 16-byte chunk `ch` of row `r` in a swizzled fp16 tile whose
// rows are D halfs: chunk index XOR (r mod 8) keeps ldmatrix conflict-free.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int ch)
{
    return static_cast<uint32_t>(r * (2 * D) + ((ch ^ (r & 7)) << 4));
}

// Convert 16 keys of q8_0 / q4_0 head segments (raw stage rows) into an fp16
// code tile (swizzled, 16 x D) and per-(key, block) fp32 scales.
template <int T, int D>
__device__ __forceinline__ void convert_codes(const uint8_t *raw, __half *code, float *scale, int lane)
{
    constexpr int SEG = Seg<T, D>::bytes;
    constexpr int BLK = T == SKV_Q8_0 ? 34 : 18;
    constexpr int C8 = D / 8;   // 8-value chunks per key
#pragma unroll 2
    for (int idx = lane; idx < 16 * C8; idx += 32) {
        const int kk = idx / C8;
        const int c8 = idx % C8;
        const int b = c8 >> 2;
        const int part = c8 & 3;
        const uint8_t *blk = raw + kk * SEG + b * BLK;
        __align__(16) __half v[8];
        if constexpr (T == SKV_Q8_0) {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __int2half_rn(static_cast<int8_t>(blk[2 + part * 8 + e]));
        } else {
            const int byte0 = (part & 1) * 8;
            const int shift = (part >> 1) * 4;
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __int2half_rn(((blk[2 + byte0 + e] >> shift) & 0xF) - 8);
        }
        *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(code) + swz<D>(kk, c8)) =
            *reinterpret_cast<const uint4 *>(v);
        if (part == 0) {
            const __half d = *reinterpret_cast<const __half *>(blk);
            scale[kk * (D / 32) + b] = __half2float(d);
        }
    }
}

template <int D, int KT, int VT>
__global__ void __launch_bounds__(128) splitkv_decode_kernel(const DecodeArgs a)
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

    extern __shared__ __align__(128) uint8_t smem[];
    int32_t *idx_s = reinterpret_cast<int32_t *>(smem + C::idx_off);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ---- unit and split -------------------------------------------------
    const int split = blockIdx.x;
    const int unit = blockIdx.y;
    const int cg = unit % a.n_cg;
    const int sk = unit / a.n_cg;
    const int kh = sk % a.Hk;
    const int s = sk / a.Hk;
    const int64_t j_lo = static_cast<int64_t>(split) * a.split_len;
    const int64_t j_hi = min(a.n_local, j_lo + a.split_len);
    const int64_t list = a.rows_per_head ? (static_cast<int64_t>(s) * a.Hk + kh) : s;
    const int lg_pr = a.row_mode == ROWS_PAGED ? (31 - __clz(a.page_rows)) : 0;
    const int64_t page_lo = j_lo >> lg_pr;

    // ---- row indices of this split (list / paged modes) -----------------
    if (a.row_mode == ROWS_LIST) {
        const int32_t *src = a.rows + list * a.rows_ld + a.rows_off;
        for (int64_t i = tid; i < j_hi - j_lo; i += C::kThreads) idx_s[i] = __ldg(src + j_lo + i);
    } else if (a.row_mode == ROWS_PAGED) {
        const int32_t *src = a.rows + list * a.rows_ld;
        const int64_t n_pages = j_hi > j_lo ? ((j_hi - 1) >> lg_pr) - page_lo + 1 : 0;
        for (int64_t i = tid; i < n_pages; i += C::kThreads) idx_s[i] = __ldg(src + page_lo + i);
    }
    __syncthreads();

    // Byte pointer of key j's head segment (nullptr: absent key).
    auto seg_ptr = [&](const uint8_t *base, int64_t row_bytes, int seg, int64_t j) -> const uint8_t * {
        if (j >= j_hi) return nullptr;
        if (a.row_mode == ROWS_DENSE) return base + (a.row0 + j) * row_bytes + static_cast<int64_t>(kh) * seg;
        if (a.row_mode == ROWS_LIST) {
            const int32_t r = idx_s[j - j_lo];
            return r < 0 ? nullptr : base + static_cast<int64_t>(r) * row_bytes + static_cast<int64_t>(kh) * seg;
        }
        const int32_t pg = idx_s[(j >> lg_pr) - page_lo];
        if (pg < 0) return nullptr;
        return base + ((static_cast<int64_t>(pg) << lg_pr) + (j & (a.page_rows - 1))) * seg;
    };

    auto load_tile = [&](int t, int st) {
        uint8_t *sk_ = smem + st * C::stage_bytes;
        uint8_t *sv_ = sk_ + C::stage_k;
        const int64_t jt = j_lo + static_cast<int64_t>(t) * kTile;
        {
            constexpr int CPR = SEGK / CHK;
            constexpr int TOT = kTile * CPR;
#pragma unroll
            for (int it = 0; it < (TOT + C::kThreads - 1) / C::kThreads; ++it) {
                const int c = tid + it * C::kThreads;
                if (TOT % C::kThreads != 0 && c >= TOT) break;
                const int r = c / CPR;
                const int ch = c % CPR;
                const uint8_t *src = seg_ptr(a.k, a.k_row_bytes, SEGK, jt + r);
                const uint32_t dst = smem_addr(sk_) + (QK ? static_cast<uint32_t>(r * SEGK + ch * CHK) : swz<D>(r, ch));
                cp_async<CHK>(dst, src ? src + ch * CHK : a.k, src != nullptr);
            }
        }
        {
            constexpr int CPR = SEGV / CHV;
            constexpr int TOT = kTile * CPR;
#pragma unroll
            for (int it = 0; it < (TOT + C::kThreads - 1) / C::kThreads; ++it) {
                const int c = tid + it * C::kThreads;
                if (TOT % C::kThreads != 0 && c >= TOT) break;
                const int r = c / CPR;
                const int ch = c % CPR;
                const uint8_t *src = seg_ptr(a.v, a.v_row_bytes, SEGV, jt + r);
                const uint32_t dst = smem_addr(sv_) + (QV ? static_cast<uint32_t>(r * SEGV + ch * CHV) : swz<D>(r, ch));
                cp_async<CHV>(dst, src ? src + ch * CHV : a.v, src != nullptr);
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

    // ---- pipeline -------------------------------------------------------
#pragma unroll
    for (int p = 0; p < STAGES - 1; ++p) {
        if (p < n_tiles) load_tile(p, p);
        cp_async_commit();
    }
    for (int i = 0; i < n_tiles; ++i) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        {
            const int nt = i + STAGES - 1;
            if (nt < n_tiles) load_tile(nt, nt % STAGES);
            cp_async_commit();
        }
        const int st = i % STAGES;
        const uint8_t *sk_ = smem + st * C::stage_bytes;
        const uint8_t *sv_ = sk_ + C::stage_k;
        const int wrow = warp * 16;
        const int64_t jw = j_lo + static_cast<int64_t>(i) * kTile + wrow;   // first key of this warp
        const int r0 = lane >> 2;
        const bool v0 = seg_ptr(a.k, a.k_row_bytes, SEGK, jw + r0) != nullptr;
        const bool v1 = seg_ptr(a.k, a.k_row_bytes, SEGK, jw + r0 + 8) != nullptr;
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
    {
        const int col = tid >> 4;
        const int sub = tid & 15;
        const int c = cg * 8 + col;
        const int t = c / a.G;
        const int g = c % a.G;
        if (t < a.nq) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, mg_m[w * 8 + col]);
            const int64_t r = (static_cast<int64_t>(s) * a.nq + t) * a.H + kh * a.G + g;
            const int64_t part = a.part0 + split;
            float *op = a.o_part + (part * a.R + r) * D;
            if (M == -INFINITY) {
                for (int d = sub; d < D; d += 16) op[d] = 0.f;
                if (sub == 0) a.lse_part[part * a.R + r] = -INFINITY;
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
                if (sub == 0) a.lse_part[part * a.R + r] = (M + __log2f(L)) * 0.6931471805599453f;
            }
        }
    }
}

template <int D, int KT, int VT>
int launch_decode_t(skv_handle *h, const DecodeArgs &a, cudaStream_t st)
{
    using C = DecodeCfg<D, KT, VT>;
    static bool attr_done = false;   // per process; the attribute is per function, not per device
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(splitkv_decode_kernel<D, KT, VT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::smem);
        if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute(decode)");
        attr_done = true;
    }
    const int units = a.S * a.Hk * a.n_cg;
    if (units > 65535) return fail(h, SKV_EUNSUPPORTED, "too many (sequence, KV head, column group) units: %d", units);
    dim3 grid(static_cast<unsigned>(a.n_splits), static_cast<unsigned>(units));
    splitkv_decode_kernel<D, KT, VT><<<grid, C::kThreads, C::smem, st>>>(a);
    return cuda_fail(h, cudaGetLastError(), "decode kernel launch");
}

template <int D, int KT, int VT>
int decode_ctas_per_sm_t(skv_handle *h)
{
    using C = DecodeCfg<D, KT, VT>;
    static int cached = -1;
    if (cached < 0) {
        if (cudaFuncSetAttribute(splitkv_decode_kernel<D, KT, VT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::smem) != cudaSuccess)
            return 0;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, splitkv_decode_kernel<D, KT, VT>, C::kThreads,
                                                          C::smem) != cudaSuccess)
            return 0;
        cached = n;
    }
    (void)h;
    return cached;
}

}  // namespace skv
