// decode_rows.cu -- split-KV decode over a dense range of quantised rows
// (q8_0 / q4_0 K and V, head dim 128), one CTA per (sequence, column group,
// key split) covering every KV head.
//
// A cell-major row holds all KV heads, so a range of rows is one contiguous
// span: each 32-row stage of K and of V arrives as 16 bulk copies of two
// whole rows each (cp.async.bulk, completion counted on an mbarrier), padded
// apart in shared memory against bank conflicts, instead of one copy per head
// segment.  Warp w owns KV head w: for its 32 keys per stage it
//   * builds the m16n8k16 A fragments of K straight from the raw codes in
//     shared memory (no converted tile): the head dimension is permuted so
//     that each thread's eight values of a 32-value block are eight adjacent
//     code bytes (q8_0) or the two nibbles of four adjacent bytes (q4_0); the
//     query fragments use the same permutation, so every dot product is
//     unchanged.  Codes become exact fp16 values by a byte permute under the
//     exponent byte 0x64 and one half2 subtract; the block's fp16 scale
//     multiplies the block's partial dot product in fp32.
//   * runs the online softmax per column in log2 units,
//   * accumulates O^T += V^T P^T with V^T fragments built from the codes the
//     same way (output dims permuted, undone when O is written) and the V
//     scale folded into that block's probabilities.
// Each warp holds the whole split of its head, so a CTA needs no merge of its
// warps; the splits of a launch are merged by the log-sum-exp combine.
#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace skv {
namespace {

constexpr int kRD = 128;        // head dim
constexpr int kRRows = 32;      // keys per stage
constexpr int kRStages = 2;

template <int T>
struct QB {
    static constexpr int blk = T == SKV_Q8_0 ? 34 : 18;   // bytes per 32-value block
    static constexpr int seg = 4 * blk;                    // bytes per head segment
};

// Pad after each 2-row chunk (16-byte multiple) that makes the chunk stride
// 8 banks mod 32, for rows whose byte stride is a multiple of 16.
__host__ __device__ __forceinline__ uint32_t chunk_pad(int64_t row_bytes)
{
    const int64_t words = 2 * (row_bytes / 4);
    return static_cast<uint32_t>(((8 - words % 32) % 32 + 32) % 32) * 4;
}
__host__ __device__ __forceinline__ int64_t rows_stage_bytes(int64_t krb, int64_t vrb)
{
    return (kRRows / 2) * (2 * krb + chunk_pad(krb) + 2 * vrb + chunk_pad(vrb));
}

__device__ __forceinline__ uint32_t ld_s16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

// Bytes 0,1 (SEL = 0x4140) or 2,3 (SEL = 0x4342) of w -> half2(1024 + b, ...)
// minus `bias` (half2): the codes' exact values as fp16.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t to_h2(uint32_t w, uint32_t bias)
{
    const uint32_t h = __byte_perm(w, 0x64646464u, SEL);
    __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&h), *reinterpret_cast<const __half2 *>(&bias));
    return *reinterpret_cast<uint32_t *>(&r);
}

constexpr uint32_t kBias8 = 0x64806480u;   // half2(1152): byte q ^ 0x80 = q + 128
constexpr uint32_t kBias4 = 0x64086408u;   // half2(1032): nibble u -> u - 8

// K A-fragment values of one key row for block b: h[0], h[1] feed k-slice 0
// (columns 2t..2t+1 and 2t+8..2t+9), h[2], h[3] k-slice 1.  `seg` is 8-byte
// aligned; the loads are as wide as each block's code offset allows.
template <int KT>
__device__ __forceinline__ void k_codes(const uint8_t *seg, int b, int t, uint32_t (&h)[4])
{
    if constexpr (KT == SKV_Q8_0) {
        // codes 8t .. 8t+7 of the block start at byte 34b + 2 + 8t, which is
        // 2, 4, 6, 0 mod 8 for b = 0..3
        const uint8_t *p = seg + 34 * b + 2 + 8 * t;
        if (b == 3) {
            const uint2 w = *reinterpret_cast<const uint2 *>(p);
            const uint32_t w0 = w.x ^ 0x80808080u, w1 = w.y ^ 0x80808080u;
            h[0] = to_h2<0x4140>(w0, kBias8);
            h[1] = to_h2<0x4342>(w0, kBias8);
            h[2] = to_h2<0x4140>(w1, kBias8);
            h[3] = to_h2<0x4342>(w1, kBias8);
        } else if (b == 1) {
            const uint32_t w0 = *reinterpret_cast<const uint32_t *>(p) ^ 0x80808080u;
            const uint32_t w1 = *reinterpret_cast<const uint32_t *>(p + 4) ^ 0x80808080u;
            h[0] = to_h2<0x4140>(w0, kBias8);
            h[1] = to_h2<0x4342>(w0, kBias8);
            h[2] = to_h2<0x4140>(w1, kBias8);
            h[3] = to_h2<0x4342>(w1, kBias8);
        } else {                                                  // 2 mod 4: three aligned words
            const uint32_t *q = reinterpret_cast<const uint32_t *>(p - 2);
            const uint32_t w0 = q[0] ^ 0x80808080u, w1 = q[1] ^ 0x80808080u, w2 = q[2] ^ 0x80808080u;
            h[0] = to_h2<0x4342>(w0, kBias8);
            h[1] = to_h2<0x4140>(w1, kBias8);
            h[2] = to_h2<0x4342>(w1, kBias8);
            h[3] = to_h2<0x4140>(w2, kBias8);
        }
    } else {
        // bytes 4t .. 4t+3 of the block start at 18b + 2 + 4t: 2, 0, 2, 0 mod 4
        const uint8_t *p = seg + 18 * b + 2 + 4 * t;
        uint32_t w;                                               // the four code bytes
        if (b & 1) {
            w = *reinterpret_cast<const uint32_t *>(p);
        } else {
            const uint32_t *q = reinterpret_cast<const uint32_t *>(p - 2);
            w = __byte_perm(q[0], q[1], 0x5432);
        }
        const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
        h[0] = to_h2<0x4140>(lo, kBias4);                         // values 4t, 4t+1
        h[1] = to_h2<0x4342>(lo, kBias4);                         // values 4t+2, 4t+3
        h[2] = to_h2<0x4140>(hi, kBias4);                         // values 16+4t, 16+4t+1
        h[3] = to_h2<0x4342>(hi, kBias4);                         // values 16+4t+2, 16+4t+3
    }
}

// Query B-fragment for block b in the permuted order of k_codes<KT>.
template <int KT>
__device__ __forceinline__ void q_frag(const __half *qrow, int b, int t, uint32_t (&f)[4])
{
    if constexpr (KT == SKV_Q8_0) {
        const uint4 v = *reinterpret_cast<const uint4 *>(qrow + 32 * b + 8 * t);
        f[0] = v.x;
        f[1] = v.y;
        f[2] = v.z;
        f[3] = v.w;
    } else {
        const uint2 lo = *reinterpret_cast<const uint2 *>(qrow + 32 * b + 4 * t);
        const uint2 hi = *reinterpret_cast<const uint2 *>(qrow + 32 * b + 16 + 4 * t);
        f[0] = lo.x;
        f[1] = lo.y;
        f[2] = hi.x;
        f[3] = hi.y;
    }
}

template <int KT, int VT>
__global__ void __launch_bounds__(256) splitkv_decode_rows_kernel(const DecodeArgs a)
{
    constexpr int SEGK = QB<KT>::seg;
    constexpr int SEGV = QB<VT>::seg;
    constexpr int BLKV = QB<VT>::blk;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[kRStages];
    __shared__ int s_abort;
    __shared__ int s_done[kRStages];             // warps finished with the stage's current tile
    __shared__ int s_issued;                     // tiles issued so far

    const int tid = threadIdx.x;
    const int kh = tid >> 5;                     // warp = KV head
    const int lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int cg = blockIdx.x;
    const int split = blockIdx.y;
    const int s = blockIdx.z;
    const int64_t j_lo = a.key_lo + static_cast<int64_t>(split) * a.split_len;
    const int64_t j_hi = min(a.n_local, j_lo + a.split_len);
    const int n_tiles = j_hi > j_lo ? static_cast<int>((j_hi - j_lo + kRRows - 1) / kRRows) : 0;
    const int64_t krb = a.k_row_bytes, vrb = a.v_row_bytes;
    // Rows land in 2-row chunks separated by a pad that shifts consecutive
    // chunks by 8 banks, so the 8 key rows one instruction reads sit on
    // different banks.
    const uint32_t chunk_k = static_cast<uint32_t>(2 * krb) + chunk_pad(krb);
    const uint32_t chunk_v = static_cast<uint32_t>(2 * vrb) + chunk_pad(vrb);
    const uint32_t stage_k = (kRRows / 2) * chunk_k;
    const uint32_t stage_bytes = stage_k + (kRRows / 2) * chunk_v;
    auto krow = [&](int r) { return (r >> 1) * chunk_k + (r & 1) * static_cast<uint32_t>(krb); };
    auto vrow = [&](int r) { return (r >> 1) * chunk_v + (r & 1) * static_cast<uint32_t>(vrb); };
    const uint32_t sbase = smem_addr(smem);
    auto bar = [&](int st) { return smem_addr(&full_bar[st]); };

    if (tid == 0) {
        s_abort = 0;
        s_issued = 0;
        for (int i = 0; i < kRStages; ++i) {
            tc::mbar_init(bar(i), 1);
            s_done[i] = 0;
        }
        tc::fence_barrier_init();
    }
    __syncthreads();

    // One warp issues a stage: lane l < 16 copies K rows 2l, 2l+1 of keys
    // [j_lo + 32 tile, ...) (all heads), lane 16 + l the same V rows.  The
    // first stages are issued by warp 0; afterwards the last warp to finish
    // with a stage refills it, so no warp waits for the others.
    auto issue = [&](int tile) {
        if (lane == 0) s_issued = tile + 1;
        const int st = tile % kRStages;
        const int64_t k0 = j_lo + static_cast<int64_t>(tile) * kRRows;
        const int rows = static_cast<int>(min(j_hi - k0, static_cast<int64_t>(kRRows)));
        if (lane == 0)
            tc::mbar_expect_tx(bar(st), static_cast<uint32_t>(rows * (krb + vrb)));
        __syncwarp();
        const int c = lane & 15;
        const int n = min(2, rows - 2 * c);
        if (n > 0) {
            const int64_t r = a.row0 + k0 + 2 * c;
            if (lane < 16)
                tc::bulk_load(sbase + st * stage_bytes + c * chunk_k, a.k + r * krb, static_cast<uint32_t>(n * krb),
                              bar(st));
            else
                tc::bulk_load(sbase + st * stage_bytes + stage_k + c * chunk_v, a.v + r * vrb,
                              static_cast<uint32_t>(n * vrb), bar(st));
        }
    };
    if (tid < 32)
        for (int p = 0; p < kRStages && p < n_tiles; ++p) issue(p);

    // This warp's columns: column n = g of the query fragment; the thread's
    // accumulator columns 2t, 2t+1.
    const bool head_ok = true;                   // one warp per KV head: blockDim = 32 * Hk
    uint32_t qf[4][4];
    {
        const int c = cg * 8 + g;
        const int tq = c / a.G;
        const bool ok = head_ok && tq < a.nq;
        const __half *qrow = a.q + ((static_cast<int64_t>(s) * a.nq + (ok ? tq : 0)) * a.H +
                                    (head_ok ? kh : 0) * a.G + c % a.G) * kRD;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            if (ok) q_frag<KT>(qrow, b, t, qf[b]);
            else qf[b][0] = qf[b][1] = qf[b][2] = qf[b][3] = 0u;
        }
    }
    int32_t col_pos[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int c = cg * 8 + 2 * t + e;
        const int tq = c / a.G;
        col_pos[e] = a.q_pos ? a.q_pos[static_cast<int64_t>(s) * a.nq + (tq < a.nq ? tq : 0)] : 0;
    }

    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};

    __syncwarp();
    for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kRStages;
        bool ok = !*reinterpret_cast<volatile int *>(&s_abort) &&
                  tc::mbar_wait(bar(st), (i / kRStages) & 1, a.status);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) {
                s_abort = 1;
                atomicOr(a.status, 1);
            }
            break;
        }
        {
            const uint8_t *sk = smem + st * stage_bytes + kh * SEGK;
            const uint8_t *sv = smem + st * stage_bytes + stage_k + kh * SEGV;
            const int64_t key0 = j_lo + static_cast<int64_t>(i) * kRRows;    // local index of stage row 0
            // ---- S^T = K Q^T for the stage's two 16-key m-tiles ----
            float x[2][4];
#pragma unroll
            for (int mh = 0; mh < 2; ++mh) {
                const uint8_t *kg = sk + krow(mh * 16 + g);
                const uint8_t *kg8 = sk + krow(mh * 16 + g + 8);
                float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    uint32_t hg[4], hg8[4];
                    k_codes<KT>(kg, b, t, hg);
                    k_codes<KT>(kg8, b, t, hg8);
                    float tb[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_16816(tb, hg[0], hg8[0], hg[1], hg8[1], qf[b][0], qf[b][1]);
                    mma_16816(tb, hg[2], hg8[2], hg[3], hg8[3], qf[b][2], qf[b][3]);
                    const float d0 = __half2float(__ushort_as_half(static_cast<unsigned short>(ld_s16(kg + QB<KT>::blk * b))));
                    const float d1 = __half2float(__ushort_as_half(static_cast<unsigned short>(ld_s16(kg8 + QB<KT>::blk * b))));
                    sacc[0] = fmaf(d0, tb[0], sacc[0]);
                    sacc[1] = fmaf(d0, tb[1], sacc[1]);
                    sacc[2] = fmaf(d1, tb[2], sacc[2]);
                    sacc[3] = fmaf(d1, tb[3], sacc[3]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int64_t j = key0 + mh * 16 + g + ((e >> 1) << 3);
                    float val = sacc[e] * a.scale_log2;
                    if (j >= j_hi) val = -INFINITY;
                    if (a.q_pos && a.key_pos0 + a.logical0 + j > col_pos[e & 1]) val = -INFINITY;
                    x[mh][e] = val;
                }
            }
            // ---- online softmax per column ----
            float mx0 = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
            float mx1 = fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3]));
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
            const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
            const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = fast_exp2(m_run[0] - ref0), al1 = fast_exp2(m_run[1] - ref1);
            float p[2][4];
#pragma unroll
            for (int mh = 0; mh < 2; ++mh) {
                p[mh][0] = fast_exp2(x[mh][0] - ref0);
                p[mh][1] = fast_exp2(x[mh][1] - ref1);
                p[mh][2] = fast_exp2(x[mh][2] - ref0);
                p[mh][3] = fast_exp2(x[mh][3] - ref1);
            }
            l_run[0] = l_run[0] * al0 + (p[0][0] + p[0][2]) + (p[1][0] + p[1][2]);
            l_run[1] = l_run[1] * al1 + (p[0][1] + p[0][3]) + (p[1][1] + p[1][3]);
            m_run[0] = mn0;
            m_run[1] = mn1;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
            // ---- O^T += V^T P^T, one 16-key k-slice per m-tile of keys ----
#pragma unroll
            for (int mh = 0; mh < 2; ++mh) {
                const uint8_t *vg = sv + vrow(mh * 16 + g);              // this thread's P rows: keys g, g+8
                const uint8_t *vg8 = sv + vrow(mh * 16 + g + 8);
                const bool ok0 = key0 + mh * 16 + g < j_hi, ok1 = key0 + mh * 16 + g + 8 < j_hi;
                const uint8_t *va = sv + vrow(mh * 16 + 2 * t);          // A-fragment keys 2t, 2t+1, 2t+8, 2t+9
                const uint8_t *vb = sv + vrow(mh * 16 + 2 * t + 1);
                const uint8_t *vc = sv + vrow(mh * 16 + 2 * t + 8);
                const uint8_t *vd = sv + vrow(mh * 16 + 2 * t + 9);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const float d0 = ok0 ? __half2float(__ushort_as_half(static_cast<unsigned short>(ld_s16(vg + BLKV * b)))) : 0.f;
                    const float d1 = ok1 ? __half2float(__ushort_as_half(static_cast<unsigned short>(ld_s16(vg8 + BLKV * b)))) : 0.f;
                    const uint32_t pb0 = movmatrix_trans(pack_half2(p[mh][0] * d0, p[mh][1] * d0));
                    const uint32_t pb1 = movmatrix_trans(pack_half2(p[mh][2] * d1, p[mh][3] * d1));
                    // m-tile 2b: output dims 32b + 2g (row g), 32b + 2g + 1 (row g+8);
                    // m-tile 2b+1: the same plus 16.
                    uint32_t x01[2], x89[2];
                    if constexpr (VT == SKV_Q4_0) {
                        const int off = 18 * b + 2 + 2 * g;                   // bytes 2g, 2g+1
                        const uint32_t w01 = __byte_perm(ld_s16(va + off), ld_s16(vb + off), 0x5140);
                        const uint32_t w89 = __byte_perm(ld_s16(vc + off), ld_s16(vd + off), 0x5140);
                        x01[0] = w01 & 0x0F0F0F0Fu;
                        x89[0] = w89 & 0x0F0F0F0Fu;
                        x01[1] = (w01 >> 4) & 0x0F0F0F0Fu;
                        x89[1] = (w89 >> 4) & 0x0F0F0F0Fu;
                    } else {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int off = 34 * b + 2 + 16 * hh + 2 * g;      // values 16hh + 2g, +1
                            x01[hh] = __byte_perm(ld_s16(va + off), ld_s16(vb + off), 0x5140) ^ 0x80808080u;
                            x89[hh] = __byte_perm(ld_s16(vc + off), ld_s16(vd + off), 0x5140) ^ 0x80808080u;
                        }
                    }
                    constexpr uint32_t bias = VT == SKV_Q4_0 ? kBias4 : kBias8;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
                        mma_16816(o[2 * b + hh], to_h2<0x4140>(x01[hh], bias), to_h2<0x4342>(x01[hh], bias),
                                  to_h2<0x4140>(x89[hh], bias), to_h2<0x4342>(x89[hh], bias), pb0, pb1);
                }
            }
        }
        // The last warp done with stage st refills it with tile i + kRStages.
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&s_done[st], 1) == a.Hk - 1;
            if (last) s_done[st] = 0;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last && i + kRStages < n_tiles) {
            tc::fence_proxy_async_smem();        // our reads of the stage before the copy's writes
            issue(i + kRStages);
        }
    }
    __syncthreads();
    if (*reinterpret_cast<volatile int *>(&s_abort) && tid == 0) {
        // drain: every issued copy must land before the CTA exits
        const int issued = s_issued;
        for (int j = max(0, issued - kRStages); j < issued; ++j)
            tc::mbar_wait(bar(j % kRStages), (j / kRStages) & 1, nullptr, 100000000ull);
    }

    // The combine that merges the splits may be scheduled from here on (it
    // waits for this whole grid before reading).
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    // ---- normalised partial O (this warp's head, 8 columns) and lse ----
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
    }
    const bool direct = a.n_splits == 1;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int c = cg * 8 + 2 * t + e;
        const int tq = c / a.G;
        if (tq >= a.nq) continue;
        const int64_t r = (static_cast<int64_t>(s) * a.nq + tq) * a.H + kh * a.G + c % a.G;
        float *op = direct ? a.o_out + r * kRD : a.o_split + (static_cast<int64_t>(split) * a.R + r) * kRD;
        float *lp = direct ? a.lse_out + r : a.lse_split + static_cast<int64_t>(split) * a.R + r;
        const bool empty = m_run[e] == -INFINITY || l_run[e] <= 0.f;
        const float inv = empty ? 0.f : 1.f / l_run[e];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int dim = 32 * (mt >> 1) + 16 * (mt & 1) + 2 * g;
            *reinterpret_cast<float2 *>(op + dim) = make_float2(o[mt][e] * inv, o[mt][2 + e] * inv);
        }
        if (g == 0) *lp = empty ? -INFINITY : (m_run[e] + __log2f(l_run[e])) * 0.6931471805599453f;
    }
}

template <int KT, int VT>
KernelAttrCache &rows_attr_cache()
{
    static KernelAttrCache c;
    return c;
}

template <int KT, int VT>
int launch_rows_t(skv_handle *h, const DecodeArgs &a, cudaStream_t st)
{
    const int smem = kRStages * static_cast<int>(rows_stage_bytes(a.k_row_bytes, a.v_row_bytes));
    cudaError_t e = kernel_smem_optin(rows_attr_cache<KT, VT>(),
                                      reinterpret_cast<const void *>(splitkv_decode_rows_kernel<KT, VT>), smem,
                                      32 * a.Hk, nullptr);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute(decode rows)");
    dim3 grid(static_cast<unsigned>(a.n_cg), static_cast<unsigned>(a.n_splits), static_cast<unsigned>(a.S));
    if (h->prof_before) cudaEventRecord(h->prof_before, st);
    splitkv_decode_rows_kernel<KT, VT><<<grid, 32 * a.Hk, smem, st>>>(a);
    if (h->prof_after) cudaEventRecord(h->prof_after, st);
    return cuda_fail(h, cudaGetLastError(), "decode rows kernel launch");
}

template <int KT, int VT>
int rows_ctas_t(int smem, int threads)
{
    int n = 0;
    if (kernel_smem_optin(rows_attr_cache<KT, VT>(), reinterpret_cast<const void *>(splitkv_decode_rows_kernel<KT, VT>),
                          smem, threads, &n) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace

bool decode_rows_eligible(const skv_shape *sh, const void *k, const void *v, const void *mask)
{
    const bool qk = sh->k_type == SKV_Q8_0 || sh->k_type == SKV_Q4_0;
    const bool qv = sh->v_type == SKV_Q8_0 || sh->v_type == SKV_Q4_0;
    const int64_t smem = kRStages * rows_stage_bytes(sh->k_row_bytes, sh->v_row_bytes);
    return qk && qv && sh->D == kRD && mask == nullptr && sh->Hk >= 1 && sh->Hk <= 8 && sh->k_row_bytes % 16 == 0 &&
           sh->v_row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(k) % 16) == 0 &&
           (reinterpret_cast<uintptr_t>(v) % 16) == 0 && smem <= 200 * 1024;
}

int decode_rows_ctas_per_sm(const skv_shape *sh)
{
    const int smem = kRStages * static_cast<int>(rows_stage_bytes(sh->k_row_bytes, sh->v_row_bytes));
    const int kt = sh->k_type, vt = sh->v_type, th = 32 * sh->Hk;
    if (kt == SKV_Q8_0 && vt == SKV_Q8_0) return rows_ctas_t<SKV_Q8_0, SKV_Q8_0>(smem, th);
    if (kt == SKV_Q8_0 && vt == SKV_Q4_0) return rows_ctas_t<SKV_Q8_0, SKV_Q4_0>(smem, th);
    if (kt == SKV_Q4_0 && vt == SKV_Q8_0) return rows_ctas_t<SKV_Q4_0, SKV_Q8_0>(smem, th);
    if (kt == SKV_Q4_0 && vt == SKV_Q4_0) return rows_ctas_t<SKV_Q4_0, SKV_Q4_0>(smem, th);
    return 0;
}

int launch_decode_rows(skv_handle *h, const DecodeArgs &a, int kt, int vt, cudaStream_t st)
{
    if (a.n_cg > 65535 || a.n_splits > 65535 || a.S > 65535)
        return fail(h, SKV_EUNSUPPORTED, "grid too large: n_cg=%d splits=%d S=%d", a.n_cg, a.n_splits, a.S);
    DecodeArgs b = a;
    b.status = h->status;
    int rc = SKV_OK;
    if (kt == SKV_Q8_0 && vt == SKV_Q8_0) rc = launch_rows_t<SKV_Q8_0, SKV_Q8_0>(h, b, st);
    else if (kt == SKV_Q8_0 && vt == SKV_Q4_0) rc = launch_rows_t<SKV_Q8_0, SKV_Q4_0>(h, b, st);
    else if (kt == SKV_Q4_0 && vt == SKV_Q8_0) rc = launch_rows_t<SKV_Q4_0, SKV_Q8_0>(h, b, st);
    else if (kt == SKV_Q4_0 && vt == SKV_Q4_0) rc = launch_rows_t<SKV_Q4_0, SKV_Q4_0>(h, b, st);
    else return fail(h, SKV_EUNSUPPORTED, "no dense-row decode kernel for K type %d / V type %d", kt, vt);
    if (rc || a.n_splits == 1) return rc;
    // merge the launch's splits (log-sum-exp combine) into its output
    rc = launch_combine(a.n_splits, a.o_split, a.lse_split, a.R, kRD, a.o_out, a.lse_out, st);
    return rc == SKV_OK ? rc : cuda_fail(h, cudaGetLastError(), "combine launch");
}

}  // namespace skv
