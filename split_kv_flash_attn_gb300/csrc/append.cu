// append.cu -- writing new KV rows into a cell-major cache of two regions (a
// device window and a page-locked host tail), converting fp32 values to fp16
// or quantising them to q8_0 / q4_0 on the way.
//
// Write routing follows the rolling-KV page (Rolling KV, "what ships": the
// K/V copies split into a window prefix [0, wc) and a host suffix [wc, n)):
// position p goes to window row p when p < n_rows0, else to tail row p - n_rows0.
//
// Quantisation of one 32-value block, in fp32 as on the Strata KV-streaming
// page (kv_append_q8 kernel: scale = amax / 127 kept as fp16, code = nearest
// integer of x / scale, clamped to +-127):
//   q8_0: d = fp16(amax / 127); q = rint(x / d) clamped to [-127, 127];
//   q4_0: d = fp16(amax / 7);   u = rint(x / d) + 8 clamped to [0, 15]
//         (the pages give no q4_0 quantiser; this reading keeps the same
//         nearest-code rule with the 4-bit range);
//   amax = 0 gives d = 0 and all codes at value zero.
// The block here is q8_0's 32 values (the page groups 64 values per scale;
// the cache rows use the q8_0 block).  x / d is divided by the STORED fp16
// scale, so d*q is the code nearest x.
//
// Both divisions are replaced by products with a reciprocal, with the exact
// division kept for the few values where the two could decide differently:
//  * the code: rd = rcp.approx(d) has a relative error of at most 2^-22, so
//    t0 = x * rd lies within 2^-21.6 |t0| of x/d (5e-5 for |x/d| < 130), and
//    the fp32 quotient fl(x/d) within 2^-17 of x/d; so when t0 is more than
//    2^-13 (1.2e-4) away from every half-integer, rint(t0) = rint(fl(x/d)).
//    Nearer than that (about 1 value in 4000, and every exact tie), the
//    codes are taken from the IEEE division itself.  With a normal fp16
//    scale |x/d| < qmax + 0.5, so only a subnormal scale needs the clamp, and
//    for it (d < 2^-14) a large |t0| rounds far from any half-integer and
//    clamps the same either way.
//  * the scale: s0 = amax * fl(1/qmax) lies within 2^-22.4 (relative) of
//    fl(amax/qmax); when s0 (1 - 2^-20) and s0 (1 + 2^-20) round to the same
//    fp16 value, so does fl(amax/qmax) (rounding is monotone); otherwise the
//    scale comes from the IEEE division.
// The stored bytes are therefore those of the plain fp32 rule, bit for bit.
#include "internal.h"

namespace skv {

__device__ __forceinline__ uint32_t pack_half2(float a, float b)
{
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// fp16(fl(amax / qmax)) without a division unless the product could round
// to another fp16 value (see the header).
__device__ __forceinline__ __half block_scale(float amax, float qmax, float inv_qmax)
{
    const float s0 = __fmul_rn(amax, inv_qmax);
    const __half h = __float2half_rn(s0);
    const __half lo = __float2half_rn(__fmul_rn(s0, 1.f - 0x1p-20f));
    const __half hi = __float2half_rn(__fmul_rn(s0, 1.f + 0x1p-20f));
    if (__half_as_ushort(lo) == __half_as_ushort(h) && __half_as_ushort(hi) == __half_as_ushort(h)) return h;
    return __float2half_rn(__fdiv_rn(amax, qmax));
}

// 1/d to within 2^-22 (relative), one instruction; d is a normal fp32 value.
__device__ __forceinline__ float rcp_approx(float d)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// Bytes 0 of four words, in order, as one word.
__device__ __forceinline__ uint32_t low_bytes4(uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Each warp takes kItemsPerWarp consecutive (row, head) items: it loads all of
// their values first, then converts and stores, so a warp keeps several loads
// in flight.  Positions outside [0, n_rows0 + n_rows1) are skipped; a
// non-negative one also sets bit 1 of *status.  The fp16 kernel gives each
// lane D/32 values of an item.
constexpr int kItemsPerWarp = 4;
constexpr int kAppendThreads = 256;

template <bool VEC8, int DD>
__global__ void __launch_bounds__(kAppendThreads) kv_append_f16_kernel(const float *__restrict__ x,
                                                                       const int32_t *__restrict__ pos, int n, int Hk,
                                                                       int64_t row_bytes, uint8_t *dst0,
                                                                       int64_t n_rows0, uint8_t *dst1,
                                                                       int64_t n_rows1, int *status)
{
    constexpr int VPL = DD / 32;                                  // values per lane per item
    const int lane = threadIdx.x & 31;
    const int64_t total = static_cast<int64_t>(n) * Hk;
    const int64_t first =
        (static_cast<int64_t>(blockIdx.x) * (kAppendThreads / 32) + (threadIdx.x >> 5)) * kItemsPerWarp;
    float v[kItemsPerWarp][VPL];
    int64_t p[kItemsPerWarp];
    int hd[kItemsPerWarp];                                        // KV head of each item
    // (row, head) of the warp's first item with one division; the next items
    // step through the heads.
    const int64_t row_first = first / Hk;
    {
        int hh = static_cast<int>(first - row_first * Hk);
#pragma unroll
        for (int it = 0; it < kItemsPerWarp; ++it) {
            hd[it] = hh;
            hh = hh + 1 == Hk ? 0 : hh + 1;
        }
    }
#pragma unroll
    for (int it = 0; it < kItemsPerWarp; ++it) {
        const int64_t item = first + it;
        p[it] = -1;
        if (item >= total) continue;
        int64_t row = row_first;
#pragma unroll
        for (int u = 1; u <= it; ++u) row += hd[u] == 0 ? 1 : 0;   // a head wrap starts the next row
        p[it] = pos[row];
        const float *src = x + item * DD;                         // values lane*VPL .. lane*VPL + VPL - 1
        if (VPL == 4) {
            const float4 a = reinterpret_cast<const float4 *>(src)[lane];
            v[it][0] = a.x; v[it][1] = a.y; v[it][2] = a.z; v[it][3] = a.w;
        } else {
            const float2 a = reinterpret_cast<const float2 *>(src)[lane];
            v[it][0] = a.x; v[it][1] = a.y;
        }
    }
#pragma unroll
    for (int it = 0; it < kItemsPerWarp; ++it) {
        const int64_t item = first + it;
        if (p[it] < 0) continue;                                  // beyond the items, or not written
        const int h = hd[it];
        if (p[it] >= n_rows0 + n_rows1) {
            if (lane == 0 && h == 0) atomicOr(status, 2);
            continue;
        }
        uint8_t *row = p[it] < n_rows0 ? dst0 + p[it] * row_bytes : dst1 + (p[it] - n_rows0) * row_bytes;
        uint8_t *out = row + static_cast<int64_t>(h) * DD * 2 + lane * VPL * 2;
        if (VPL == 4) {
            const uint32_t w0 = pack_half2(v[it][0], v[it][1]), w1 = pack_half2(v[it][2], v[it][3]);
            if (VEC8) {
                *reinterpret_cast<uint2 *>(out) = make_uint2(w0, w1);
            } else {
                reinterpret_cast<uint32_t *>(out)[0] = w0;        // rows are 4-byte aligned
                reinterpret_cast<uint32_t *>(out)[1] = w1;
            }
        } else {
            *reinterpret_cast<uint32_t *>(out) = pack_half2(v[it][0], v[it][1]);
        }
    }
}

// Quantising append with eight values a lane: LPI = D / 8 lanes per (row,
// head) item and four lanes per 32-value block, so 32 / LPI items share each
// warp instruction and the per-block work (maximum, scale, reciprocal) and the
// per-item work (position, destination) are spread over eight values.  Each
// warp takes kItemsPerWarp consecutive items; all their values are loaded
// before any is converted.  The codes are decided as described at the top.
template <int T, int DD>
__global__ void __launch_bounds__(kAppendThreads) kv_append_quant_kernel(const float *__restrict__ x,
                                                                         const int32_t *__restrict__ pos, int n,
                                                                         int Hk, int64_t row_bytes, uint8_t *dst0,
                                                                         int64_t n_rows0, uint8_t *dst1,
                                                                         int64_t n_rows1, int *status)
{
    constexpr int LPI = DD / 8;                                   // lanes per item
    constexpr int IPS = 32 / LPI;                                 // items per warp step
    constexpr int STEPS = kItemsPerWarp / IPS;
    static_assert(STEPS * IPS == kItemsPerWarp, "items per warp");
    constexpr int BLK = T == SKV_Q8_0 ? 34 : 18;
    constexpr float QMAX = T == SKV_Q8_0 ? 127.f : 7.f;
    constexpr float INV_QMAX = 1.f / QMAX;
    const int lane = threadIdx.x & 31;
    const int l = lane % LPI;                                     // lane within its item
    const int b = l >> 2, j0 = (l & 3) * 8;                       // block, first value of the lane
    const int64_t total = static_cast<int64_t>(n) * Hk;
    const int64_t first =
        (static_cast<int64_t>(blockIdx.x) * (kAppendThreads / 32) + (threadIdx.x >> 5)) * kItemsPerWarp;
    // (row, head) of the warp's first item with one division; the lane's items
    // first + s * IPS + lane / LPI step through the heads from there.
    const int64_t row_first = first / Hk;
    const int h_first = static_cast<int>(first - row_first * Hk);
    float v[STEPS][8];
    int64_t p[STEPS];
    int hd[STEPS];
#pragma unroll
    for (int s = 0; s < STEPS; ++s) {
        const int o = s * IPS + lane / LPI;                       // item offset within the warp, < kItemsPerWarp
        int hh = h_first;
        int64_t row = row_first;
#pragma unroll
        for (int k = 0; k < kItemsPerWarp - 1; ++k) {
            if (k < o) {
                if (++hh == Hk) {
                    hh = 0;
                    ++row;
                }
            }
        }
        hd[s] = hh;
        const int64_t item = first + o;
        p[s] = -1;
        if (item < total) {
            p[s] = pos[row];
            const float4 *src = reinterpret_cast<const float4 *>(x + item * DD) + 2 * l;
            const float4 a0 = src[0], a1 = src[1];
            v[s][0] = a0.x; v[s][1] = a0.y; v[s][2] = a0.z; v[s][3] = a0.w;
            v[s][4] = a1.x; v[s][5] = a1.y; v[s][6] = a1.z; v[s][7] = a1.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[s][i] = 0.f;
        }
    }
#pragma unroll
    for (int s = 0; s < STEPS; ++s) {
        // every lane takes part in the block's shuffles; only valid items store
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[s][i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const __half d16 = block_scale(amax, QMAX, INV_QMAX);
        const float d = __half2float(d16);
        const float rd = d > 0.f ? rcp_approx(d) : 0.f;           // d = 0: every code 0
        int q[8];
        float off = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float t0 = __fmul_rn(v[s][i], rd);
            const float r0 = rintf(t0);
            off = fmaxf(off, fabsf(t0 - r0));
            q[i] = static_cast<int>(r0);
        }
        if (off >= 0.5f - 0x1p-13f) {
#pragma unroll
            for (int i = 0; i < 8; ++i) q[i] = __float2int_rn(__fdiv_rn(v[s][i], d));
        }
        if (d < 0x1p-14f) {
            constexpr int QLO = T == SKV_Q8_0 ? -127 : -8, QHI = T == SKV_Q8_0 ? 127 : 7;   // codes -127..127, 0..15
#pragma unroll
            for (int i = 0; i < 8; ++i) q[i] = max(QLO, min(QHI, q[i]));
        }
        uint32_t c[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = static_cast<uint32_t>(T == SKV_Q8_0 ? q[i] : q[i] + 8);
        uint32_t w0 = low_bytes4(c[0], c[1], c[2], c[3]), w1 = low_bytes4(c[4], c[5], c[6], c[7]);
        if (T == SKV_Q4_0) {
            // byte j holds value j (low nibble) and value j + 16 (high nibble):
            // the lane two further on holds values j0 + 16 ..
            const uint32_t h0 = __shfl_down_sync(0xffffffffu, w0, 2), h1 = __shfl_down_sync(0xffffffffu, w1, 2);
            w0 |= h0 << 4;
            w1 |= h1 << 4;
        }
        const int64_t ps = p[s];
        if (ps < 0) continue;                                     // beyond the items, or not written
        const int h = hd[s];
        if (ps >= n_rows0 + n_rows1) {
            if (l == 0 && h == 0) atomicOr(status, 2);
            continue;
        }
        uint8_t *row = ps < n_rows0 ? dst0 + ps * row_bytes : dst1 + (ps - n_rows0) * row_bytes;
        uint8_t *blk = row + static_cast<int64_t>(h) * (DD / 32) * BLK + b * BLK;   // 2-byte aligned
        if (T == SKV_Q8_0 || j0 < 16) {
            uint16_t *dst = reinterpret_cast<uint16_t *>(blk + 2 + j0);
            dst[0] = static_cast<uint16_t>(w0);
            dst[1] = static_cast<uint16_t>(w0 >> 16);
            dst[2] = static_cast<uint16_t>(w1);
            dst[3] = static_cast<uint16_t>(w1 >> 16);
        }
        if (j0 == 0) *reinterpret_cast<__half *>(blk) = d16;
    }
}

// A device-accessible address for a destination region: device memory as is,
// page-locked host memory through its mapped device address.
static int device_address(skv_handle *h, void *p, uint8_t **out)
{
    *out = nullptr;
    if (!p) return SKV_OK;
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess || at.type == cudaMemoryTypeUnregistered) {
        cudaGetLastError();
        return fail(h, SKV_ENOTPINNED, "append destination %p is neither device nor page-locked host memory", p);
    }
    if (at.type == cudaMemoryTypeHost && !at.devicePointer)
        return fail(h, SKV_ENOTPINNED, "append destination %p is page-locked but not device-mapped", p);
    *out = static_cast<uint8_t *>(at.type == cudaMemoryTypeHost ? at.devicePointer : p);
    return SKV_OK;
}

}  // namespace skv

using namespace skv;

extern "C" int skv_kv_append(skv_handle *h, int32_t type, int32_t Hk, int32_t D, int64_t row_bytes, const float *x,
                             const int32_t *positions, int32_t n, void *dst0, int64_t n_rows0, void *dst1,
                             int64_t n_rows1, void *stream)
{
    if (!h) return SKV_EINVAL;
    h->err[0] = 0;
    if (n < 0 || Hk <= 0 || (D != 64 && D != 128) || n_rows0 < 0 || n_rows1 < 0)
        return fail(h, SKV_EINVAL, "bad sizes (n=%d Hk=%d D=%d rows %lld + %lld)", n, Hk, D, (long long)n_rows0,
                    (long long)n_rows1);
    if (segment_bytes(type, D) < 0) return fail(h, SKV_EINVAL, "unknown element type %d", type);
    if (row_bytes < Hk * segment_bytes(type, D)) return fail(h, SKV_EINVAL, "row stride smaller than Hk segments");
    if ((n_rows0 > 0 && !dst0) || (n_rows1 > 0 && !dst1)) return fail(h, SKV_EINVAL, "NULL destination region");
    if (n == 0) return SKV_OK;
    if (!x || !positions) return fail(h, SKV_EINVAL, "NULL pointer");
    if (reinterpret_cast<uintptr_t>(x) % 16) return fail(h, SKV_EUNSUPPORTED, "x must be 16-byte aligned");
    uint8_t *d0 = nullptr, *d1 = nullptr;
    int rc = device_address(h, n_rows0 > 0 ? dst0 : nullptr, &d0);
    if (!rc) rc = device_address(h, n_rows1 > 0 ? dst1 : nullptr, &d1);
    if (rc) return rc;
    const int align = type == SKV_F16 ? 4 : 2;
    if (row_bytes % align || reinterpret_cast<uintptr_t>(d0) % align || reinterpret_cast<uintptr_t>(d1) % align)
        return fail(h, SKV_EUNSUPPORTED, "destination base and row stride must be %d-byte aligned", align);
    const bool vec8 = row_bytes % 8 == 0 && reinterpret_cast<uintptr_t>(d0) % 8 == 0 &&
                      reinterpret_cast<uintptr_t>(d1) % 8 == 0;
    const int64_t items = static_cast<int64_t>(n) * Hk;
    const int64_t per_block = static_cast<int64_t>(kAppendThreads / 32) * kItemsPerWarp;
    if ((items + per_block - 1) / per_block > 0x7fffffffLL)
        return fail(h, SKV_EUNSUPPORTED, "too many rows for one launch");
    const unsigned grid = static_cast<unsigned>((items + per_block - 1) / per_block);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
#define SKV_APPEND(V, DDD)                                                                                    \
    kv_append_f16_kernel<V, DDD><<<grid, kAppendThreads, 0, st>>>(x, positions, n, Hk, row_bytes, d0, n_rows0, d1, \
                                                                  n_rows1, h->status)
    if (type == SKV_F16) {
        if (vec8) {
            if (D == 64) SKV_APPEND(true, 64);
            else SKV_APPEND(true, 128);
        } else {
            if (D == 64) SKV_APPEND(false, 64);
            else SKV_APPEND(false, 128);
        }
    } else {
#define SKV_APPEND_Q(TT, DDD)                                                                              \
    kv_append_quant_kernel<TT, DDD><<<grid, kAppendThreads, 0, st>>>(x, positions, n, Hk, row_bytes, d0, \
                                                                     n_rows0, d1, n_rows1, h->status)
        if (type == SKV_Q8_0) {
            if (D == 64) SKV_APPEND_Q(SKV_Q8_0, 64);
            else SKV_APPEND_Q(SKV_Q8_0, 128);
        } else {
            if (D == 64) SKV_APPEND_Q(SKV_Q4_0, 64);
            else SKV_APPEND_Q(SKV_Q4_0, 128);
        }
#undef SKV_APPEND_Q
    }
#undef SKV_APPEND
    return cuda_fail(h, cudaGetLastError(), "append launch");
}
