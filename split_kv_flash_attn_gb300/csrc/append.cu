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
#include "internal.h"

namespace skv {

__device__ __forceinline__ float warp_max32(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b)
{
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Each warp takes kItemsPerWarp consecutive (row, head) items: it loads all of
// their values first (D/32 per lane each), then converts and stores, so a warp
// keeps several loads in flight.  Positions outside [0, n_rows0 + n_rows1) are
// skipped; a non-negative one also sets bit 1 of *status.
constexpr int kItemsPerWarp = 4;
constexpr int kAppendThreads = 256;

template <int T, bool VEC8, int DD>
__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(const float *__restrict__ x,
                                                                   const int32_t *__restrict__ pos, int n, int Hk,
                                                                   int64_t row_bytes, uint8_t *dst0, int64_t n_rows0,
                                                                   uint8_t *dst1, int64_t n_rows1, int *status)
{
    constexpr int VPL = DD / 32;                                  // values per lane per item
    const int lane = threadIdx.x & 31;
    const int64_t total = static_cast<int64_t>(n) * Hk;
    const int64_t first =
        (static_cast<int64_t>(blockIdx.x) * (kAppendThreads / 32) + (threadIdx.x >> 5)) * kItemsPerWarp;
    float v[kItemsPerWarp][VPL];
    int64_t p[kItemsPerWarp];
#pragma unroll
    for (int it = 0; it < kItemsPerWarp; ++it) {
        const int64_t item = first + it;
        p[it] = -1;
        if (item >= total) continue;
        p[it] = pos[item / Hk];
        const float *src = x + item * DD;
        if (T == SKV_F16) {                                       // values lane*VPL .. lane*VPL + VPL - 1
            if (VPL == 4) {
                const float4 a = reinterpret_cast<const float4 *>(src)[lane];
                v[it][0] = a.x; v[it][1] = a.y; v[it][2] = a.z; v[it][3] = a.w;
            } else {
                const float2 a = reinterpret_cast<const float2 *>(src)[lane];
                v[it][0] = a.x; v[it][1] = a.y;
            }
        } else {                                                  // value b*32 + lane of block b
#pragma unroll
            for (int b = 0; b < VPL; ++b) v[it][b] = src[b * 32 + lane];
        }
    }
#pragma unroll
    for (int it = 0; it < kItemsPerWarp; ++it) {
        const int64_t item = first + it;
        if (p[it] < 0) continue;                                  // beyond the items, or not written
        const int h = static_cast<int>(item % Hk);
        if (p[it] >= n_rows0 + n_rows1) {
            if (lane == 0 && h == 0) atomicOr(status, 2);
            continue;
        }
        uint8_t *row = p[it] < n_rows0 ? dst0 + p[it] * row_bytes : dst1 + (p[it] - n_rows0) * row_bytes;
        if constexpr (T == SKV_F16) {
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
        } else {
            constexpr int BLK = T == SKV_Q8_0 ? 34 : 18;
            constexpr float QMAX = T == SKV_Q8_0 ? 127.f : 7.f;
            uint8_t *seg = row + static_cast<int64_t>(h) * VPL * BLK;
#pragma unroll
            for (int b = 0; b < VPL; ++b) {
                const float xv = v[it][b];
                const float amax = warp_max32(fabsf(xv));
                const __half d16 = __float2half_rn(__fdiv_rn(amax, QMAX));
                const float d = __half2float(d16);
                const int q = d > 0.f ? __float2int_rn(__fdiv_rn(xv, d)) : 0;
                uint8_t *blk = seg + b * BLK;                     // 2-byte aligned
                if (T == SKV_Q8_0) {
                    const int c = max(-127, min(127, q)) & 0xff;
                    const int next = __shfl_down_sync(0xffffffffu, c, 1);
                    if (!(lane & 1)) reinterpret_cast<uint16_t *>(blk + 2)[lane >> 1] = static_cast<uint16_t>(c | (next << 8));
                } else {
                    const int u = max(0, min(15, q + 8));
                    const int hi = __shfl_down_sync(0xffffffffu, u, 16);   // value j + 16: high nibble of byte j
                    const int byte = u | (hi << 4);
                    const int next = __shfl_down_sync(0xffffffffu, byte, 1);
                    if (lane < 16 && !(lane & 1))
                        reinterpret_cast<uint16_t *>(blk + 2)[lane >> 1] = static_cast<uint16_t>(byte | (next << 8));
                }
                if (lane == 0) *reinterpret_cast<__half *>(blk) = d16;
            }
        }
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
#define SKV_APPEND(TT, V, DDD)                                                                                     \
    kv_append_kernel<TT, V, DDD><<<grid, kAppendThreads, 0, st>>>(x, positions, n, Hk, row_bytes, d0, n_rows0, d1, \
                                                                  n_rows1, h->status)
#define SKV_APPEND_D(TT, V) \
    do {                    \
        if (D == 64)        \
            SKV_APPEND(TT, V, 64); \
        else                \
            SKV_APPEND(TT, V, 128); \
    } while (0)
    if (type == SKV_F16) {
        if (vec8) SKV_APPEND_D(SKV_F16, true);
        else SKV_APPEND_D(SKV_F16, false);
    } else if (type == SKV_Q8_0) {
        SKV_APPEND_D(SKV_Q8_0, false);
    } else {
        SKV_APPEND_D(SKV_Q4_0, false);
    }
#undef SKV_APPEND_D
#undef SKV_APPEND
    return cuda_fail(h, cudaGetLastError(), "append launch");
}
