// quant.cu -- q8_0 / q4_0 block decoding to fp32 and the row gather.
//
// Block formats (32 values each): q8_0 = fp16 scale d + 32 int8 codes, value
// d*q; q4_0 = fp16 scale d + 16 bytes, byte j holding u_j (low nibble) and
// u_{j+16} (high nibble), value d*(u-8).  The pages name these types (Rolling KV
// patch sizer, q8_0 block of 32; opencoti patch 0102 on raw quant bytes) but do
// not print their bytes; this is the ggml layout.  fp16 has an 11-bit
// significand and a code needs at most 8 bits, so d*q is exact in fp32.
//
// The gather copies whole rows through a row list; a negative entry writes a
// zero row and reads nothing (the flash_attn_ext_rows thread's fused-kernel
// fix gathers through the index list with padding clamped).
#include "internal.h"

namespace skv {

// One thread per 8 output values; consecutive threads cover consecutive
// values, so both the block reads and the fp32 writes are contiguous.
template <int T>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ blocks, int64_t n_values,
                                                      float *__restrict__ out)
{
    const int64_t n8 = n_values / 8;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = i >> 2;        // block
        const int part = static_cast<int>(i & 3);
        float v[8];
        if constexpr (T == SKV_Q8_0) {
            const uint8_t *blk = blocks + b * 34;
            const float d = __half2float(*reinterpret_cast<const __half *>(blk));
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = d * static_cast<float>(static_cast<int8_t>(blk[2 + part * 8 + e]));
        } else {
            const uint8_t *blk = blocks + b * 18;
            const float d = __half2float(*reinterpret_cast<const __half *>(blk));
            const int byte0 = (part & 1) * 8;
            const int shift = (part >> 1) * 4;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                v[e] = d * static_cast<float>(static_cast<int>((blk[2 + byte0 + e] >> shift) & 0xF) - 8);
        }
        float4 *o4 = reinterpret_cast<float4 *>(out + i * 8);
        o4[0] = make_float4(v[0], v[1], v[2], v[3]);
        o4[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
}

int launch_dequant(int type, const void *blocks, int64_t n_values, float *out, cudaStream_t st)
{
    if (n_values <= 0) return SKV_OK;
    const int64_t n8 = n_values / 8;
    const int threads = 256;
    const int64_t want = (n8 + threads - 1) / threads;
    const unsigned grid = static_cast<unsigned>(want < 65536 ? want : 65536);
    if (type == SKV_Q8_0)
        dequant_kernel<SKV_Q8_0><<<grid, threads, 0, st>>>(static_cast<const uint8_t *>(blocks), n_values, out);
    else
        dequant_kernel<SKV_Q4_0><<<grid, threads, 0, st>>>(static_cast<const uint8_t *>(blocks), n_values, out);
    return cudaGetLastError() == cudaSuccess ? SKV_OK : SKV_ECUDA;
}

// Row gather with a vector width W (16, 4 or 1 bytes) that divides the row
// size and both base addresses.  One warp per row.
template <typename V>
__global__ void __launch_bounds__(256) gather_kernel(const uint8_t *__restrict__ src, int64_t row_bytes,
                                                     const int32_t *__restrict__ rows, int64_t n,
                                                     uint8_t *__restrict__ dst)
{
    const int64_t nv = row_bytes / static_cast<int64_t>(sizeof(V));
    const int lane = threadIdx.x & 31;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); i < n;
         i += static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5)) {
        const int32_t r = rows[i];
        V *d = reinterpret_cast<V *>(dst + i * row_bytes);
        if (r < 0) {
            V z;
            memset(&z, 0, sizeof(V));
            for (int64_t e = lane; e < nv; e += 32) d[e] = z;
        } else {
            const V *s = reinterpret_cast<const V *>(src + static_cast<int64_t>(r) * row_bytes);
            for (int64_t e = lane; e < nv; e += 32) d[e] = s[e];
        }
    }
}

int launch_gather(const void *src, int64_t row_bytes, const int32_t *rows, int64_t n, void *dst, cudaStream_t st)
{
    if (n <= 0 || row_bytes <= 0) return SKV_OK;
    const uintptr_t al = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
                         static_cast<uintptr_t>(row_bytes);
    const int threads = 256;
    const int64_t want = (n + 7) / 8;
    const unsigned grid = static_cast<unsigned>(want < 65536 ? want : 65536);
    const uint8_t *s = static_cast<const uint8_t *>(src);
    uint8_t *d = static_cast<uint8_t *>(dst);
    if ((al & 15) == 0) gather_kernel<uint4><<<grid, threads, 0, st>>>(s, row_bytes, rows, n, d);
    else if ((al & 3) == 0) gather_kernel<uint32_t><<<grid, threads, 0, st>>>(s, row_bytes, rows, n, d);
    else gather_kernel<uint8_t><<<grid, threads, 0, st>>>(s, row_bytes, rows, n, d);
    return cudaGetLastError() == cudaSuccess ? SKV_OK : SKV_ECUDA;
}

}  // namespace skv
