// combine.cu -- log-sum-exp merge of partial attention results.
//
// For each output row: M = max_t lse_t; w_t = e^{lse_t - M} (0 when
// lse_t = -inf); O = sum_t w_t O_t / sum_t w_t; lse = M + ln sum_t w_t.  This is
// the tile merge of the Rolling KV patch (fattn.cu key-axis tiling comment and
// streaming_combine_kernel), with the merged lse also written so that merged
// results can be merged again.
#include "internal.h"

namespace skv {

// One CTA per output row.  The parts' weights are computed in parallel into
// shared memory (after the maximum); then warp w takes parts w, w + W, ...
// (W warps) and lane l elements 4l .. 4l+3 (16-byte loads), so each warp keeps
// several parts' loads in flight; the warps' sums are added in shared memory.
// Few rows with many parts (a long range split across the whole GPU for a
// handful of query rows) take 1024 threads a row, so that each warp walks
// fewer parts; otherwise 256.
constexpr int kCombineMaxParts = 4096;

template <int kCombineThreads>
__global__ void __launch_bounds__(kCombineThreads) splitkv_combine_kernel(int n_parts,
                                                                          const float *__restrict__ o_parts,
                                                                          const float *__restrict__ lse_parts,
                                                                          int64_t rows, int D, float *__restrict__ o,
                                                                          float *__restrict__ lse)
{
    __shared__ float w_s[kCombineMaxParts];
    __shared__ float red[kCombineThreads / 32];
    __shared__ float4 acc_s[kCombineThreads / 32][32];
    static_assert(kCombineThreads % 32 == 0 && kCombineThreads <= 1024, "threads per row");
    // Launched as a programmatic dependent of the kernel that wrote the
    // parts: wait until that grid has completed and its writes are visible
    // (at once when there is no such grid).
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float M = -INFINITY;
    for (int p = tid; p < n_parts; p += kCombineThreads) M = fmaxf(M, lse_parts[static_cast<int64_t>(p) * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < kCombineThreads / 32; ++w) M = fmaxf(M, red[w]);
    if (M == -INFINITY) {
        for (int d = tid; d < D; d += kCombineThreads) o[row * D + d] = 0.f;
        if (tid == 0) lse[row] = -INFINITY;
        return;
    }
    float W = 0.f;
    for (int p = tid; p < n_parts; p += kCombineThreads) {
        const float l = lse_parts[static_cast<int64_t>(p) * rows + row];
        const float w = l == -INFINITY ? 0.f : expf(l - M);
        w_s[p] = w;
        W += w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
    __syncthreads();                                  // w_s complete; red[] free again
    if (lane == 0) red[warp] = W;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const int d0 = 4 * lane;
    if (d0 < D) {
        const int64_t stride = rows * D;
        const float *base = o_parts + row * D + d0;
        int p = warp;
        for (; p + 3 * (kCombineThreads / 32) < n_parts; p += 4 * (kCombineThreads / 32)) {
            float4 x[4];
            float w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int q = p + u * (kCombineThreads / 32);
                x[u] = *reinterpret_cast<const float4 *>(base + q * stride);
                w[u] = w_s[q];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (w[u] != 0.f) {
                    acc.x = fmaf(w[u], x[u].x, acc.x);
                    acc.y = fmaf(w[u], x[u].y, acc.y);
                    acc.z = fmaf(w[u], x[u].z, acc.z);
                    acc.w = fmaf(w[u], x[u].w, acc.w);
                }
            }
        }
        for (; p < n_parts; p += kCombineThreads / 32) {
            const float w = w_s[p];
            if (w != 0.f) {
                const float4 x = *reinterpret_cast<const float4 *>(base + p * stride);
                acc.x = fmaf(w, x.x, acc.x);
                acc.y = fmaf(w, x.y, acc.y);
                acc.z = fmaf(w, x.z, acc.z);
                acc.w = fmaf(w, x.w, acc.w);
            }
        }
    }
    acc_s[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float Wt = 0.f;
#pragma unroll
        for (int w = 0; w < kCombineThreads / 32; ++w) Wt += red[w];
        if (d0 < D) {
            float4 t = acc_s[0][lane];
#pragma unroll
            for (int w = 1; w < kCombineThreads / 32; ++w) {
                const float4 u = acc_s[w][lane];
                t.x += u.x;
                t.y += u.y;
                t.z += u.z;
                t.w += u.w;
            }
            const float inv = 1.f / Wt;
            *reinterpret_cast<float4 *>(o + row * D + d0) = make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
        }
        if (lane == 0) lse[row] = M + logf(Wt);
    }
}

int launch_combine(int n_parts, const float *o_parts, const float *lse_parts, int64_t rows, int D, float *o,
                   float *lse, cudaStream_t st)
{
    if (rows <= 0) return SKV_OK;
    if (rows > 0x7fffffff || n_parts > kCombineMaxParts || D > 128 || D % 4) return SKV_EUNSUPPORTED;
    // Programmatic dependent launch: the combine's CTAs may be scheduled
    // while the kernel before it on the stream finishes (that kernel lets its
    // dependents launch once its CTAs are past their main loop); each waits
    // for the whole of it before reading a part.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows));
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (n_parts >= 64 && rows <= 512) {
        cfg.blockDim = dim3(1024);
        e = cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<1024>, n_parts, o_parts, lse_parts, rows, D, o, lse);
    } else {
        cfg.blockDim = dim3(256);
        e = cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<256>, n_parts, o_parts, lse_parts, rows, D, o, lse);
    }
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? SKV_OK : SKV_ECUDA;
}

}  // namespace skv
