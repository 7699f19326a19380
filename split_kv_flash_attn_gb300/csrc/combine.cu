// combine.cu -- log-sum-exp merge of partial attention results.
//
// For each output row: M = max_t lse_t; w_t = e^{lse_t - M} (0 when
// lse_t = -inf); O = sum_t w_t O_t / sum_t w_t; lse = M + ln sum_t w_t.  This is
// the tile merge of the Rolling KV patch (fattn.cu key-axis tiling comment and
// streaming_combine_kernel), with the merged lse also written so that merged
// results can be merged again.
#include "internal.h"

namespace skv {

// One CTA of 128 threads per output row: the lse of all parts are read in
// parallel (one part per thread) for the maximum, then in chunks of 128 the
// weights go to shared memory and thread d accumulates element d over the
// chunk's parts, whose loads are independent of one another.
__global__ void __launch_bounds__(128) splitkv_combine_kernel(int n_parts, const float *__restrict__ o_parts,
                                                              const float *__restrict__ lse_parts, int64_t rows,
                                                              int D, float *__restrict__ o, float *__restrict__ lse)
{
    __shared__ float w_s[128];
    __shared__ float red[4];
    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x;
    float M = -INFINITY;
    for (int p = tid; p < n_parts; p += 128) M = fmaxf(M, lse_parts[static_cast<int64_t>(p) * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if ((tid & 31) == 0) red[tid >> 5] = M;
    __syncthreads();
    M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    if (M == -INFINITY) {
        if (tid < D) o[row * D + tid] = 0.f;
        if (tid == 0) lse[row] = -INFINITY;
        return;
    }
    float acc = 0.f;
    float W = 0.f;
    for (int base = 0; base < n_parts; base += 128) {
        const int cnt = min(128, n_parts - base);
        __syncthreads();
        if (tid < cnt) {
            const float l = lse_parts[static_cast<int64_t>(base + tid) * rows + row];
            w_s[tid] = l == -INFINITY ? 0.f : expf(l - M);
        }
        __syncthreads();
        if (tid < D) {
            const float *op = o_parts + (static_cast<int64_t>(base) * rows + row) * D + tid;
            const int64_t stride = rows * D;
#pragma unroll 8
            for (int i = 0; i < cnt; ++i) {
                const float w = w_s[i];
                const float x = op[i * stride];
                acc = w != 0.f ? fmaf(w, x, acc) : acc;
            }
        }
        for (int i = 0; i < cnt; ++i) W += w_s[i];
    }
    if (tid < D) o[row * D + tid] = acc / W;
    if (tid == 0) lse[row] = M + logf(W);
}

int launch_combine(int n_parts, const float *o_parts, const float *lse_parts, int64_t rows, int D, float *o,
                   float *lse, cudaStream_t st)
{
    if (rows <= 0) return SKV_OK;
    if (rows > 0x7fffffff) return SKV_EUNSUPPORTED;
    splitkv_combine_kernel<<<static_cast<unsigned>(rows), 128, 0, st>>>(n_parts, o_parts, lse_parts, rows, D, o, lse);
    return cudaGetLastError() == cudaSuccess ? SKV_OK : SKV_ECUDA;
}

}  // namespace skv
