// combine.cu -- log-sum-exp merge of partial attention results.
//
// For each output row: M = max_t lse_t; w_t = e^{lse_t - M} (0 when
// lse_t = -inf); O = sum_t w_t O_t / sum_t w_t; lse = M + ln sum_t w_t.  This is
// the tile merge of the Rolling KV patch (fattn.cu key-axis tiling comment and
// streaming_combine_kernel), with the merged lse also written so that merged
// results can be merged again.  One warp per row: lanes take parts for the
// max, then head-dim elements for the weighted sum (coalesced 128-byte reads
// of each part's row).
#include "internal.h"

namespace skv {

__global__ void __launch_bounds__(256) splitkv_combine_kernel(int n_parts, const float *__restrict__ o_parts,
                                                              const float *__restrict__ lse_parts, int64_t rows,
                                                              int D, float *__restrict__ o, float *__restrict__ lse)
{
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float M = -INFINITY;
    for (int p = lane; p < n_parts; p += 32) M = fmaxf(M, lse_parts[static_cast<int64_t>(p) * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float *orow = o + row * D;
    if (M == -INFINITY) {
        for (int d = lane; d < D; d += 32) orow[d] = 0.f;
        if (lane == 0) lse[row] = -INFINITY;
        return;
    }
    // Up to 4 head-dim elements per lane stay in registers (D <= 128).
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float W = 0.f;
    for (int p = 0; p < n_parts; ++p) {
        const float l = lse_parts[static_cast<int64_t>(p) * rows + row];
        if (l == -INFINITY) continue;
        const float w = expf(l - M);
        W += w;
        const float *op = o_parts + (static_cast<int64_t>(p) * rows + row) * D;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int d = lane + 32 * e;
            if (d < D) acc[e] = fmaf(w, op[d], acc[e]);
        }
    }
    const float inv = 1.f / W;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int d = lane + 32 * e;
        if (d < D) orow[d] = acc[e] * inv;
    }
    if (lane == 0) lse[row] = M + logf(W);
}

int launch_combine(int n_parts, const float *o_parts, const float *lse_parts, int64_t rows, int D, float *o,
                   float *lse, cudaStream_t st)
{
    if (rows <= 0) return SKV_OK;
    const int rows_per_block = 8;
    const int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
    splitkv_combine_kernel<<<static_cast<unsigned>(blocks), 32 * rows_per_block, 0, st>>>(n_parts, o_parts, lse_parts,
                                                                                         rows, D, o, lse);
    return cudaGetLastError() == cudaSuccess ? SKV_OK : SKV_ECUDA;
}

}  // namespace skv
