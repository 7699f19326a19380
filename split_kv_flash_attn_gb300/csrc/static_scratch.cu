// static_scratch.cu -- skv_attn_partial_static: the split-KV decode attention
// of skv_attn_partial for callers that must not allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not an option -- an engine
// that reserves all device memory up front and hands out slices from its own
// pool (a raw cudaMalloc would fail or fragment that reservation), a latency-
// critical path that cannot take the device-wide synchronisation a
// cudaMalloc/cudaFree may cause, or a caller with no library handle at all
// (skv_create itself allocates).  Such a caller passes its inputs and outputs;
// the only scratch, the per-split partial results and the per-unit arrival
// counters of the in-kernel merge, lives in one fixed-size array in device
// global memory that the library image carries.  Every GPU that loads the
// library holds that array until the process exits.
#include <mutex>
#include <string.h>

#include <algorithm>

#include "internal.h"

namespace skv {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;      // 16 MiB per device
constexpr int kStaticUnits = 4096;                             // arrival counters at the start
constexpr size_t kStaticCounterBytes = sizeof(int) * kStaticUnits;
constexpr int kStaticMaxDevices = 64;

// Host code must not use this symbol's address directly: on the host it names
// a stand-in, not device memory.  Its device address is looked up once per
// device (cudaGetSymbolAddress) and passed to the kernels.  The address is
// kept for the life of the process: after cudaDeviceReset on a device it is
// stale, so this entry point must not be called on a device that was reset.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kStaticMaxDevices] = {};
int g_sm_count[kStaticMaxDevices] = {};

// First call on a device, with that device current: look up the array's
// device address and the SM count.
int static_setup(int dev, void **addr, int *sm_count)
{
    if (dev < 0 || dev >= kStaticMaxDevices) return SKV_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return SKV_ECUDA;
        }
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess || n <= 0) {
            cudaGetLastError();
            return SKV_ECUDA;
        }
        g_scratch_addr[dev] = p;
        g_sm_count[dev] = n;
    }
    *addr = g_scratch_addr[dev];
    *sm_count = g_sm_count[dev];
    return SKV_OK;
}

int64_t seg_of(int type, int D)
{
    return type == SKV_F16 ? 2 * int64_t(D) : type == SKV_Q8_0 ? 34 * int64_t(D / 32) : 18 * int64_t(D / 32);
}

}  // namespace
}  // namespace skv

using namespace skv;

extern "C" int skv_attn_partial_static(const skv_shape *shape, const void *q, const void *k, const void *v,
                                       const void *mask, int64_t mask_ld, const int32_t *q_pos, int64_t key_pos0,
                                       const int32_t *kv_rows, int64_t kv_rows_ld, int32_t kv_rows_per_head,
                                       int64_t kv_begin, int64_t kv_end, float *o, float *lse, void *stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!shape || !q || !k || !v || !o || !lse) return SKV_EINVAL;
    const skv_shape &sh = *shape;
    if (sh.S <= 0 || sh.nq <= 0 || sh.H <= 0 || sh.Hk <= 0 || sh.H % sh.Hk != 0) return SKV_EINVAL;
    if (sh.D != 64 && sh.D != 128) return SKV_EUNSUPPORTED;
    if (sh.k_type < SKV_F16 || sh.k_type > SKV_Q4_0 || sh.v_type < SKV_F16 || sh.v_type > SKV_Q4_0) return SKV_EINVAL;
    if ((sh.k_type == SKV_F16) != (sh.v_type == SKV_F16)) return SKV_EUNSUPPORTED;
    const int64_t segk = seg_of(sh.k_type, sh.D), segv = seg_of(sh.v_type, sh.D);
    if (sh.k_row_bytes < sh.Hk * segk || sh.v_row_bytes < sh.Hk * segv) return SKV_EINVAL;
    const int ck = sh.k_type == SKV_F16 ? 16 : (segk % 8 == 0 ? 8 : 4);
    const int cv = sh.v_type == SKV_F16 ? 16 : (segv % 8 == 0 ? 8 : 4);
    if ((reinterpret_cast<uintptr_t>(k) % ck) || (sh.k_row_bytes % ck) || (reinterpret_cast<uintptr_t>(v) % cv) ||
        (sh.v_row_bytes % cv))
        return SKV_EUNSUPPORTED;
    if (kv_begin < 0 || kv_end < kv_begin) return SKV_EINVAL;
    if (kv_rows && kv_rows_ld < kv_end) return SKV_EINVAL;
    if (mask && mask_ld < kv_end) return SKV_EINVAL;
    const int G = sh.H / sh.Hk;
    const int n_cg = (sh.nq * G + 7) / 8;
    const int64_t units = int64_t(sh.S) * sh.Hk * n_cg;
    if (units > 65535) return SKV_EUNSUPPORTED;
    const int64_t R = int64_t(sh.S) * sh.nq * sh.H;
    const int D = sh.D;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SKV_ECUDA;
    }
    void *scratch = nullptr;
    int sm_count = 0;
    int rc = static_setup(dev, &scratch, &sm_count);
    if (rc) return rc;

    const int64_t n_local = kv_end - kv_begin;
    if (n_local == 0) return launch_combine(0, nullptr, nullptr, R, D, o, lse, st);
    const bool f16 = sh.k_type == SKV_F16;
    const int ctas = f16 ? decode_ctas_f16(nullptr, D) : decode_ctas_quant(nullptr, sh.k_type, sh.v_type, D);
    if (ctas <= 0) return SKV_EUNSUPPORTED;
    // The stated maximum: one arrival counter per unit in the array's head.
    if (units > kStaticUnits) return SKV_ENOMEM;
    int64_t split_len = 0;
    int32_t n_splits = 0;
    rc = skv_plan_splits(n_local, units, sm_count, ctas, kDecodeTile, 0, &split_len,
                         &n_splits);
    if (rc) return rc;
    // The split count is free: when the planned splits' partials do not fit
    // the array, use as many as fit (one split writes o/lse directly and
    // needs no scratch at all).
    const size_t per_split = size_t(R) * D * sizeof(float) + size_t(R) * sizeof(float);
    const int64_t max_fit = int64_t((kStaticScratchBytes - kStaticCounterBytes - 256) / per_split);
    if (n_splits > 1 && n_splits > max_fit) {
        const int64_t want = max_fit > 1 ? max_fit : 1;
        split_len = (n_local + want - 1) / want;
        split_len = (split_len + kDecodeTile - 1) / kDecodeTile * kDecodeTile;
        n_splits = static_cast<int32_t>((n_local + split_len - 1) / split_len);
    }
    if (n_splits > kMaxSplits) return SKV_EUNSUPPORTED;
    // The fixed scratch: counters, then O partials, then lse partials.
    const size_t o_bytes = (size_t(n_splits) * R * D * sizeof(float) + 255) / 256 * 256;
    const size_t l_bytes = size_t(n_splits) * R * sizeof(float);
    if (n_splits > 1 && kStaticCounterBytes + o_bytes + l_bytes > kStaticScratchBytes) return SKV_ENOMEM;

    DecodeArgs a;
    memset(&a, 0, sizeof(a));
    a.q = static_cast<const __half *>(q);
    a.k = static_cast<const uint8_t *>(k);
    a.v = static_cast<const uint8_t *>(v);
    a.k_row_bytes = sh.k_row_bytes;
    a.v_row_bytes = sh.v_row_bytes;
    if (kv_rows) {
        a.row_mode = ROWS_LIST;
        a.rows = kv_rows;
        a.rows_ld = kv_rows_ld;
        a.rows_per_head = kv_rows_per_head ? 1 : 0;
        a.rows_off = kv_begin;
    } else {
        a.row_mode = ROWS_DENSE;
        a.row0 = kv_begin;
    }
    a.mask = static_cast<const __half *>(mask);
    a.mask_ld = mask_ld;
    a.q_pos = q_pos;
    a.key_pos0 = key_pos0;
    a.logical0 = kv_begin;
    a.n_local = n_local;
    a.S = sh.S;
    a.nq = sh.nq;
    a.H = sh.H;
    a.Hk = sh.Hk;
    a.G = G;
    a.scale_log2 = sh.scale * 1.4426950408889634f;
    a.n_cg = n_cg;
    a.n_splits = n_splits;
    a.split_len = split_len;
    a.R = R;
    a.o_out = o;
    a.lse_out = lse;
    uint8_t *base = static_cast<uint8_t *>(scratch);
    a.counters = reinterpret_cast<int *>(base);
    a.o_split = reinterpret_cast<float *>(base + kStaticCounterBytes);
    a.lse_split = reinterpret_cast<float *>(base + kStaticCounterBytes + o_bytes);
    if (n_splits > 1) {
        // The array keeps whatever the last call left: the merge's arrival
        // counters must start at zero.
        cudaError_t e = cudaMemsetAsync(a.counters, 0, sizeof(int) * size_t(units), st);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return SKV_ECUDA;
        }
    }
    return f16 ? launch_decode_f16(nullptr, a, D, st) : launch_decode_quant(nullptr, a, sh.k_type, sh.v_type, D, st);
}
