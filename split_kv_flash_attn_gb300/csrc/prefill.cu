// prefill.cu -- host side of the tensor-core prefill kernel
// (prefill_kernel.cuh): eligibility, tensor maps, split arguments, and the
// TMA instance over dense fp16 regions.  Dense q8_0 / q4_0 keys with q4_0
// values over two or more query tiles use the two-query-tile instance
// (prefill_pairq.cu); other row lists and quantised rows the
// software-producer instances in prefill_sw.cu.
#include "prefill_kernel.cuh"

namespace skv {

using namespace pf;

// ---- host side ------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver entry point is process-wide (not per device); it is looked up
// once, under C++'s thread-safe initialisation of a local static.
static EncodeTiledFn encode_fn()
{
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
        return nullptr;
    }();
    return fn;
}

// 2-D map over a cell-major fp16 cache region: x = element within the row
// (Hk*D wide), y = row; box 64 x 128 with the 128-byte swizzle.
static int make_map(skv_handle *h, CUtensorMap *map, const void *base, int64_t n_rows, int Hk, int64_t row_bytes)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(h, SKV_ECUDA, "cuTensorMapEncodeTiled is not available");
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(Hk) * kPD, static_cast<cuuint64_t>(n_rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {64, kPN};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(h, SKV_EUNSUPPORTED, "tensor map encoding failed (%d)", static_cast<int>(r));
    return SKV_OK;
}

bool prefill_eligible(const skv_shape *sh, const void *mask)
{
    // fp16 rows move in 16-byte pieces, quantised segments in 8-byte loads
    const bool f16 = sh->k_type == SKV_F16 && sh->v_type == SKV_F16;
    const bool quant = sh->k_type != SKV_F16 && sh->v_type != SKV_F16;
    const int64_t al = f16 ? 16 : 8;
    return (f16 || quant) && sh->D == kPD && mask == nullptr && (kPM % (sh->H / sh->Hk)) == 0 &&
           static_cast<int64_t>(sh->nq) * (sh->H / sh->Hk) >= 64 && sh->k_row_bytes % al == 0 &&
           sh->v_row_bytes % al == 0;
}

// Dense q8_0 / q4_0 keys with q4_0 values and at least two query tiles: the
// two-query-tile instance, which decodes each K and V tile once for both.
bool prefill_pairs(const skv_shape *sh, bool rows)
{
    const int m_tiles = (sh->nq * (sh->H / sh->Hk) + kPM - 1) / kPM;
    return !rows && (sh->k_type == SKV_Q8_0 || sh->k_type == SKV_Q4_0) && sh->v_type == SKV_Q4_0 && m_tiles >= 2;
}

int prefill_units(const skv_shape *sh, bool rows)
{
    const int m_tiles = (sh->nq * (sh->H / sh->Hk) + kPM - 1) / kPM;
    return sh->Hk * (prefill_pairs(sh, rows) ? (m_tiles + 1) / 2 : m_tiles);
}

int launch_prefill(skv_handle *h, const PrefillLaunch &L, cudaStream_t st)
{
    const skv_shape *sh = L.shape;
    const int G = sh->H / sh->Hk;
    const bool f16 = sh->k_type == SKV_F16 && sh->v_type == SKV_F16;
    PrefillArgs a;
    memset(&a, 0, sizeof(a));
    a.q = static_cast<const __half *>(L.q);
    a.S = sh->S;
    a.nq = sh->nq;
    a.H = sh->H;
    a.Hk = sh->Hk;
    a.G = G;
    a.scale_log2 = sh->scale * 1.4426950408889634f;
    a.q_pos = L.q_pos;
    a.key_pos0 = L.key_pos0;
    a.logical0 = L.logical0;
    a.row0 = L.row0;
    a.n_local = L.n_local;
    a.m_tiles = (sh->nq * G + kPM - 1) / kPM;
    a.n_splits = L.n_splits;
    a.split_len = L.split_len;
    a.o_split = L.o_split;
    a.lse_split = L.lse_split;
    a.counters = h->counters;
    a.o_out = L.o_out;
    a.lse_out = L.lse_out;
    a.R = static_cast<int64_t>(sh->S) * sh->nq * sh->H;
    a.status = h->status;
    a.k = static_cast<const uint8_t *>(L.k);
    a.v = static_cast<const uint8_t *>(L.v);
    a.k_row_bytes = sh->k_row_bytes;
    a.v_row_bytes = sh->v_row_bytes;
    a.rows = L.rows;
    a.rows_ld = L.rows_ld;
    a.rows_off = L.rows_off;
    a.rows_per_head = L.rows_per_head;
    if (a.split_len % kPN) return fail(h, SKV_EINVAL, "prefill split length must be a multiple of %d", kPN);
    if (sh->Hk * a.m_tiles > 65535 || a.n_splits > 65535 || sh->S > 65535)
        return fail(h, SKV_EUNSUPPORTED, "prefill grid too large");
    // split index slowest: every CTA of split 0 is dispatched before any of
    // split 1 (head-and-tail plans rely on it)
    dim3 grid(static_cast<unsigned>(sh->Hk * a.m_tiles), static_cast<unsigned>(sh->S),
              static_cast<unsigned>(a.n_splits));
    if ((reinterpret_cast<uintptr_t>(L.k) | reinterpret_cast<uintptr_t>(L.v)) % (f16 ? 16 : 8))
        return fail(h, SKV_EUNSUPPORTED, "K/V bases must be %d-byte aligned for the prefill kernel", f16 ? 16 : 8);
    if (prefill_pairs(sh, L.rows != nullptr)) {
        const int n_pairs = (a.m_tiles + 1) / 2;
        return launch_prefill_pairq(h, a, sh->k_type,
                                    dim3(static_cast<unsigned>(sh->Hk * n_pairs), grid.y, grid.z), st);
    }
    if (!f16 || L.rows) return launch_prefill_sw(h, a, sh->k_type, sh->v_type, grid, st);
    CUtensorMap mk, mv;
    int rc = make_map(h, &mk, L.k, L.n_rows, sh->Hk, sh->k_row_bytes);
    if (rc == SKV_OK) rc = make_map(h, &mv, L.v, L.n_rows, sh->Hk, sh->v_row_bytes);
    if (rc) return rc;
    if (L.row0 + L.n_local > 0x7fffffff) return fail(h, SKV_EUNSUPPORTED, "region too long for the tensor map");
    return launch_prefill_t<0, SKV_F16, SKV_F16>(h, mk, mv, a, grid, st);
}

}  // namespace skv
