// prefill_sw.cu -- software-producer instances of the tensor-core prefill
// kernel: fp16 rows through row lists (MODE 2), and q8_0 / q4_0 rows (listed,
// or dense with q8_0 values or a single query tile) decoded into the fp16
// operand tiles (MODE 1).
#include "prefill_kernel.cuh"

namespace skv {
namespace pf {

int launch_prefill_sw(skv_handle *h, const PrefillArgs &a, int kt, int vt, dim3 grid, cudaStream_t st)
{
    CUtensorMap none;
    memset(&none, 0, sizeof(none));
#define SKV_PF(KT, VT) \
    if (kt == KT && vt == VT) return launch_prefill_t<1, KT, VT>(h, none, none, a, grid, st)
    SKV_PF(SKV_Q8_0, SKV_Q8_0);
    SKV_PF(SKV_Q8_0, SKV_Q4_0);
    SKV_PF(SKV_Q4_0, SKV_Q8_0);
    SKV_PF(SKV_Q4_0, SKV_Q4_0);
#undef SKV_PF
    if (kt == SKV_F16 && vt == SKV_F16 && a.rows) return launch_prefill_t<2, SKV_F16, SKV_F16>(h, none, none, a, grid, st);
    return fail(h, SKV_EUNSUPPORTED, "no prefill kernel for K type %d / V type %d", kt, vt);
}

}  // namespace pf
}  // namespace skv
