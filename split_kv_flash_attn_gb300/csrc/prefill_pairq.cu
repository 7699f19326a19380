// prefill_pairq.cu -- instances of the two-query-tile prefill kernel over
// dense q8_0 / q4_0 keys and q4_0 values (prefill_pairq.cuh).
#include "prefill_pairq.cuh"

namespace skv {
namespace pf {

int launch_prefill_pairq(skv_handle *h, const PrefillArgs &a, int kt, dim3 grid, cudaStream_t st)
{
    if (kt == SKV_Q8_0) return launch_prefill_pairq_t<SKV_Q8_0>(h, a, grid, st);
    if (kt == SKV_Q4_0) return launch_prefill_pairq_t<SKV_Q4_0>(h, a, grid, st);
    return fail(h, SKV_EUNSUPPORTED, "no pair prefill kernel for K type %d", kt);
}

}  // namespace pf
}  // namespace skv
