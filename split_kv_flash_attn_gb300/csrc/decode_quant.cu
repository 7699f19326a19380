// decode_quant.cu -- q8_0 / q4_0 instances of the split-KV decode kernel
// (codes staged raw, converted per warp to fp16 codes + fp32 block scales).
#include "decode_kernel.cuh"

namespace skv {

template <int D>
static int launch_q(skv_handle *h, const DecodeArgs &a, int kt, int vt, cudaStream_t st)
{
    if (kt == SKV_Q8_0 && vt == SKV_Q4_0) return launch_decode_t<D, SKV_Q8_0, SKV_Q4_0>(h, a, st);
    if (kt == SKV_Q8_0 && vt == SKV_Q8_0) return launch_decode_t<D, SKV_Q8_0, SKV_Q8_0>(h, a, st);
    if (kt == SKV_Q4_0 && vt == SKV_Q4_0) return launch_decode_t<D, SKV_Q4_0, SKV_Q4_0>(h, a, st);
    if (kt == SKV_Q4_0 && vt == SKV_Q8_0) return launch_decode_t<D, SKV_Q4_0, SKV_Q8_0>(h, a, st);
    return fail(h, SKV_EUNSUPPORTED, "K/V type pairing (%d, %d)", kt, vt);
}

template <int D>
static int ctas_q(skv_handle *h, int kt, int vt)
{
    if (kt == SKV_Q8_0 && vt == SKV_Q4_0) return decode_ctas_per_sm_t<D, SKV_Q8_0, SKV_Q4_0>(h);
    if (kt == SKV_Q8_0 && vt == SKV_Q8_0) return decode_ctas_per_sm_t<D, SKV_Q8_0, SKV_Q8_0>(h);
    if (kt == SKV_Q4_0 && vt == SKV_Q4_0) return decode_ctas_per_sm_t<D, SKV_Q4_0, SKV_Q4_0>(h);
    if (kt == SKV_Q4_0 && vt == SKV_Q8_0) return decode_ctas_per_sm_t<D, SKV_Q4_0, SKV_Q8_0>(h);
    return 0;
}

int launch_decode_quant(skv_handle *h, const DecodeArgs &a, int kt, int vt, int D, cudaStream_t st)
{
    if (D == 128) return launch_q<128>(h, a, kt, vt, st);
    if (D == 64) return launch_q<64>(h, a, kt, vt, st);
    return fail(h, SKV_EUNSUPPORTED, "head dim %d (supported: 64, 128)", D);
}

int decode_ctas_quant(skv_handle *h, int kt, int vt, int D)
{
    if (D == 128) return ctas_q<128>(h, kt, vt);
    if (D == 64) return ctas_q<64>(h, kt, vt);
    return 0;
}

}  // namespace skv
