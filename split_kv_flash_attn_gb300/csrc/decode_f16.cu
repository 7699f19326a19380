// decode_f16.cu -- fp16-row instances of the split-KV decode kernel.
#include "decode_kernel.cuh"

namespace skv {

int launch_decode_f16(skv_handle *h, const DecodeArgs &a, int D, cudaStream_t st)
{
    if (D == 128) return launch_decode_t<128, SKV_F16, SKV_F16>(h, a, st);
    if (D == 64) return launch_decode_t<64, SKV_F16, SKV_F16>(h, a, st);
    return fail(h, SKV_EUNSUPPORTED, "head dim %d (supported: 64, 128)", D);
}

int launch_decode_fused(skv_handle *h, const DecodeArgs &a, int D, cudaStream_t st)
{
    if (D == 128) return launch_decode_fused_t<128>(h, a, st);
    if (D == 64) return launch_decode_fused_t<64>(h, a, st);
    return fail(h, SKV_EUNSUPPORTED, "head dim %d (supported: 64, 128)", D);
}

int decode_ctas_f16(skv_handle *h, int D)
{
    if (D == 128) return decode_ctas_per_sm_t<128, SKV_F16, SKV_F16>(h);
    if (D == 64) return decode_ctas_per_sm_t<64, SKV_F16, SKV_F16>(h);
    return 0;
}

}  // namespace skv
