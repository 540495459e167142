// attn_fwd_dmix.cu -- instantiations of the persistent attention forward kernel
// for value heads of another width than the query/key heads (d_k != d_v).
#include "attn_kernel_dp.cuh"

namespace attn {

template <int DK, int DV>
static cudaError_t launch_mix(int mask, const TensorMaps& maps, const FwdParams& p, int num_sms,
                              cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return dp::launch<DK, DV, MASK_NONE>(maps, p, num_sms, stream);
    case MASK_CAUSAL: return dp::launch<DK, DV, MASK_CAUSAL>(maps, p, num_sms, stream);
    case MASK_KEY_PADDING: return dp::launch<DK, DV, MASK_KEY_PADDING>(maps, p, num_sms, stream);
    case MASK_CAUSAL_KEY_PADDING: return dp::launch<DK, DV, MASK_CAUSAL_KEY_PADDING>(maps, p, num_sms, stream);
    case MASK_CAUSAL_CACHE: return dp::launch<DK, DV, MASK_CAUSAL_CACHE>(maps, p, num_sms, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_fwd_dmix(int d_k, int d_v, int mask, const TensorMaps& maps, const FwdParams& p,
                            int num_sms, cudaStream_t stream)
{
    if (d_k == 64 && d_v == 128) return launch_mix<64, 128>(mask, maps, p, num_sms, stream);
    if (d_k == 128 && d_v == 64) return launch_mix<128, 64>(mask, maps, p, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
