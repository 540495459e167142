// attn_fwd_d64.cu -- instantiations of the persistent attention forward kernel for
// head dim 64 (d_k = d_v = 64).
#include "attn_kernel_dp.cuh"

namespace attn {

cudaError_t launch_fwd_d64(int mask, const TensorMaps& maps, const FwdParams& p, int num_sms, cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return dp::launch<64, 64, MASK_NONE>(maps, p, num_sms, stream);
    case MASK_CAUSAL: return dp::launch<64, 64, MASK_CAUSAL>(maps, p, num_sms, stream);
    case MASK_KEY_PADDING: return dp::launch<64, 64, MASK_KEY_PADDING>(maps, p, num_sms, stream);
    case MASK_CAUSAL_KEY_PADDING: return dp::launch<64, 64, MASK_CAUSAL_KEY_PADDING>(maps, p, num_sms, stream);
    case MASK_CAUSAL_CACHE: return dp::launch<64, 64, MASK_CAUSAL_CACHE>(maps, p, num_sms, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
