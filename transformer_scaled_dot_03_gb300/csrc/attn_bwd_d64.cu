// attn_bwd_d64.cu -- instantiations of the attention backward kernel for head dim 64.
#include "attn_kernel_bwd.cuh"

namespace attn {

cudaError_t launch_bwd_d64(int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return bwd::launch<64, 64, MASK_NONE>(maps, p, stream);
    case MASK_CAUSAL: return bwd::launch<64, 64, MASK_CAUSAL>(maps, p, stream);
    case MASK_KEY_PADDING: return bwd::launch<64, 64, MASK_KEY_PADDING>(maps, p, stream);
    case MASK_CAUSAL_KEY_PADDING: return bwd::launch<64, 64, MASK_CAUSAL_KEY_PADDING>(maps, p, stream);
    case MASK_CAUSAL_CACHE: return bwd::launch<64, 64, MASK_CAUSAL_CACHE>(maps, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
