// attn_fwd_d64.cu -- instantiations of the attention forward kernel for head dim 64.
#include "attn_kernel.cuh"

namespace attn {

cudaError_t launch_fwd_d64(int mask, const TensorMaps& maps, const FwdParams& p, int64_t num_ctas,
                           cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return launch_fwd<64, MASK_NONE>(maps, p, num_ctas, stream);
    case MASK_CAUSAL: return launch_fwd<64, MASK_CAUSAL>(maps, p, num_ctas, stream);
    case MASK_KEY_PADDING: return launch_fwd<64, MASK_KEY_PADDING>(maps, p, num_ctas, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
