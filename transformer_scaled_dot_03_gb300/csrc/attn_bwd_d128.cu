// attn_bwd_d128.cu -- instantiations of the attention backward for head dim 128
// (d_k = d_v = 128): the pipelined 64-query-step kernel.
#include "attn_kernel_bwd128.cuh"

namespace attn {

cudaError_t launch_bwd_d128(int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return bwd128::launch<MASK_NONE>(maps, p, stream);
    case MASK_CAUSAL: return bwd128::launch<MASK_CAUSAL>(maps, p, stream);
    case MASK_KEY_PADDING: return bwd128::launch<MASK_KEY_PADDING>(maps, p, stream);
    case MASK_CAUSAL_KEY_PADDING: return bwd128::launch<MASK_CAUSAL_KEY_PADDING>(maps, p, stream);
    case MASK_CAUSAL_CACHE: return bwd128::launch<MASK_CAUSAL_CACHE>(maps, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
