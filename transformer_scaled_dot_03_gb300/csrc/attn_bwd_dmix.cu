// attn_bwd_dmix.cu -- instantiations of the attention backward kernel for value
// heads of another width than the query/key heads (d_k != d_v).
#include "attn_kernel_bwd.cuh"

namespace attn {

template <int DK, int DV>
static cudaError_t launch_mix(int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return bwd::launch<DK, DV, MASK_NONE>(maps, p, stream);
    case MASK_CAUSAL: return bwd::launch<DK, DV, MASK_CAUSAL>(maps, p, stream);
    case MASK_KEY_PADDING: return bwd::launch<DK, DV, MASK_KEY_PADDING>(maps, p, stream);
    case MASK_CAUSAL_KEY_PADDING: return bwd::launch<DK, DV, MASK_CAUSAL_KEY_PADDING>(maps, p, stream);
    case MASK_CAUSAL_CACHE: return bwd::launch<DK, DV, MASK_CAUSAL_CACHE>(maps, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_dmix(int d_k, int d_v, int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    if (d_k == 64 && d_v == 128) return launch_mix<64, 128>(mask, maps, p, stream);
    if (d_k == 128 && d_v == 64) return launch_mix<128, 64>(mask, maps, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
