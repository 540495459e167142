// attn_bwd_alibi.cu -- instantiations of the attention backward kernels with the
// linear distance bias (ALiBi, "第2章：完整的 Transformer 架构" §5.3), for head
// dims d_k = d_v = 64 and 128.
#include "attn_kernel_bwd.cuh"

namespace attn {

template <int D>
static cudaError_t launch_bias(int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return bwd::launch<D, D, MASK_NONE, true>(maps, p, stream);
    case MASK_CAUSAL: return bwd::launch<D, D, MASK_CAUSAL, true>(maps, p, stream);
    case MASK_KEY_PADDING: return bwd::launch<D, D, MASK_KEY_PADDING, true>(maps, p, stream);
    case MASK_CAUSAL_KEY_PADDING: return bwd::launch<D, D, MASK_CAUSAL_KEY_PADDING, true>(maps, p, stream);
    case MASK_CAUSAL_CACHE: return bwd::launch<D, D, MASK_CAUSAL_CACHE, true>(maps, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_alibi(int d, int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    if (d == 64) return launch_bias<64>(mask, maps, p, stream);
    if (d == 128) return launch_bias<128>(mask, maps, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
