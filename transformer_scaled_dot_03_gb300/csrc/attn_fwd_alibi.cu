// attn_fwd_alibi.cu -- instantiations of the persistent attention forward kernel
// with the linear distance bias (ALiBi, "第2章：完整的 Transformer 架构" §5.3),
// for head dims d_k = d_v = 64 and 128.
#include "attn_kernel_dp.cuh"

namespace attn {

template <int D>
static cudaError_t launch_bias(int mask, const TensorMaps& maps, const FwdParams& p, int num_sms,
                               cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return dp::launch<D, D, MASK_NONE, true>(maps, p, num_sms, stream);
    case MASK_CAUSAL: return dp::launch<D, D, MASK_CAUSAL, true>(maps, p, num_sms, stream);
    case MASK_KEY_PADDING: return dp::launch<D, D, MASK_KEY_PADDING, true>(maps, p, num_sms, stream);
    case MASK_CAUSAL_KEY_PADDING: return dp::launch<D, D, MASK_CAUSAL_KEY_PADDING, true>(maps, p, num_sms, stream);
    case MASK_CAUSAL_CACHE: return dp::launch<D, D, MASK_CAUSAL_CACHE, true>(maps, p, num_sms, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_fwd_alibi(int d, int mask, const TensorMaps& maps, const FwdParams& p, int num_sms,
                             cudaStream_t stream)
{
    if (d == 64) return launch_bias<64>(mask, maps, p, num_sms, stream);
    if (d == 128) return launch_bias<128>(mask, maps, p, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
