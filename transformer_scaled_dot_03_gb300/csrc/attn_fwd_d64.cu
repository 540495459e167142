// attn_fwd_d64.cu -- instantiations of the attention forward kernels for head dim 64.
#include "attn_kernel.cuh"
#include "attn_kernel_dp.cuh"

namespace attn {

template <int NT>
static cudaError_t launch_nt(int mask, const TensorMaps& maps, const FwdParams& p, int64_t num_ctas,
                             cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return launch_fwd<64, MASK_NONE, NT>(maps, p, num_ctas, stream);
    case MASK_CAUSAL: return launch_fwd<64, MASK_CAUSAL, NT>(maps, p, num_ctas, stream);
    case MASK_KEY_PADDING: return launch_fwd<64, MASK_KEY_PADDING, NT>(maps, p, num_ctas, stream);
    default: return cudaErrorInvalidValue;
    }
}

static cudaError_t launch_dp(int mask, const TensorMaps& maps, const FwdParams& p, int num_sms,
                             cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return dp::launch<64, 64, MASK_NONE>(maps, p, num_sms, stream);
    case MASK_CAUSAL: return dp::launch<64, 64, MASK_CAUSAL>(maps, p, num_sms, stream);
    case MASK_KEY_PADDING: return dp::launch<64, 64, MASK_KEY_PADDING>(maps, p, num_sms, stream);
    case MASK_CAUSAL_KEY_PADDING:
        return dp::launch<64, 64, MASK_CAUSAL_KEY_PADDING>(maps, p, num_sms, stream);
    case MASK_CAUSAL_CACHE: return dp::launch<64, 64, MASK_CAUSAL_CACHE>(maps, p, num_sms, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_fwd_d64(int mask, int variant, const TensorMaps& maps, const FwdParams& p,
                           int64_t num_ctas, int num_sms, cudaStream_t stream)
{
    switch (variant) {
    case KERNEL_DP: return launch_dp(mask, maps, p, num_sms, stream);
    case KERNEL_NT1: return launch_nt<1>(mask, maps, p, num_ctas, stream);
    default: return launch_nt<2>(mask, maps, p, num_ctas, stream);
    }
}

}  // namespace attn
