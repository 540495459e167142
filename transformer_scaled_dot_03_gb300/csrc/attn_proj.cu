// attn_proj.cu -- instantiations of the projection GEMM around the attention.
#include "attn_kernel_proj.cuh"

namespace attn {

cudaError_t launch_proj(bool heads_in, bool heads_out, const ProjMaps& maps, const ProjParams& p, int num_sms,
                        cudaStream_t stream)
{
    if (!heads_in && heads_out) return proj::launch<false, true>(maps, p, num_sms, stream);
    if (heads_in && !heads_out) return proj::launch<true, false>(maps, p, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
