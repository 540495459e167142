// attn_bwd_alibi.cu -- instantiations of the attention backward kernels with the
// linear distance bias (ALiBi, "第2章：完整的 Transformer 架构" §5.3), for head
// dims 64 and 128 (d_k != d_v included).
#include "attn_kernel_bwd.cuh"
#include "attn_kernel_bwd128.cuh"

namespace attn {

template <int DK, int DV>
static cudaError_t launch_bias(int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return bwd::launch<DK, DV, MASK_NONE, true>(maps, p, stream);
    case MASK_CAUSAL: return bwd::launch<DK, DV, MASK_CAUSAL, true>(maps, p, stream);
    case MASK_KEY_PADDING: return bwd::launch<DK, DV, MASK_KEY_PADDING, true>(maps, p, stream);
    case MASK_CAUSAL_KEY_PADDING: return bwd::launch<DK, DV, MASK_CAUSAL_KEY_PADDING, true>(maps, p, stream);
    case MASK_CAUSAL_CACHE: return bwd::launch<DK, DV, MASK_CAUSAL_CACHE, true>(maps, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

static cudaError_t launch_bias128(int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    switch (mask) {
    case MASK_NONE: return bwd128::launch<MASK_NONE, true>(maps, p, stream);
    case MASK_CAUSAL: return bwd128::launch<MASK_CAUSAL, true>(maps, p, stream);
    case MASK_KEY_PADDING: return bwd128::launch<MASK_KEY_PADDING, true>(maps, p, stream);
    case MASK_CAUSAL_KEY_PADDING: return bwd128::launch<MASK_CAUSAL_KEY_PADDING, true>(maps, p, stream);
    case MASK_CAUSAL_CACHE: return bwd128::launch<MASK_CAUSAL_CACHE, true>(maps, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_alibi(int d_k, int d_v, int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    if (d_k == 64 && d_v == 64) return launch_bias<64, 64>(mask, maps, p, stream);
    if (d_k == 128 && d_v == 128) return launch_bias128(mask, maps, p, stream);
    if (d_k == 64 && d_v == 128) return launch_bias<64, 128>(mask, maps, p, stream);
    if (d_k == 128 && d_v == 64) return launch_bias<128, 64>(mask, maps, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
