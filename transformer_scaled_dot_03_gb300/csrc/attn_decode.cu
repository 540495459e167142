// attn_decode.cu -- instantiations of the few-row (decoding) forward kernel.
#include "attn_kernel_decode.cuh"

namespace attn {

template <int DK, int DV>
static cudaError_t launch_rows(int rows, const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeParams& p,
                               cudaStream_t stream)
{
    switch (rows) {
    case 1: return dec::launch<DK, DV, 1>(tmK, tmV, p, stream);
    case 2: return dec::launch<DK, DV, 2>(tmK, tmV, p, stream);
    case 4: return dec::launch<DK, DV, 4>(tmK, tmV, p, stream);
    case 8: return dec::launch<DK, DV, 8>(tmK, tmV, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode(int d_k, int d_v, int rows, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const DecodeParams& p, cudaStream_t stream)
{
    if (d_k == 64 && d_v == 64) return launch_rows<64, 64>(rows, tmK, tmV, p, stream);
    if (d_k == 128 && d_v == 128) return launch_rows<128, 128>(rows, tmK, tmV, p, stream);
    if (d_k == 64 && d_v == 128) return launch_rows<64, 128>(rows, tmK, tmV, p, stream);
    if (d_k == 128 && d_v == 64) return launch_rows<128, 64>(rows, tmK, tmV, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
