// attn_internal.h -- declarations shared by the host launcher (attn_api.cu) and
// the kernel translation units. Not part of the public C ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

enum { MASK_NONE = 0, MASK_CAUSAL = 1, MASK_KEY_PADDING = 2, MASK_CAUSAL_KEY_PADDING = 3, MASK_CAUSAL_CACHE = 4 };

__host__ __device__ constexpr bool mask_is_causal(int mask)
{
    return mask == MASK_CAUSAL || mask == MASK_CAUSAL_KEY_PADDING || mask == MASK_CAUSAL_CACHE;
}
__host__ __device__ constexpr bool mask_has_lengths(int mask)
{
    return mask == MASK_KEY_PADDING || mask == MASK_CAUSAL_KEY_PADDING || mask == MASK_CAUSAL_CACHE;
}
// Offset of a query row's position among the keys (row i sits at i + offset): the
// n queries are the last n of the m keys, or of the kv_len filled keys of each
// entry's cache under MASK_CAUSAL_CACHE.
__host__ __device__ constexpr int causal_offset(int mask, int m_minus_n, int kv_len, int n)
{
    return mask == MASK_CAUSAL_CACHE ? kv_len - n : m_minus_n;
}

// Bits of the device status word: which bounded wait gave up.
enum : uint32_t {
    STATUS_TMA_WAIT = 1u,      // producer waiting for a free K/V stage
    STATUS_MMA_WAIT = 2u,      // MMA issuer waiting for data or for P
    STATUS_SOFTMAX_WAIT = 4u,  // softmax/epilogue waiting for S or O
    STATUS_FORCED = 8u,        // debug: wait on a barrier that nothing completes
};

enum : uint32_t { DEBUG_FORCE_TIMEOUT = 1u };

struct FwdParams {
    int B, H, n, m;
    int causal_off;               // m - n: query row i sees keys j <= i + causal_off (causal masks)
    int num_qblocks;              // ceil(n / rows per work unit)
    int num_units;                // work units (query tiles, paired under the causal masks)
    void* O;                      // bf16 [B,H,n,d_v] (persistent kernel stores rows directly)
    const int32_t* key_lengths;   // device int32 [B] (key-padding masks only)
    float scale_log2;             // scale * log2(e)
    float* LSE;                   // fp32 [B,H,n] or null
    const float* slopes;          // fp32 [H]: distance-bias slope per head (bias kernels only)
    uint32_t* status;             // device status word
    uint64_t watchdog_ns;         // wall-clock limit of one bounded wait
    uint32_t debug_flags;
};

struct TensorMaps {
    CUtensorMap q, k, v, o;
};

// Launches `kern` with programmatic stream serialization: the grid may start
// before the previous kernel in the stream has finished. Every kernel launched
// this way executes griddepcontrol.wait before its first global-memory access,
// so it still sees all the previous kernel's writes; what overlaps is the
// launch itself and the set-up before that wait.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Backward (attn_kernel_bwd.cuh): one CTA per (b, h, 128-key tile).
struct BwdParams {
    int B, H, n, m;
    int causal_off;               // m - n
    int num_kblocks;              // ceil(m / 128)
    int n_pad;                    // query rows padded to whole tiles (lse2 / dd row stride)
    int num_sms;                  // sizes the persistent grid (d = 64)
    const int32_t* key_lengths;   // device int32 [B] (key-padding masks only)
    const float* lse2;            // [B*H, n_pad]: LSE * log2(e), 0 in the padding
    const float* dd;              // [B*H, n_pad]: D = rowsum(dO * O), 0 in the padding
    void* dK;                     // bf16 [B,H,m,d] (plain stores for key tiles no query sees)
    void* dV;
    float scale_log2;             // scale * log2(e)
    float scale;
    const float* slopes;          // fp32 [H]: distance-bias slope per head (bias kernels only)
    uint32_t* status;
    uint64_t watchdog_ns;
    uint32_t debug_flags;
};

struct BwdMaps {
    CUtensorMap q, k, v, dout, dk, dv, dq_acc;
};

cudaError_t launch_bwd_d64(int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_d128(int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream);
// Backward for d_k != d_v (64 and 128 either way round).
cudaError_t launch_bwd_dmix(int d_k, int d_v, int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream);
// Backward with the linear distance bias (p.slopes), d_k, d_v in {64, 128}.
cudaError_t launch_bwd_alibi(int d_k, int d_v, int mask, const BwdMaps& maps, const BwdParams& p, cudaStream_t stream);

// Few-row forward (attn_kernel_decode.cuh): one CTA per (b, h, key chunk).
// CTAs per SM of its kernel: three at d_k = 128 with one or two query rows (the
// merge area then shares the key stage; the kernel fits 136 registers), else two.
__host__ __device__ constexpr int decode_ctas_per_sm(int d_k, int d_v, int rows)
{
    return (d_k == 64 && d_v == 64) ? 2 : (d_k == 128 && rows <= 2 ? 3 : 2);
}

struct DecodeParams {
    const uint16_t* Q;            // bf16 [B,H,n,d_k]
    int B, H, n, m;
    int causal_off;               // m - n
    int mask;
    const int32_t* key_lengths;   // device int32 [B] (key-padding masks only)
    float scale_log2;             // scale * log2(e)
    int split_len;                // keys per chunk (multiple of 128)
    int num_splits;               // chunks per (b, h)
    uint16_t* O;                  // bf16 [B,H,n,d_v]
    float* LSE;                   // fp32 [B,H,n] or null
    float* part_o;                // fp32 [B*H, num_splits, n, d_v] (num_splits > 1)
    float* part_ml;               // fp32 [B*H, num_splits, n, 2]: max (log2 domain), sum
    const float* slopes;          // fp32 [H]: distance-bias slope per head, or null (no bias)
    uint32_t* status;
    uint64_t watchdog_ns;
    uint32_t debug_flags;
};

// rows: the kernel variant handles n <= rows (1, 2, 4 or 8).
cudaError_t launch_decode(int d_k, int d_v, int rows, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const DecodeParams& p, cudaStream_t stream);

// Projections around the attention (attn_kernel_proj.cuh): Y = A Wᵀ (+ bias).
struct ProjParams {
    int R, N, K;                  // rows (B*n), output columns, reduction length
    int n, H, d;                  // rows per batch entry, heads, head dim (head-shaped operands)
    int d_block;                  // output columns per head-split output (d_model)
    int a_box_rows;               // head-shaped A: rows per 4-D load box (128 when n % 128 == 0, else 32)
    int tiles_m, tiles_n;
    const uint16_t* bias;         // bf16 [N] or null
    uint32_t* status;
    uint64_t watchdog_ns;
    uint32_t debug_flags;
};

struct ProjMaps {
    CUtensorMap a, w, c[3];
};

// heads_in: A is O [B,H,n,d] read merged; heads_out: Y split per head into c[0..2].
cudaError_t launch_proj(bool heads_in, bool heads_out, const ProjMaps& maps, const ProjParams& p, int num_sms,
                        cudaStream_t stream);

// The persistent forward kernel; num_sms sizes its grid.
cudaError_t launch_fwd_d64(int mask, const TensorMaps& maps, const FwdParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_fwd_d128(int mask, const TensorMaps& maps, const FwdParams& p, int num_sms, cudaStream_t stream);
// d_k != d_v (64 and 128 either way round).
cudaError_t launch_fwd_dmix(int d_k, int d_v, int mask, const TensorMaps& maps, const FwdParams& p,
                            int num_sms, cudaStream_t stream);
// Forward with the linear distance bias (p.slopes), d_k, d_v in {64, 128}.
cudaError_t launch_fwd_alibi(int d_k, int d_v, int mask, const TensorMaps& maps, const FwdParams& p, int num_sms,
                             cudaStream_t stream);

}  // namespace attn
