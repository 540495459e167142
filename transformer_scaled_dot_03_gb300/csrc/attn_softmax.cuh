// attn_softmax.cuh -- the per-tile softmax arithmetic of the forward kernels: one
// thread holds one query row's 128 scores of one key tile.
//
// For the row's scores s_c = q_i . k_(key0+c) ("Transformer 详解" §4.1: scores
// Q Kᵀ, scaled by 1/sqrt(d_k)), it applies the mask (keys past the row's column
// limit are -inf: the causal mask of §5.3, the key-padding mask of §3.4), adds
// the linear distance bias of "第2章：完整的 Transformer 架构" §5.3 when BIAS is
// set, and performs one step of the online softmax in the log2 domain: the
// running reference maximum m_ref is raised only when the tile's maximum exceeds
// it by more than 2^RESCALE_LOG2, the weights p_c = 2^(x_c - m_ref) are summed
// into l_run and packed to bf16 pairs for the P·V product, and alpha is the
// factor by which earlier partial outputs must be rescaled (1 when m_ref stays).
#pragma once

#include <cstdint>

#include "attn_internal.h"
#include "sm103a.cuh"

namespace attn {
namespace smx {

using namespace sm103a;

constexpr int BN = 128;
constexpr float LOG2E = 1.44269504088896341f;
// The reference maximum of a row is only raised when a new score exceeds it by
// more than 2^8; until then exp2(x - m_ref) <= 2^8, which bf16 P and the fp32
// sums hold as well as values <= 1, and O needs no rescaling.
constexpr float RESCALE_LOG2 = 8.0f;

// One 128-key tile of one row. s: the raw scores (overwritten). key0: the tile's
// first key. kv_len: keys past it are masked; qlim: under a causal mask the last
// key the row sees. sl2 = scale * log2(e); sb: the bias slope of the head times
// log2(e) (BIAS only). m_ref, l_run: the row's online-softmax state. Returns
// alpha; pk receives the 64 packed bf16 pairs of p.
template <int MASK, bool BIAS>
__device__ __forceinline__ float tile_step(float (&s)[BN], int key0, int kv_len, int qlim, float sl2, float sb,
                                           float& m_ref, float& l_run, uint32_t (&pk)[BN / 2])
{
    const bool need_mask = __any_sync(
        0xffffffffu, (key0 + BN > kv_len) || (mask_is_causal(MASK) && key0 + BN - 1 > qlim));
    if (need_mask) {
        // this row sees the tile's columns c < c_hi
        const int c_hi = (mask_is_causal(MASK) ? min(kv_len, qlim + 1) : kv_len) - key0;
#pragma unroll
        for (int c = 0; c < BN; ++c)
            if (c >= c_hi) s[c] = -INFINITY;
    }
    const uint64_t sl22 = f2_pack(sl2, sl2);
    if (BIAS) {
        // x_c = s_c * scale*log2e - sb |d0 - c|, d0 the row's key position
        // relative to the tile's first key
        const float d0 = static_cast<float>(qlim - key0);
        // Under a causal mask every column past d0 is already -inf, so the
        // left-side ramp serves the diagonal tile too.
        const bool left = mask_is_causal(MASK) || __all_sync(0xffffffffu, d0 >= static_cast<float>(BN - 1));
        const bool right = !left && __all_sync(0xffffffffu, d0 <= 0.f);
        if (left || right) {
            // the tile lies on one side of every row's diagonal: the bias is
            // sg (c - d0), stepped along four interleaved column ramps
            const float sg = left ? sb : -sb;
            uint64_t r2[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                r2[k] = f2_pack(sg * (static_cast<float>(2 * k) - d0), sg * (static_cast<float>(2 * k + 1) - d0));
            const uint64_t st2 = f2_pack(8.f * sg, 8.f * sg);
#pragma unroll
            for (int c = 0; c < BN / 2; ++c) {
                const uint64_t x2 = f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), sl22, r2[c % 4]);
                r2[c % 4] = f2_add(r2[c % 4], st2);
                f2_unpack(x2, s[2 * c], s[2 * c + 1]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < BN; ++c) s[c] = fmaf(-sb, fabsf(d0 - static_cast<float>(c)), s[c] * sl2);
        }
    }
    // row maximum: eight independent chains of three-input max
    float mx[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) mx[k] = fmaxf(s[2 * k], s[2 * k + 1]);
#pragma unroll
    for (int c = 16; c < BN; c += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = max3f(mx[k], s[c + 2 * k], s[c + 2 * k + 1]);
    // (with the bias the scores are already in the log2 domain)
    const float tile_max = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) *
                           (BIAS ? 1.f : sl2);
    const bool raise = tile_max > m_ref + RESCALE_LOG2;
    const float m_new = raise ? tile_max : m_ref;
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = raise ? ex2_approx(m_ref - m_use) : 1.f;

    // p = exp2(s * scale*log2e - m) on score pairs (packed fp32 arithmetic)
    const uint64_t mul2 = BIAS ? f2_pack(1.f, 1.f) : sl22;
    const uint64_t nm2 = f2_pack(-m_use, -m_use);
    uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int c = 0; c < BN / 2; ++c) {
        const uint64_t x2 = f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), mul2, nm2);
        float a, b;
        f2_unpack(x2, a, b);
        const uint64_t p2 = f2_pack(ex2_approx(a), ex2_approx(b));
        rs2[c % 4] = f2_add(rs2[c % 4], p2);
        float p0, p1;
        f2_unpack(p2, p0, p1);
        pk[c] = pack_bf16x2(p0, p1);
    }
    float r0, r1;
    f2_unpack(f2_add(f2_add(rs2[0], rs2[1]), f2_add(rs2[2], rs2[3])), r0, r1);
    l_run = l_run * alpha + (r0 + r1);
    m_ref = m_new;
    return alpha;
}

}  // namespace smx
}  // namespace attn
