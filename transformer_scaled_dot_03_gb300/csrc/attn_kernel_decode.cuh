// attn_kernel_decode.cuh -- sm_103a attention forward for a few query rows
// against a long key/value sequence (decoding against a key/value cache).
//
// The same operation as the forward kernels ("Transformer 详解" §4.1-§4.2, the
// masks of §3.4 and §5.3): for n <= 8 query rows per (b, h) the work is reading
// K and V once, so the kernel is built around the memory system instead of the
// tensor cores. Keys are split into chunks of `split_len` (a multiple of 128);
// a CTA takes one (b, h, chunk), streams its K/V tiles of 128 keys through a
// TMA ring in shared memory and keeps an online softmax per query row:
//
//   warp 4       TMA producer (K and V tiles, 128 keys each)
//   warps 0-3    warp w takes keys [32w, 32w+32) of every tile: lane l scores key
//                32w + l against the rows (queries in shared memory, fp32), the
//                warp takes the row maximum with shuffles, and for P V each lane
//                owns d/32 output columns and receives the 32 weights by shuffle.
//
// At the end the four warps merge their (max, sum, O) in shared memory. With one
// chunk per (b, h) the CTA writes O (bf16) and LSE directly; otherwise it writes
// its partial (max and sum in the log2 domain, unnormalised O, fp32) and a
// second kernel merges the chunks: M = max_s m_s, L = sum_s l_s 2^(m_s - M),
// O = sum_s o_s 2^(m_s - M) / L, LSE = (M + log2 L) ln 2.
//
// With slopes (the linear distance bias of "第2章：完整的 Transformer 架构" §5.3,
// ALiBi) each score of row i and key j also gets -m_h |i + (m - n) - j|: one more
// FMA per score, which the memory-bound kernel absorbs.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "sm103a.cuh"

namespace attn {

using namespace sm103a;

namespace dec {

constexpr int TILE_KEYS = 128;
constexpr int CHUNK_BYTES = 128 * 64 * 2;   // 128 rows x 64 bf16 columns
constexpr int NQ_MAX = 8;
constexpr float LN2 = 0.693147180559945309f;
constexpr float LOG2E = 1.44269504088896341f;

// DK: query/key head dim, DV: value head dim, CTAS: CTAs per SM.
template <int DK, int DV, int CTAS>
struct Layout {
    static constexpr int CHK = DK / 64;
    static constexpr int CHV = DV / 64;
    static constexpr int TILE_K = CHK * CHUNK_BYTES;        // 128 keys x DK
    static constexpr int TILE_V = CHV * CHUNK_BYTES;        // 128 keys x DV
    static constexpr bool SMALL = DK == 64 && DV == 64;
    // Two or three CTAs per SM: with d = 128 a 128-key stage is 64 KB, so each CTA
    // holds one (the CTAs' loads and consumers interleave). At three the merge area
    // shares the key stage, which no copy writes once the last tile is consumed.
    static constexpr int STAGES = SMALL ? 3 : 1;
    static constexpr int NUM_THREADS = 160;
    static constexpr int WARP_TMA = 4;
    static constexpr int CTAS_PER_SM = CTAS;
    static constexpr bool RED_IN_STAGE = CTAS == 3;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + STAGES * TILE_K;
    static constexpr int Q_OFF = V_OFF + STAGES * TILE_V;    // fp32 [NQ_MAX][DK]
    static constexpr int RED_WARP = (2 * NQ_MAX + NQ_MAX * DV) * 4;
    // per warp: m, l [NQ_MAX] then O [NQ_MAX][DV]
    static constexpr int RED_OFF = RED_IN_STAGE ? K_OFF : Q_OFF + NQ_MAX * DK * 4;
    static constexpr int BAR_OFF = RED_IN_STAGE ? Q_OFF + NQ_MAX * DK * 4 : RED_OFF + 4 * RED_WARP;
    static_assert(!RED_IN_STAGE || 4 * RED_WARP <= STAGES * TILE_K, "merge area inside the key stage");
    static constexpr int B_FULL = 0;
    static constexpr int B_EMPTY = STAGES;
    static constexpr int B_NEVER = 2 * STAGES;               // debug: completed by nothing
    static constexpr int NBARS = B_NEVER + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BYTES = MISC_OFF + 16 + 1024;
    static_assert(BYTES * CTAS_PER_SM <= 232448, "shared memory budget");
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Byte offset of element (row, col) in a 128-row tile stored as 64-column chunks
// with the TMA 128-byte swizzle (16-byte pieces permuted by row % 8).
__device__ __forceinline__ uint32_t tile_off(int row, int col)
{
    return static_cast<uint32_t>((col / 64) * CHUNK_BYTES + row * 128 +
                                 ((((col % 64) / 8) ^ (row & 7)) << 4) + (col % 8) * 2);
}

template <int DK, int DV, int NQ>
__global__ void __launch_bounds__(160, decode_ctas_per_sm(DK, DV, NQ))
attn_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const DecodeParams p)
{
    using L = Layout<DK, DV, decode_ctas_per_sm(DK, DV, NQ)>;
    static_assert(L::NUM_THREADS == 160, "launch bounds");
    griddep_wait();   // the previous grid's writes (Q, the cache, the lengths) are visible
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::BAR_OFF;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
    volatile uint32_t* abort_word = reinterpret_cast<volatile uint32_t*>(smem + L::MISC_OFF);
    float* sq = reinterpret_cast<float*>(smem + L::Q_OFF);
    float* sred = reinterpret_cast<float*>(smem + L::RED_OFF);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int split = static_cast<int>(blockIdx.x) % p.num_splits;
    const int bh = static_cast<int>(blockIdx.x) / p.num_splits;
    const uint64_t limit = p.watchdog_ns;

    // keys this CTA covers: [j0, j1), cut to the last key any row can see
    int kv_len = p.m;
    if (mask_has_lengths(p.mask)) {
        const int len = __ldg(p.key_lengths + bh / p.H);
        kv_len = len < 0 ? 0 : (len > p.m ? p.m : len);
    }
    int last = kv_len;                                   // one past the last visible key
    const int off = causal_offset(p.mask, p.causal_off, kv_len, p.n);   // row i sits at key position i + off
    if (mask_is_causal(p.mask)) last = min(last, max(0, p.n - 1 + off + 1));
    const int j0 = split * p.split_len;
    const int j1 = min(j0 + p.split_len, last);
    const int ntiles = j1 > j0 ? (j1 - j0 + TILE_KEYS - 1) / TILE_KEYS : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(bar(L::B_FULL + s), 1);
            mbar_init(bar(L::B_EMPTY + s), 4);
        }
        mbar_init(bar(L::B_NEVER), 1);
        *abort_word = 0u;
        fence_mbar_init();
    }
    // queries as fp32 (rows >= n are zero)
    for (int e = threadIdx.x; e < NQ * DK; e += blockDim.x) {
        const int i = e / DK, c = e % DK;
        float v = 0.f;
        if (i < p.n) {
            const uint16_t b = p.Q[(static_cast<int64_t>(bh) * p.n + i) * DK + c];
            v = __uint_as_float(static_cast<uint32_t>(b) << 16);
        }
        sq[i * DK + c] = v;
    }
    __syncthreads();

    if (warp == L::WARP_TMA) {
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int issued = 0;
            for (int t = 0; t < ntiles; ++t) {
                const int s = t % L::STAGES;
                if (t >= L::STAGES &&
                    !mbar_wait(bar(L::B_EMPTY + s), static_cast<uint32_t>(t / L::STAGES - 1) & 1u, abort_word,
                               p.status, STATUS_TMA_WAIT, limit))
                    break;
                const int key0 = j0 + t * TILE_KEYS;
                mbar_arrive_expect_tx(bar(L::B_FULL + s), L::TILE_K + L::TILE_V);
                for (int c = 0; c < L::CHK; ++c)
                    tma_load_3d(sbase + L::K_OFF + s * L::TILE_K + c * CHUNK_BYTES, &tmK, bar(L::B_FULL + s), c * 64,
                                key0, bh);
                for (int c = 0; c < L::CHV; ++c)
                    tma_load_3d(sbase + L::V_OFF + s * L::TILE_V + c * CHUNK_BYTES, &tmV, bar(L::B_FULL + s), c * 64,
                                key0, bh);
                ++issued;
            }
            // land every copy still in flight (only possible after an abort)
            for (int t = issued - 1; t >= 0 && t >= issued - L::STAGES; --t) {
                const uint32_t b = bar(L::B_FULL + t % L::STAGES);
                const uint32_t par = static_cast<uint32_t>(t / L::STAGES) & 1u;
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_test(b, par) && globaltimer_ns() - t0 < 100000000ull) {
                }
            }
        }
        return;
    }

    // ================================================== consumers (warps 0-3)
    constexpr int CPL = DV / 32;           // output columns per lane
    float m_run[NQ], l_run[NQ], o[NQ][CPL];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) o[i][c] = 0.f;
    }
    const float sl2 = p.scale_log2;
    // distance-bias slope of the head in the log2 domain (0: no bias)
    const float sb = p.slopes != nullptr ? __ldg(p.slopes + bh % p.H) * LOG2E : 0.f;
    const int row = 32 * warp + lane;       // this lane's key row within a tile
    bool ok = true;
    if (p.debug_flags & DEBUG_FORCE_TIMEOUT) {
        ok = mbar_wait(bar(L::B_NEVER), 0, abort_word, p.status, STATUS_FORCED, 20000000ull);
        ok = __all_sync(0xffffffffu, ok);
    }
    for (int t = 0; ok && t < ntiles; ++t) {
        const int s = t % L::STAGES;
        ok = mbar_wait(bar(L::B_FULL + s), static_cast<uint32_t>(t / L::STAGES) & 1u, abort_word, p.status,
                       STATUS_SOFTMAX_WAIT, limit);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint8_t* kt = smem + L::K_OFF + s * L::TILE_K;
        const uint8_t* vt = smem + L::V_OFF + s * L::TILE_V;
        const int key = j0 + t * TILE_KEYS + row;

        // scores of this lane's key against every row
        float sc[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) sc[i] = 0.f;
#pragma unroll 4
        for (int c8 = 0; c8 < DK / 8; ++c8) {
            const uint4 kv = *reinterpret_cast<const uint4*>(kt + tile_off(row, 8 * c8));
            const float k[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                                bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                const float4 qa = *reinterpret_cast<const float4*>(sq + i * DK + 8 * c8);
                const float4 qb = *reinterpret_cast<const float4*>(sq + i * DK + 8 * c8 + 4);
                float a = sc[i];
                a = fmaf(qa.x, k[0], a);
                a = fmaf(qa.y, k[1], a);
                a = fmaf(qa.z, k[2], a);
                a = fmaf(qa.w, k[3], a);
                a = fmaf(qb.x, k[4], a);
                a = fmaf(qb.y, k[5], a);
                a = fmaf(qb.z, k[6], a);
                a = fmaf(qb.w, k[7], a);
                sc[i] = a;
            }
        }
        // mask, online softmax (log2 domain)
        float pr[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            const bool vis = key < j1 && (!mask_is_causal(p.mask) || key <= i + off);
            const float x =
                vis ? fmaf(-sb, fabsf(static_cast<float>(i + off - key)), sc[i] * sl2) : -INFINITY;
            float mx = x;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m_run[i], mx);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = ex2_approx(m_run[i] - m_use);
            pr[i] = ex2_approx(x - m_use);
            l_run[i] = l_run[i] * alpha + pr[i];
#pragma unroll
            for (int c = 0; c < CPL; ++c) o[i][c] *= alpha;
            m_run[i] = m_new;
        }
        // O += P V: lane owns columns [CPL*lane, CPL*lane + CPL)
#pragma unroll 4
        for (int jj = 0; jj < 32; ++jj) {
            const int vrow = 32 * warp + jj;
            float v[CPL];
            if (CPL == 4) {
                const uint2 vv = *reinterpret_cast<const uint2*>(vt + tile_off(vrow, 4 * lane));
                v[0] = bf16_lo(vv.x);
                v[1] = bf16_hi(vv.x);
                v[2] = bf16_lo(vv.y);
                v[3] = bf16_hi(vv.y);
            } else {
                const uint32_t vv = *reinterpret_cast<const uint32_t*>(vt + tile_off(vrow, 2 * lane));
                v[0] = bf16_lo(vv);
                v[1] = bf16_hi(vv);
            }
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                const float pj = __shfl_sync(0xffffffffu, pr[i], jj);
#pragma unroll
                for (int c = 0; c < CPL; ++c) o[i][c] = fmaf(pj, v[c], o[i][c]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::B_EMPTY + s));
    }

    // ---------------------------------------------- merge the four warps
    // (the merge area may be the key stage: every warp must be done with the last tile)
    if (L::RED_IN_STAGE) asm volatile("bar.sync 1, 128;" ::: "memory");
    float* red = sred + warp * (L::RED_WARP / 4);
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        float l = l_run[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0) {
            red[i] = m_run[i];
            red[NQ_MAX + i] = l;
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) red[2 * NQ_MAX + i * DV + CPL * lane + c] = o[i][c];
    }
    // the producer warp has returned: synchronise the four consumer warps only
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const int rows = min(p.n, NQ);
    for (int e = threadIdx.x; e < rows * DV; e += 128) {
        const int i = e / DV, c = e % DV;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, sred[w * (L::RED_WARP / 4) + i]);
        const float M_use = M == -INFINITY ? 0.f : M;
        float Lsum = 0.f, Oc = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float* rw = sred + w * (L::RED_WARP / 4);
            const float f = ex2_approx(rw[i] - M_use);
            Lsum = fmaf(rw[NQ_MAX + i], f, Lsum);
            Oc = fmaf(rw[2 * NQ_MAX + i * DV + c], f, Oc);
        }
        const int64_t orow = static_cast<int64_t>(bh) * p.n + i;
        if (p.num_splits == 1) {
            const float out = Lsum > 0.f ? Oc / Lsum : 0.f;
            const uint32_t pk = pack_bf16x2(out, 0.f);
            p.O[orow * DV + c] = static_cast<uint16_t>(pk & 0xFFFFu);
            if (c == 0 && p.LSE != nullptr) p.LSE[orow] = Lsum > 0.f ? (M + __log2f(Lsum)) * LN2 : -INFINITY;
        } else {
            const int64_t prow = (static_cast<int64_t>(bh) * p.num_splits + split) * p.n + i;
            p.part_o[prow * DV + c] = Oc;
            if (c == 0) {
                p.part_ml[2 * prow] = M;
                p.part_ml[2 * prow + 1] = Lsum;
            }
        }
    }
}

// Merge of the chunks of one (b, h, row): one thread per output column.
template <int D>
__global__ void __launch_bounds__(D)
attn_decode_combine_kernel(const DecodeParams p)
{
    griddep_wait();   // the partial results of the chunk kernel are visible
    const int64_t r = blockIdx.x;                 // (b*H + h) * n + i
    const int64_t bh = r / p.n, i = r % p.n;
    const int c = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < p.num_splits; ++s) M = fmaxf(M, p.part_ml[2 * ((bh * p.num_splits + s) * p.n + i)]);
    const float M_use = M == -INFINITY ? 0.f : M;
    float Lsum = 0.f, Oc = 0.f;
    for (int s = 0; s < p.num_splits; ++s) {
        const int64_t prow = (bh * p.num_splits + s) * p.n + i;
        const float f = ex2_approx(p.part_ml[2 * prow] - M_use);
        Lsum = fmaf(p.part_ml[2 * prow + 1], f, Lsum);
        Oc = fmaf(p.part_o[prow * D + c], f, Oc);
    }
    const float out = Lsum > 0.f ? Oc / Lsum : 0.f;
    p.O[r * D + c] = static_cast<uint16_t>(pack_bf16x2(out, 0.f) & 0xFFFFu);
    if (c == 0 && p.LSE != nullptr) p.LSE[r] = Lsum > 0.f ? (M + __log2f(Lsum)) * LN2 : -INFINITY;
}

template <int DK, int DV, int NQ>
cudaError_t launch(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeParams& p, cudaStream_t stream)
{
    using L = Layout<DK, DV, decode_ctas_per_sm(DK, DV, NQ)>;
    auto kern = attn_decode_kernel<DK, DV, NQ>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int64_t grid = static_cast<int64_t>(p.B) * p.H * p.num_splits;
    e = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(L::NUM_THREADS), L::BYTES, stream, tmK, tmV, p);
    if (e != cudaSuccess || p.num_splits == 1) return e;
    return launch_pdl(attn_decode_combine_kernel<DV>, dim3(static_cast<unsigned>(static_cast<int64_t>(p.B) * p.H * p.n)),
                      dim3(DV), 0, stream, p);
}

}  // namespace dec
}  // namespace attn
