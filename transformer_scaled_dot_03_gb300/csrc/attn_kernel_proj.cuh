// attn_kernel_proj.cuh -- sm_103a GEMM for the projections around the attention:
// the input projections with the per-head split of their output, and the output
// projection that reads the heads merged.
//
// "从 RNN 到 Transformer（二）" §4.6 and "Transformer 详解" §4.2: the heads are
// W(x).view(B, n, h, d).transpose(1, 2), and after the attention the heads are put
// back side by side (out.transpose(1, 2).reshape(B, n, h d)) and multiplied by W_O.
// Both are Y = A Wᵀ (+ bias) with A [R = B·n rows, K] and W [N, K] in nn.Linear
// layout; what differs is where A comes from and where Y goes:
//
//   A_HEADS = false  A is a plain [R, K] matrix (the input x)
//   A_HEADS = true   A is the attention output O [B, H, n, d] read as [R, H·d]:
//                    each 64-column chunk of A is one head's slice, loaded as one
//                    128-row box of a 4-D tensor map when n is a multiple of 128
//                    (a row tile then lies in one batch entry), else as four
//                    32-row boxes (the merge costs nothing)
//   C_HEADS = false  Y is a plain [R, N] matrix
//   C_HEADS = true   Y's column block t (of width d_model) is written to output t
//                    in [B, H, n, d] (the split costs nothing: every 64-column,
//                    32-row piece of a tile goes to its head with a 4-D store)
//
// Persistent tcgen05 GEMM, 128 x 256 output tiles, K in chunks of 64:
//   warps 0-3  epilogue: tensor memory -> (+ bias) -> bf16 -> staging -> TMA store
//   warp  4    TMA producer (A and W chunks through a 4-stage ring)
//   warp  5    MMA issuer (M = 128, N = 256, K = 16 per instruction)
// Two 256-column accumulators in tensor memory: the epilogue of one tile runs
// while the next tile accumulates into the other.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "sm103a.cuh"

namespace attn {

using namespace sm103a;

namespace proj {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int ST_BYTES = 32 * BK * 2;           // one warp's staging piece: 32 rows x 64 bf16
constexpr int NUM_THREADS = 192;
constexpr int WARP_TMA = 4;
constexpr int WARP_MMA = 5;
constexpr int A_OFF = 0;
constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
constexpr int ST_OFF = B_OFF + STAGES * B_BYTES;  // 4 warps x 2 buffers
constexpr int BAR_OFF = ST_OFF + 4 * 2 * ST_BYTES;
constexpr int B_FULL = 0;
constexpr int B_EMPTY = STAGES;
constexpr int B_ACC_FULL = 2 * STAGES;
constexpr int B_ACC_EMPTY = B_ACC_FULL + 2;
constexpr int B_DRAIN = B_ACC_EMPTY + 2;        // every MMA issued is complete   (commit)
constexpr int B_NEVER = B_DRAIN + 1;            // debug: completed by nothing
constexpr int NBARS = B_NEVER + 1;
constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
constexpr int BYTES = MISC_OFF + 16 + 1024;
constexpr uint32_t TMEM_COLS = 512;
static_assert(BYTES <= 232448, "shared memory budget");

template <bool A_HEADS, bool C_HEADS>
__global__ void __launch_bounds__(NUM_THREADS, 1)
attn_proj_kernel(const __grid_constant__ ProjMaps maps, const ProjParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + BAR_OFF;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + MISC_OFF);
    volatile uint32_t* abort_word = reinterpret_cast<volatile uint32_t*>(smem + MISC_OFF + 4);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint64_t limit = p.watchdog_ns;
    const int num_tiles = p.tiles_m * p.tiles_n;
    const int nk = p.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(B_FULL + s), 1);
            mbar_init(bar(B_EMPTY + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(B_ACC_FULL + a), 1);
            mbar_init(bar(B_ACC_EMPTY + a), 128);
        }
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_NEVER), 1);
        *abort_word = 0u;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == WARP_TMA && lane == 0) {
        tma_prefetch_desc(&maps.a);
        tma_prefetch_desc(&maps.w);
        for (int t = 0; t < (C_HEADS ? 3 : 1); ++t) tma_prefetch_desc(&maps.c[t]);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_wait();   // nothing above reads global memory; A, W and the bias come after

    if (warp == WARP_TMA) {
        if (lane == 0) {
            // ================================================== TMA producer
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int m0 = (tile / p.tiles_n) * BM;
                const int n0 = (tile % p.tiles_n) * BN;
                // A_HEADS in 32-row boxes: the groups that hold rows (the rest of the smem
                // tile is never stored)
                const int groups = (A_HEADS && p.a_box_rows == 32) ? min(4, (p.R - m0 + 31) / 32) : 4;
                for (int kc = 0; kc < nk; ++kc, ++it) {
                    const int s = it % STAGES;
                    if (it >= STAGES &&
                        !mbar_wait(bar(B_EMPTY + s), static_cast<uint32_t>(it / STAGES - 1) & 1u, abort_word,
                                   p.status, STATUS_TMA_WAIT, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + A_OFF + s * A_BYTES;
                    mbar_arrive_expect_tx(bar(B_FULL + s), groups * ST_BYTES + B_BYTES);
                    if (A_HEADS) {
                        const int c = kc * BK;
                        const int h = c / p.d, j0 = c % p.d;
                        if (p.a_box_rows == 128) {
                            tma_load_4d(sa, &maps.a, bar(B_FULL + s), j0, m0 % p.n, h, m0 / p.n);
                        } else {
                            for (int g = 0; g < groups; ++g) {
                                const int r0 = m0 + 32 * g;
                                tma_load_4d(sa + g * ST_BYTES, &maps.a, bar(B_FULL + s), j0, r0 % p.n, h,
                                            r0 / p.n);
                            }
                        }
                    } else {
                        tma_load_3d(sa, &maps.a, bar(B_FULL + s), kc * BK, m0, 0);
                    }
                    tma_load_3d(sbase + B_OFF + s * B_BYTES, &maps.w, bar(B_FULL + s), kc * BK, n0, 0);
                }
            }
            // land every copy still in flight (only possible after an abort)
            for (int i = it - 1; i >= 0 && i >= it - STAGES; --i) {
                const uint32_t b = bar(B_FULL + i % STAGES);
                const uint32_t par = static_cast<uint32_t>(i / STAGES) & 1u;
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_test(b, par) && globaltimer_ns() - t0 < 100000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ================================================== MMA issuer (whole warp, one elected lane)
        constexpr uint32_t ID = idesc_bf16_f32(BM, BN, false, false);
        const uint64_t dA0 = sdesc_sw128(sbase + A_OFF, 16, 1024);
        const uint64_t dB0 = sdesc_sw128(sbase + B_OFF, 16, 1024);
        auto wait = [&](int b, uint32_t parity) -> bool {
            const bool r = mbar_wait(bar(b), parity, abort_word, p.status, STATUS_MMA_WAIT, limit);
            return __all_sync(0xffffffffu, r);
        };
        int it = 0, tl = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++tl) {
            const int acc = tl & 1;
            if (tl >= 2 && !wait(B_ACC_EMPTY + acc, static_cast<uint32_t>(tl / 2 - 1) & 1u)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
            for (int kc = 0; kc < nk; ++kc, ++it) {
                const int s = it % STAGES;
                if (!wait(B_FULL + s, static_cast<uint32_t>(it / STAGES) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t dA = dA0 + static_cast<uint64_t>((s * A_BYTES) >> 4);
                const uint64_t dB = dB0 + static_cast<uint64_t>((s * B_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    mma_ss_warp(d_tmem, dA + static_cast<uint64_t>((k * 32) >> 4),
                                dB + static_cast<uint64_t>((k * 32) >> 4), ID, (kc > 0 || k > 0) ? 1u : 0u);
                mma_commit_warp(bar(B_EMPTY + s));
            }
            if (!ok) break;
            mma_commit_warp(bar(B_ACC_FULL + acc));
        }
        // every MMA issued completes before the tensor memory is released (after an
        // abort some may still be running)
        mma_commit_warp(bar(B_DRAIN));
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_test(bar(B_DRAIN), 0) && globaltimer_ns() - t0 < 100000000ull) {
        }
        __syncwarp();
    } else {
        // ================================================== epilogue (warps 0-3, thread = row)
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        const uint32_t st0 = sbase + ST_OFF + static_cast<uint32_t>(warp) * 2 * ST_BYTES;
        int tl = 0, piece_count = 0;
        bool ok = true;
        if (p.debug_flags & DEBUG_FORCE_TIMEOUT) {
            ok = mbar_wait(bar(B_NEVER), 0, abort_word, p.status, STATUS_FORCED, 20000000ull);
            ok = __all_sync(0xffffffffu, ok);
        }
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++tl) {
            const int acc = tl & 1;
            const int m0 = (tile / p.tiles_n) * BM;
            const int n0 = (tile % p.tiles_n) * BN;
            ok = mbar_wait(bar(B_ACC_FULL + acc), static_cast<uint32_t>(tl / 2) & 1u, abort_word, p.status,
                           STATUS_SOFTMAX_WAIT, limit);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int r0 = m0 + 32 * warp;                   // first row of this warp's 32
#pragma unroll 1
            for (int q = 0; q < BN / BK; ++q) {
                const int c0 = n0 + q * BK;
                uint32_t a[32], b[32];
                tmem_ld32(tmem + lane_base + static_cast<uint32_t>(acc * BN + q * BK), a);
                tmem_ld32(tmem + lane_base + static_cast<uint32_t>(acc * BN + q * BK + 32), b);
                tmem_wait_ld();
                if (q == BN / BK - 1) {
                    tc_fence_before();
                    mbar_arrive(bar(B_ACC_EMPTY + acc));      // the accumulator may be reused
                }
                if (c0 >= p.N) continue;
                float bias[BK];
#pragma unroll
                for (int e = 0; e < BK; ++e) bias[e] = 0.f;
                if (p.bias != nullptr) {
#pragma unroll
                    for (int e = 0; e < BK / 2; ++e) {
                        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(p.bias + c0) + e);
                        bias[2 * e] = __uint_as_float(w << 16);
                        bias[2 * e + 1] = __uint_as_float(w & 0xFFFF0000u);
                    }
                }
                // this warp's staging buffer alternates; the store that used it two pieces
                // ago must have read it
                const uint32_t sb = st0 + static_cast<uint32_t>(piece_count & 1) * ST_BYTES;
                if (lane == 0 && piece_count >= 2) bulk_wait_group_read<1>();
                __syncwarp();
#pragma unroll
                for (int pc = 0; pc < 8; ++pc) {
                    const uint32_t* src = pc < 4 ? a : b;
                    const int e0 = 8 * (pc % 4);
                    uint32_t v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        v[e] = pack_bf16x2(__uint_as_float(src[e0 + 2 * e]) + bias[8 * pc + 2 * e],
                                           __uint_as_float(src[e0 + 2 * e + 1]) + bias[8 * pc + 2 * e + 1]);
                    const uint32_t addr = sb + lane * 128 +
                                          ((static_cast<uint32_t>(pc) ^ static_cast<uint32_t>(lane & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]),
                                 "r"(v[2]), "r"(v[3])
                                 : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (r0 < p.R) {
                        if (C_HEADS) {
                            const int t = c0 / p.d_block;
                            const int cc = c0 % p.d_block;
                            tma_store_4d(&maps.c[t], sb, cc % p.d, r0 % p.n, cc / p.d, r0 / p.n);
                        } else {
                            tma_store_3d(&maps.c[0], sb, c0, r0, 0);
                        }
                    }
                    bulk_commit_group();
                }
                ++piece_count;
                __syncwarp();
            }
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <bool A_HEADS, bool C_HEADS>
cudaError_t launch(const ProjMaps& maps, const ProjParams& p, int num_sms, cudaStream_t stream)
{
    auto kern = attn_proj_kernel<A_HEADS, C_HEADS>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BYTES);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int tiles = p.tiles_m * p.tiles_n;
    const int grid = tiles < num_sms ? tiles : num_sms;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(NUM_THREADS), BYTES, stream, maps, p);
}

}  // namespace proj
}  // namespace attn
