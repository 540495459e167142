// attn_kernel_bwd.cuh -- sm_103a attention backward: dK, dV and the dQ partial
// sums of one 128-key tile per CTA.
//
// The gradient of the scaled dot-product attention of "Transformer 详解"
// §4.1-§4.2 (with the masks of §3.4 and §5.3) for an upstream gradient dO,
// with the weights recomputed from the saved LSE instead of stored:
//
//   P   = exp(scale * Q Kᵀ - LSE)          (0 where masked)
//   dV  = Pᵀ dO
//   dP  = dO Vᵀ,   dS = P ∘ (dP - D),  D_i = dO_i · O_i
//   dK  = scale * dSᵀ Q,   dQ = scale * dS K
//
// A CTA holds one 128-key tile of one (b, h) pair (K and V stay in shared
// memory) and walks the 128-row query tiles that can see it. The tensor cores
// compute the transposed tiles Sᵀ = K Qᵀ and dPᵀ = V dOᵀ, so that a TMEM lane
// is a key: the four softmax warps (thread = key) turn them into Pᵀ and dSᵀ
// (bf16, written back over Sᵀ and dPᵀ) and into dS in shared memory, and the
// tensor cores accumulate dV += Pᵀ dO and dK += dSᵀ Q with A taken from tensor
// memory, and compute the tile's dQ = dS K with dS read MN-major from shared
// memory. dQ leaves through a staging tile and a TMA reduce-add into an fp32
// accumulator in global memory (every key tile of the head adds to it). D and
// LSE·log2(e) come from a preparation kernel, padded to whole query tiles.
//
//   warps 0-3   Pᵀ/dSᵀ (thread = key), dQ read-out (thread = query), dK/dV epilogue
//   warp  4     TMA producer: K and V once, then Q, dO, LSE, D per query tile
//   warp  5     tcgen05.mma issuer, owns the TMEM allocation
//   warps 6-7   idle
// Tensor memory (512 columns): Sᵀ [0,128) then Pᵀ [0,64); dPᵀ [128,256) then dSᵀ
// [128,192); dV [256,256+d); dK [256+d,256+2d); dQ at d = 64 in [384,448), at
// d = 128 as two 64-column halves in [64,128) and [192,256).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "sm103a.cuh"

namespace attn {

using namespace sm103a;

namespace bwd {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // keys per CTA
constexpr int CHUNK_BYTES = 128 * 64 * 2;

template <int D>
struct Layout {
    static constexpr int CH = D / 64;
    static constexpr int TILE = CH * CHUNK_BYTES;        // a 128 x D bf16 tile
    static constexpr int NUM_THREADS = 256;
    static constexpr int WARP_TMA = 4;
    static constexpr int WARP_MMA = 5;
    static constexpr int QS = D == 64 ? 2 : 1;             // Q/dO/LSE/D ring depth
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + TILE;
    static constexpr int Q_OFF = V_OFF + TILE;
    static constexpr int DO_OFF = Q_OFF + QS * TILE;
    static constexpr int DS_OFF = DO_OFF + QS * TILE;      // dS (bf16, MN-major) / staging, 32 KB
    static constexpr int LSE_OFF = DS_OFF + 2 * CHUNK_BYTES;
    static constexpr int DD_OFF = LSE_OFF + QS * BM * 4;
    static constexpr int BAR_OFF = DD_OFF + QS * BM * 4;
    static constexpr int B_KVFULL = 0;
    static constexpr int B_QFULL = 1;
    static constexpr int B_QEMPTY = B_QFULL + QS;
    static constexpr int B_SFULL = B_QEMPTY + QS;   // Sᵀ and dPᵀ computed        (commit)
    static constexpr int B_PFULL = B_SFULL + 1;     // Pᵀ, dSᵀ and dS written     (128 arrivals)
    static constexpr int B_DQFULL = B_PFULL + 1;    // dQ of the tile computed    (commit)
    static constexpr int B_DQFREE = B_DQFULL + 1;   // dQ read out of TMEM        (128 arrivals)
    static constexpr int B_TILEDONE = B_DQFREE + 1; // every MMA of the tile done (commit)
    static constexpr int B_DKVDONE = B_TILEDONE + 1;
    static constexpr int B_NEVER = B_DKVDONE + 1;
    static constexpr int NBARS = B_NEVER + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BYTES = MISC_OFF + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0, DP_COL = 128, P_COL = 0, DS_COL = 128;
    static constexpr uint32_t DV_COL = 256, DK_COL = 256 + D;
    static constexpr bool DQ_OVER_S = D == 128;            // dQ halves reuse the upper Sᵀ/dPᵀ columns
    __host__ __device__ static constexpr uint32_t dq_col(int h) { return DQ_OVER_S ? (h == 0 ? 64u : 192u) : 384u; }
    static_assert(DK_COL + D <= TMEM_COLS, "tensor memory layout");
    static_assert(BYTES <= 232448, "shared memory budget");
};

__device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_test(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

template <int D, int MASK>
__global__ void __launch_bounds__(Layout<D>::NUM_THREADS, 1)
attn_bwd_kernel(const __grid_constant__ BwdMaps maps, const BwdParams p)
{
    using L = Layout<D>;
    const int kb = static_cast<int>(blockIdx.x) % p.num_kblocks;
    const int bh = static_cast<int>(blockIdx.x) / p.num_kblocks;
    const int k0 = kb * BN;
    int kv_len = p.m;
    if (mask_has_lengths(MASK)) {
        const int len = __ldg(p.key_lengths + bh / p.H);
        kv_len = len < 0 ? 0 : (len > p.m ? p.m : len);
    }
    if (k0 >= kv_len) {
        // no query sees these keys: their gradients are zero
        const int rows = min(BN, p.m - k0);
        const int64_t base = (static_cast<int64_t>(bh) * p.m + k0) * D;
        uint4* gk = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dK) + base);
        uint4* gv = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dV) + base);
        for (int i = threadIdx.x; i < rows * D / 8; i += blockDim.x) {
            gk[i] = make_uint4(0u, 0u, 0u, 0u);
            gv[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        return;
    }
    // query tiles that can see this key tile
    const int nqb = (p.n + BM - 1) / BM;
    int qb_lo = 0;
    if (mask_is_causal(MASK)) {
        const int first_q = k0 - p.causal_off;     // first row that sees key k0
        qb_lo = first_q <= 0 ? 0 : first_q / BM;
    }
    const int nt = nqb - qb_lo;                    // >= 1: the last row sees every key < kv_len

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::BAR_OFF;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
    volatile uint32_t* abort_word = reinterpret_cast<volatile uint32_t*>(smem + L::MISC_OFF + 4);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint64_t limit = p.watchdog_ns;

    if (threadIdx.x == 0) {
        mbar_init(bar(L::B_KVFULL), 1);
        for (int s = 0; s < L::QS; ++s) {
            mbar_init(bar(L::B_QFULL + s), 1);
            mbar_init(bar(L::B_QEMPTY + s), 1);
        }
        mbar_init(bar(L::B_SFULL), 1);
        mbar_init(bar(L::B_PFULL), BN);
        mbar_init(bar(L::B_DQFULL), 1);
        mbar_init(bar(L::B_DQFREE), BN);
        mbar_init(bar(L::B_TILEDONE), 1);
        mbar_init(bar(L::B_DKVDONE), 1);
        mbar_init(bar(L::B_NEVER), 1);
        *abort_word = 0u;
        fence_mbar_init();
    }
    if (warp == L::WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == L::WARP_TMA && lane == 0) {
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
        tma_prefetch_desc(&maps.dout);
        tma_prefetch_desc(&maps.dk);
        tma_prefetch_desc(&maps.dv);
        tma_prefetch_desc(&maps.dq_acc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const uint32_t sK = sbase + L::K_OFF;
    const uint32_t sV = sbase + L::V_OFF;
    const uint32_t sQ = sbase + L::Q_OFF;
    const uint32_t sdO = sbase + L::DO_OFF;
    const uint32_t sdS = sbase + L::DS_OFF;

    if (warp >= 4) {
        if (warp == L::WARP_TMA && lane == 0) {
            // ================================================== TMA producer
            mbar_arrive_expect_tx(bar(L::B_KVFULL), 2 * L::TILE);
            for (int c = 0; c < L::CH; ++c) {
                tma_load_3d(sK + c * CHUNK_BYTES, &maps.k, bar(L::B_KVFULL), c * 64, k0, bh);
                tma_load_3d(sV + c * CHUNK_BYTES, &maps.v, bar(L::B_KVFULL), c * 64, k0, bh);
            }
            int issued = 0;
            for (int t = 0; t < nt; ++t) {
                const int s = t % L::QS;
                if (t >= L::QS &&
                    !mbar_wait(bar(L::B_QEMPTY + s), static_cast<uint32_t>(t / L::QS - 1) & 1u, abort_word,
                               p.status, STATUS_TMA_WAIT, limit))
                    break;
                const int q0 = (qb_lo + t) * BM;
                mbar_arrive_expect_tx(bar(L::B_QFULL + s), 2 * L::TILE + 2 * BM * 4);
                for (int c = 0; c < L::CH; ++c) {
                    tma_load_3d(sQ + s * L::TILE + c * CHUNK_BYTES, &maps.q, bar(L::B_QFULL + s), c * 64, q0, bh);
                    tma_load_3d(sdO + s * L::TILE + c * CHUNK_BYTES, &maps.dout, bar(L::B_QFULL + s), c * 64, q0,
                                bh);
                }
                const int64_t row0 = static_cast<int64_t>(bh) * p.n_pad + q0;
                bulk_load(sbase + L::LSE_OFF + s * BM * 4, p.lse2 + row0, BM * 4, bar(L::B_QFULL + s));
                bulk_load(sbase + L::DD_OFF + s * BM * 4, p.dd + row0, BM * 4, bar(L::B_QFULL + s));
                ++issued;
            }
            // land every copy still in flight (only possible after an abort)
            drain(bar(L::B_KVFULL), 0, 100000000ull);
            for (int t = issued - 1; t >= 0 && t >= issued - L::QS; --t)
                drain(bar(L::B_QFULL + t % L::QS), static_cast<uint32_t>(t / L::QS) & 1u, 100000000ull);
        } else if (warp == L::WARP_MMA) {
            // ================================================== MMA issuer (whole warp, one elected lane)
            constexpr uint32_t ID_S = idesc_bf16_f32(BN, BM, false, false);   // M = keys, N = queries
            constexpr uint32_t ID_KV = idesc_bf16_f32(BN, D, false, true);    // M = keys, N = d
            constexpr uint32_t ID_DQ = idesc_bf16_f32(BM, 64, true, true);    // M = queries, N = 64
            const uint64_t dK_k = sdesc_sw128(sK, 16, 1024);
            const uint64_t dV_k = sdesc_sw128(sV, 16, 1024);
            const uint64_t dS_mn = sdesc_sw128(sdS, CHUNK_BYTES, 1024);
            auto wait = [&](int b, uint32_t parity) -> bool {
                const bool r = mbar_wait(bar(b), parity, abort_word, p.status, STATUS_MMA_WAIT, limit);
                return __all_sync(0xffffffffu, r);
            };
            bool ok = wait(L::B_KVFULL, 0);
            for (int t = 0; ok && t < nt; ++t) {
                const int s = t % L::QS;
                const uint32_t parity = static_cast<uint32_t>(t) & 1u;
                ok = wait(L::B_QFULL + s, static_cast<uint32_t>(t / L::QS) & 1u);
                // the previous tile's MMAs read Pᵀ/dSᵀ and dS: they must be complete
                if (ok && t > 0) ok = wait(L::B_TILEDONE, parity ^ 1u);
                if (ok && L::DQ_OVER_S && t > 0) ok = wait(L::B_DQFREE, parity ^ 1u);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dQ_k = sdesc_sw128(sQ + s * L::TILE, 16, 1024);
                const uint64_t dO_k = sdesc_sw128(sdO + s * L::TILE, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk / 4) * CHUNK_BYTES + (kk % 4) * 32) >> 4);
                    mma_ss_warp(tmem + L::S_COL, dK_k + off, dQ_k + off, ID_S, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk / 4) * CHUNK_BYTES + (kk % 4) * 32) >> 4);
                    mma_ss_warp(tmem + L::DP_COL, dV_k + off, dO_k + off, ID_S, kk > 0 ? 1u : 0u);
                }
                mma_commit_warp(bar(L::B_SFULL));
                ok = wait(L::B_PFULL, parity);
                if (ok && !L::DQ_OVER_S && t > 0) ok = wait(L::B_DQFREE, parity ^ 1u);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dO_mn = sdesc_sw128(sdO + s * L::TILE, CHUNK_BYTES, 1024);
                const uint64_t dQ_mn = sdesc_sw128(sQ + s * L::TILE, CHUNK_BYTES, 1024);
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>((kk * 2048) >> 4);
                    mma_ts_warp(tmem + L::DV_COL, tmem + L::P_COL + kk * 8, dO_mn + off, ID_KV,
                                (t > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>((kk * 2048) >> 4);
                    mma_ts_warp(tmem + L::DK_COL, tmem + L::DS_COL + kk * 8, dQ_mn + off, ID_KV,
                                (t > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int h = 0; h < D / 64; ++h) {
                    const uint64_t dKh_mn = sdesc_sw128(sK + h * CHUNK_BYTES, CHUNK_BYTES, 1024);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        const uint64_t off = static_cast<uint64_t>((kk * 2048) >> 4);
                        mma_ss_warp(tmem + L::dq_col(h), dS_mn + off, dKh_mn + off, ID_DQ, kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit_warp(bar(L::B_DQFULL));
                mma_commit_warp(bar(L::B_QEMPTY + s));
                mma_commit_warp(bar(L::B_TILEDONE));
            }
            mma_commit_warp(bar(L::B_DKVDONE));
            drain(bar(L::B_DKVDONE), 0, 100000000ull);
        }
        __syncwarp();
    } else {
        // ================================================== Pᵀ / dSᵀ, dQ read-out, epilogue
        const int r = 32 * warp + lane;               // TMEM lane: a key here, a query row for dQ
        const int key = k0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        const float sl2 = p.scale_log2;
        bool ok = true;
        bool store_pending = false;

        if (p.debug_flags & DEBUG_FORCE_TIMEOUT) {
            ok = mbar_wait(bar(L::B_NEVER), 0, abort_word, p.status, STATUS_FORCED, 20000000ull);
            ok = __all_sync(0xffffffffu, ok);
        }
        auto wait_stores_read = [&]() {
            if (store_pending && lane == 0) bulk_wait_group_read0();
            __syncwarp();
        };

        for (int t = 0; ok && t < nt; ++t) {
            const int s = t % L::QS;
            const uint32_t parity = static_cast<uint32_t>(t) & 1u;
            const int q0 = (qb_lo + t) * BM;
            ok = mbar_wait(bar(L::B_QFULL + s), static_cast<uint32_t>(t / L::QS) & 1u, abort_word, p.status,
                           STATUS_SOFTMAX_WAIT, limit) &&
                 mbar_wait(bar(L::B_SFULL), parity, abort_word, p.status, STATUS_SOFTMAX_WAIT, limit);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            wait_stores_read();   // this warp's staging rows (the dS rows it writes) are free again
            const uint32_t lse_s = sbase + L::LSE_OFF + s * BM * 4;
            const uint32_t dd_s = sbase + L::DD_OFF + s * BM * 4;
            const bool need_mask = __any_sync(0xffffffffu, key >= kv_len || q0 + BM - 1 >= p.n ||
                                                               (mask_is_causal(MASK) && key > q0 + p.causal_off));
            // Pᵀ: the whole row of Sᵀ (this key against the tile's 128 queries) at once
            uint32_t sr[BM];
            tmem_ld32(tmem + lane_base + L::S_COL + 0, sr + 0);
            tmem_ld32(tmem + lane_base + L::S_COL + 32, sr + 32);
            tmem_ld32(tmem + lane_base + L::S_COL + 64, sr + 64);
            tmem_ld32(tmem + lane_base + L::S_COL + 96, sr + 96);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < BM / 32; ++c) {
                float lz[32];
#pragma unroll
                for (int v = 0; v < 8; ++v) lds_v4f(lse_s + (32 * c + 4 * v) * 4, lz + 4 * v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int j = 32 * c + i;
                    sr[j] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(sr[j]), sl2, -lz[i])));
                }
            }
            if (need_mask) {
                // this key is visible to the tile's query columns j in [j_lo, j_hi)
                const int q_first = key >= kv_len ? INT32_MAX : (mask_is_causal(MASK) ? key - p.causal_off : 0);
                const int j_lo = q_first == INT32_MAX ? BM : max(q_first - q0, 0);
                const int j_hi = min(p.n - q0, BM);
#pragma unroll
                for (int j = 0; j < BM; ++j)
                    if (j < j_lo || j >= j_hi) sr[j] = 0u;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(sr[64 * h + 2 * i]), __uint_as_float(sr[64 * h + 2 * i + 1]));
                tmem_st32(tmem + lane_base + L::P_COL + 32 * h, pk);   // over Sᵀ, already read
            }
            // dSᵀ = Pᵀ ∘ (dPᵀ - D), 32 queries at a time; dSᵀ goes over the dPᵀ columns
            // already read and, MN-major (row = key, 64-query chunks), into shared memory
#pragma unroll
            for (int c = 0; c < BM / 32; ++c) {
                uint32_t dr[32];
                float dz[32];
                tmem_ld32(tmem + lane_base + L::DP_COL + 32 * c, dr);
#pragma unroll
                for (int v = 0; v < 8; ++v) lds_v4f(dd_s + (32 * c + 4 * v) * 4, dz + 4 * v);
                tmem_wait_ld();
                uint32_t dk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float a = __uint_as_float(sr[32 * c + 2 * i]) * (__uint_as_float(dr[2 * i]) - dz[2 * i]);
                    const float b =
                        __uint_as_float(sr[32 * c + 2 * i + 1]) * (__uint_as_float(dr[2 * i + 1]) - dz[2 * i + 1]);
                    dk[i] = pack_bf16x2(a, b);
                }
                tmem_st16(tmem + lane_base + L::DS_COL + 16 * c, dk);
                const uint32_t row_base = sdS + (c / 2) * CHUNK_BYTES + r * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t piece = static_cast<uint32_t>((c % 2) * 4 + q);
                    const uint32_t addr = row_base + ((piece ^ static_cast<uint32_t>(r & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(dk[4 * q]),
                                 "r"(dk[4 * q + 1]), "r"(dk[4 * q + 2]), "r"(dk[4 * q + 3])
                                 : "memory");
                }
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(L::B_PFULL));

            // ---------------------------------------- dQ of this tile: TMEM -> staging -> reduce-add
            ok = mbar_wait(bar(L::B_DQFULL), parity, abort_word, p.status, STATUS_SOFTMAX_WAIT, limit);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int h = 0; h < D / 64; ++h) {
                uint32_t a[32], b[32];
                tmem_ld32(tmem + lane_base + L::dq_col(h), a);
                tmem_ld32(tmem + lane_base + L::dq_col(h) + 32, b);
                tmem_wait_ld();
                if (h == D / 64 - 1) {
                    tc_fence_before();
                    mbar_arrive(bar(L::B_DQFREE));
                }
                wait_stores_read();
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const uint32_t* src = cc == 0 ? a : b;
                    const uint32_t row_base = sdS + cc * CHUNK_BYTES + r * 128;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint32_t addr = row_base + ((static_cast<uint32_t>(q) ^ static_cast<uint32_t>(r & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(src[4 * q]),
                                     "r"(src[4 * q + 1]), "r"(src[4 * q + 2]), "r"(src[4 * q + 3])
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && q0 + 32 * warp < p.n) {
                    for (int cc = 0; cc < 2; ++cc)
                        tma_reduce_add_3d(&maps.dq_acc, sdS + cc * CHUNK_BYTES + warp * 32 * 128, 64 * h + 32 * cc,
                                          q0 + 32 * warp, bh);
                    bulk_commit_group();
                    store_pending = true;
                }
                __syncwarp();
            }
        }

        // ---------------------------------------- dV, then dK (x scale): TMEM -> bf16 staging -> TMA store
        if (ok) {
            ok = mbar_wait(bar(L::B_DKVDONE), 0, abort_word, p.status, STATUS_SOFTMAX_WAIT, limit);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = which == 0 ? L::DV_COL : L::DK_COL;
                const float mul = which == 0 ? 1.f : p.scale;
                wait_stores_read();
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_base + col + 32 * cc, o);
                    tmem_wait_ld();
                    const uint32_t chunk_base = sdS + (cc / 2) * CHUNK_BYTES + r * 128;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            v[e] = pack_bf16x2(__uint_as_float(o[8 * q + 2 * e]) * mul,
                                               __uint_as_float(o[8 * q + 2 * e + 1]) * mul);
                        const uint32_t piece = static_cast<uint32_t>((cc % 2) * 4 + q);
                        const uint32_t addr = chunk_base + ((piece ^ static_cast<uint32_t>(r & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]),
                                     "r"(v[2]), "r"(v[3])
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && k0 + 32 * warp < p.m) {
                    const CUtensorMap* map = which == 0 ? &maps.dv : &maps.dk;
                    for (int c = 0; c < L::CH; ++c)
                        tma_store_3d(map, sdS + c * CHUNK_BYTES + warp * 32 * 128, c * 64, k0 + 32 * warp, bh);
                    bulk_commit_group();
                    store_pending = true;
                }
                __syncwarp();
            }
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == L::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

template <int D, int MASK>
cudaError_t launch(const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    using L = Layout<D>;
    auto kern = attn_bwd_kernel<D, MASK>;
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
    const int64_t grid = static_cast<int64_t>(p.B) * p.H * p.num_kblocks;
    kern<<<static_cast<unsigned>(grid), L::NUM_THREADS, L::BYTES, stream>>>(maps, p);
    return cudaGetLastError();
}

}  // namespace bwd
}  // namespace attn
