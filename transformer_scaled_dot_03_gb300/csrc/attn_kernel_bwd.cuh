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
//   warps 0-7   Pᵀ/dSᵀ (thread = key), dQ read-out (thread = query), dK/dV epilogue;
//               warp w serves tensor-memory lanes 32(w % 4)..+31 and the half
//               w / 4 of the columns (queries for Pᵀ/dSᵀ, head dims for dQ, dK, dV):
//               every element of Pᵀ and dSᵀ is independent (P comes from the saved
//               LSE), so two warpgroups share a row without exchanging anything
//   warp  8     TMA producer: K and V once, then Q, dO, LSE, D per query tile
//   warp  9     tcgen05.mma issuer, owns the TMEM allocation
// Tensor memory (512 columns): Sᵀ [0,128) then Pᵀ [0,64); dPᵀ [128,256) then dSᵀ
// [128,192); dV [256,256+d); dK [256+d,256+2d); dQ at d = 64 in [384,448), at
// d = 128 as two 64-column halves in [64,128) and [192,256).
#pragma once

#include <cstdint>
#include <type_traits>
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

// The dQ reduce-add (3-D tiled, shared -> global, bulk group) with an L2 evict_last
// policy: the fp32 accumulator is zeroed, added into and read back within one
// backward pass, and the streamed Q, K, V and dO tiles should leave L2 before it
// does (the preparation kernel's zero stores carry the same policy).
__device__ __forceinline__ void dq_reduce_add(const CUtensorMap* map, uint32_t src, int32_t c0, int32_t c1,
                                              int32_t c2)
{
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group.L2::cache_hint"
        " [%0, {%2, %3, %4}], [%1], %5;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "l"(l2_policy_evict_last())
        : "memory");
}

// DK: query/key head dim, DV: value head dim.
template <int DK, int DV>
struct Layout {
    static constexpr int CHK = DK / 64;
    static constexpr int CHV = DV / 64;
    static constexpr int TILE_K = CHK * CHUNK_BYTES;     // a 128 x DK bf16 tile (K, Q)
    static constexpr int TILE_V = CHV * CHUNK_BYTES;     // a 128 x DV bf16 tile (V, dO)
    static constexpr int NUM_THREADS = 320;
    static constexpr int COMPUTE_THREADS = 256;
    static constexpr int WARP_TMA = 8;
    static constexpr int WARP_MMA = 9;
    static constexpr int QS = DK == 64 && DV == 64 ? 2 : 1;   // Q/dO/LSE/D ring depth
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + TILE_K;
    static constexpr int Q_OFF = V_OFF + TILE_V;
    static constexpr int DO_OFF = Q_OFF + QS * TILE_K;
    static constexpr int DS_OFF = DO_OFF + QS * TILE_V;    // dS (bf16, MN-major) / staging, 32 KB
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
    static constexpr int B_RDONE = B_DKVDONE + 1;   // Sᵀ and dPᵀ of the tile read    (256 arrivals)
    static constexpr int B_EPI = B_RDONE + 1;       // epilogue staging steps         (256 arrivals)
    static constexpr int B_NEVER = B_EPI + 1;
    static constexpr int NBARS = B_NEVER + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BYTES = MISC_OFF + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0, DP_COL = 128, P_COL = 0, DS_COL = 128;
    static constexpr uint32_t DV_COL = 256, DK_COL = 256 + DV;
    static constexpr bool DQ_OVER_S = DK == 128;           // dQ halves reuse the upper Sᵀ/dPᵀ columns
    __host__ __device__ static constexpr uint32_t dq_col(int h)
    {
        return DQ_OVER_S ? (h == 0 ? 64u : 192u) : DK_COL + DK;
    }
    static_assert(DK_COL + DK <= TMEM_COLS && (DQ_OVER_S || DK_COL + 2 * DK <= TMEM_COLS), "tensor memory layout");
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

template <int DK, int DV, int MASK, bool BIAS>
__global__ void __launch_bounds__(Layout<DK, DV>::NUM_THREADS, 1)
attn_bwd_kernel(const __grid_constant__ BwdMaps maps, const BwdParams p)
{
    using L = Layout<DK, DV>;
    griddep_wait();   // the preparation kernel's D, LSE rows and zeroed dQ accumulator are visible
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
        const int64_t base = static_cast<int64_t>(bh) * p.m + k0;
        uint4* gk = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dK) + base * DK);
        uint4* gv = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dV) + base * DV);
        for (int i = threadIdx.x; i < rows * DK / 8; i += blockDim.x) gk[i] = make_uint4(0u, 0u, 0u, 0u);
        for (int i = threadIdx.x; i < rows * DV / 8; i += blockDim.x) gv[i] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    // query tiles that can see this key tile
    const int off = causal_offset(MASK, p.causal_off, kv_len, p.n);   // row i sits at key position i + off
    const int nqb = (p.n + BM - 1) / BM;
    int qb_lo = 0;
    if (mask_is_causal(MASK)) {
        const int first_q = k0 - off;              // first row that sees key k0
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
        mbar_init(bar(L::B_PFULL), L::COMPUTE_THREADS);
        mbar_init(bar(L::B_DQFULL), 1);
        mbar_init(bar(L::B_DQFREE), L::COMPUTE_THREADS);
        mbar_init(bar(L::B_TILEDONE), 1);
        mbar_init(bar(L::B_DKVDONE), 1);
        mbar_init(bar(L::B_RDONE), L::COMPUTE_THREADS);
        mbar_init(bar(L::B_EPI), L::COMPUTE_THREADS);
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

    if (warp >= L::WARP_TMA) {
        if (warp == L::WARP_TMA && lane == 0) {
            // ================================================== TMA producer
            mbar_arrive_expect_tx(bar(L::B_KVFULL), L::TILE_K + L::TILE_V);
            for (int c = 0; c < L::CHK; ++c)
                tma_load_3d(sK + c * CHUNK_BYTES, &maps.k, bar(L::B_KVFULL), c * 64, k0, bh);
            for (int c = 0; c < L::CHV; ++c)
                tma_load_3d(sV + c * CHUNK_BYTES, &maps.v, bar(L::B_KVFULL), c * 64, k0, bh);
            int issued = 0;
            for (int t = 0; t < nt; ++t) {
                const int s = t % L::QS;
                if (t >= L::QS &&
                    !mbar_wait(bar(L::B_QEMPTY + s), static_cast<uint32_t>(t / L::QS - 1) & 1u, abort_word,
                               p.status, STATUS_TMA_WAIT, limit))
                    break;
                const int q0 = (qb_lo + t) * BM;
                mbar_arrive_expect_tx(bar(L::B_QFULL + s), L::TILE_K + L::TILE_V + 2 * BM * 4);
                for (int c = 0; c < L::CHK; ++c)
                    tma_load_3d(sQ + s * L::TILE_K + c * CHUNK_BYTES, &maps.q, bar(L::B_QFULL + s), c * 64, q0, bh);
                for (int c = 0; c < L::CHV; ++c)
                    tma_load_3d(sdO + s * L::TILE_V + c * CHUNK_BYTES, &maps.dout, bar(L::B_QFULL + s), c * 64, q0,
                                bh);
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
            constexpr uint32_t ID_DV = idesc_bf16_f32(BN, DV, false, true);   // M = keys, N = d_v
            constexpr uint32_t ID_DK = idesc_bf16_f32(BN, DK, false, true);   // M = keys, N = d_k
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
                const uint64_t dQ_k = sdesc_sw128(sQ + s * L::TILE_K, 16, 1024);
                const uint64_t dO_k = sdesc_sw128(sdO + s * L::TILE_V, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk / 4) * CHUNK_BYTES + (kk % 4) * 32) >> 4);
                    mma_ss_warp(tmem + L::S_COL, dK_k + off, dQ_k + off, ID_S, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < DV / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk / 4) * CHUNK_BYTES + (kk % 4) * 32) >> 4);
                    mma_ss_warp(tmem + L::DP_COL, dV_k + off, dO_k + off, ID_S, kk > 0 ? 1u : 0u);
                }
                mma_commit_warp(bar(L::B_SFULL));
                ok = wait(L::B_PFULL, parity);
                if (ok && !L::DQ_OVER_S && t > 0) ok = wait(L::B_DQFREE, parity ^ 1u);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dO_mn = sdesc_sw128(sdO + s * L::TILE_V, CHUNK_BYTES, 1024);
                const uint64_t dQ_mn = sdesc_sw128(sQ + s * L::TILE_K, CHUNK_BYTES, 1024);
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>((kk * 2048) >> 4);
                    mma_ts_warp(tmem + L::DV_COL, tmem + L::P_COL + kk * 8, dO_mn + off, ID_DV,
                                (t > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>((kk * 2048) >> 4);
                    mma_ts_warp(tmem + L::DK_COL, tmem + L::DS_COL + kk * 8, dQ_mn + off, ID_DK,
                                (t > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int h = 0; h < DK / 64; ++h) {
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
        const int wq = warp % 4;                      // lane quadrant
        const int half = warp / 4;                    // column half
        const int r = 32 * wq + lane;                 // TMEM lane: a key here, a query row for dQ
        const int key = k0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;
        const float sl2 = p.scale_log2;
        const float sb = BIAS ? __ldg(p.slopes + bh % p.H) * 1.44269504088896341f : 0.f;   // log2 domain
        bool ok = true;
        bool store_pending = false;
        // Rendezvous of the eight compute warps through an mbarrier (every thread
        // arrives, then waits with the usual bound), so that a warp leaving on a
        // timeout cannot strand the others.
        auto rendezvous = [&](int b, uint32_t parity) -> bool {
            mbar_arrive(bar(b));
            const bool r = mbar_wait(bar(b), parity, abort_word, p.status, STATUS_SOFTMAX_WAIT, limit);
            return __all_sync(0xffffffffu, r);
        };
        int epi_phase = 0;

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
            const int c0 = 64 * half;                 // this warpgroup's first query column
            const uint32_t lse_s = sbase + L::LSE_OFF + (s * BM + c0) * 4;
            const uint32_t dd_s = sbase + L::DD_OFF + (s * BM + c0) * 4;
            const bool need_mask =
                __any_sync(0xffffffffu, key >= kv_len || q0 + c0 + 63 >= p.n ||
                                            (mask_is_causal(MASK) && key > q0 + c0 + off));
            // this warpgroup's half of the row of Sᵀ and of dPᵀ (64 queries each)
            uint32_t sr[64], dr[64];
            tmem_ld32(tmem + lane_base + L::S_COL + c0, sr);
            tmem_ld32(tmem + lane_base + L::S_COL + c0 + 32, sr + 32);
            tmem_ld32(tmem + lane_base + L::DP_COL + c0, dr);
            tmem_ld32(tmem + lane_base + L::DP_COL + c0 + 32, dr + 32);
            tmem_wait_ld();
            // P = exp2(S·scale·log2 e − LSE·log2 e), with the distance bias
            // −sb |i' − key| of query column j (i' = q0 + c0 + j + m − n) under BIAS
            const float d1 = static_cast<float>(q0 + c0 + off - key);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float lz[32];
#pragma unroll
                for (int v = 0; v < 8; ++v) lds_v4f(lse_s + (32 * c + 4 * v) * 4, lz + 4 * v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int j = 32 * c + i;
                    const float z = BIAS ? fmaf(-sb, fabsf(d1 + static_cast<float>(j)), -lz[i]) : -lz[i];
                    sr[j] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(sr[j]), sl2, z)));
                }
            }
            if (need_mask) {
                // this key is visible to the query columns j in [j_lo, j_hi) of the tile
                const int q_first = key >= kv_len ? INT32_MAX : (mask_is_causal(MASK) ? key - off : 0);
                const int j_lo = q_first == INT32_MAX ? BM : max(q_first - q0, 0) - c0;
                const int j_hi = min(p.n - q0, BM) - c0;
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    if (j < j_lo || j >= j_hi) sr[j] = 0u;
            }
            // dS = P ∘ (dP − D), kept in dr
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float dz[32];
#pragma unroll
                for (int v = 0; v < 8; ++v) lds_v4f(dd_s + (32 * c + 4 * v) * 4, dz + 4 * v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int j = 32 * c + i;
                    dr[j] = __float_as_uint(__uint_as_float(sr[j]) * (__uint_as_float(dr[j]) - dz[i]));
                }
            }
            // Pᵀ and dSᵀ go over the first columns of Sᵀ and dPᵀ, which the other
            // warpgroup reads: every read of this tile's Sᵀ and dPᵀ comes first
            ok = rendezvous(L::B_RDONE, parity);
            if (!ok) break;
            {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]));
                tmem_st32(tmem + lane_base + L::P_COL + 32 * half, pk);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1]));
                tmem_st32(tmem + lane_base + L::DS_COL + 32 * half, pk);
                // this warp's staging rows (the dS rows it writes) must have been read by
                // the previous tile's dQ reduce-add
                wait_stores_read();
                // dS, MN-major: row = key r, chunk = this warpgroup's 64 queries
                const uint32_t row_base = sdS + half * CHUNK_BYTES + r * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint32_t addr = row_base + ((static_cast<uint32_t>(q) ^ static_cast<uint32_t>(r & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * q]),
                                 "r"(pk[4 * q + 1]), "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
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
            // d = 64: this warpgroup's 32 of the 64 dQ columns; d = 128: its 64 (two chunks
            // of 32, one after the other through this warp's staging rows)
#pragma unroll 1
            for (int k = 0; k < DK / 64; ++k) {
                const int col = DK == 64 ? 32 * half : 64 * half + 32 * k;   // dQ column of the chunk
                uint32_t a[32];
                tmem_ld32(tmem + lane_base + L::dq_col(col / 64) + (col % 64), a);
                tmem_wait_ld();
                if (k == DK / 64 - 1) {
                    tc_fence_before();
                    mbar_arrive(bar(L::B_DQFREE));
                }
                wait_stores_read();
                const uint32_t row_base = sdS + half * CHUNK_BYTES + r * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint32_t addr = row_base + ((static_cast<uint32_t>(q) ^ static_cast<uint32_t>(r & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a[4 * q]),
                                 "r"(a[4 * q + 1]), "r"(a[4 * q + 2]), "r"(a[4 * q + 3])
                                 : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && q0 + 32 * wq < p.n) {
                    dq_reduce_add(&maps.dq_acc, sdS + half * CHUNK_BYTES + wq * 32 * 128, col, q0 + 32 * wq, bh);
                    bulk_commit_group();
                    store_pending = true;
                }
                __syncwarp();
            }
        }

        // ---------------------------------------- dV, then dK (x scale): TMEM -> bf16 staging -> TMA store
        // Each warpgroup converts its half of the columns; at d = 64 the two halves
        // share one 64-column staging chunk and warpgroup 0 stores it.
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
                const int Dw = which == 0 ? DV : DK;   // head dim of the gradient
                wait_stores_read();
                // both warpgroups' earlier stores have read the staging
                ok = rendezvous(L::B_EPI, static_cast<uint32_t>(epi_phase++) & 1u);
                if (!ok) break;
#pragma unroll
                for (int cc = 0; cc < Dw / 64; ++cc) {
                    const int c = half * (Dw / 2) + 32 * cc;   // first column of this 32-column piece
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_base + col + c, o);
                    tmem_wait_ld();
                    const uint32_t chunk_base = sdS + (c / 64) * CHUNK_BYTES + r * 128;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            v[e] = pack_bf16x2(__uint_as_float(o[8 * q + 2 * e]) * mul,
                                               __uint_as_float(o[8 * q + 2 * e + 1]) * mul);
                        const uint32_t piece = static_cast<uint32_t>(((c % 64) / 32) * 4 + q);
                        const uint32_t addr = chunk_base + ((piece ^ static_cast<uint32_t>(r & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]),
                                     "r"(v[2]), "r"(v[3])
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                // both halves of every staged row are written
                ok = rendezvous(L::B_EPI, static_cast<uint32_t>(epi_phase++) & 1u);
                if (!ok) break;
                const bool storer = Dw == 64 ? half == 0 : true;
                if (storer && lane == 0 && k0 + 32 * wq < p.m) {
                    const CUtensorMap* map = which == 0 ? &maps.dv : &maps.dk;
                    const int c = Dw == 64 ? 0 : half;
                    tma_store_3d(map, sdS + c * CHUNK_BYTES + wq * 32 * 128, c * 64, k0 + 32 * wq, bh);
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

// ---------------------------------------------------------------------------
// d = 64: the same computation, persistent and with the query tiles pipelined.
//
// dK += dSᵀ Q takes dS from shared memory (the tile written for dQ, row = key with
// the queries contiguous, is exactly the K-major layout of A = dSᵀ), so dSᵀ needs
// no tensor memory and Pᵀ gets columns of its own. Then nothing the MMAs of tile t
// read overlaps what Sᵀ and dPᵀ of the next tile write, and the MMA warp issues
//     Sᵀ, dPᵀ (next)  as soon as the softmax warps have loaded Sᵀ, dPᵀ (t)
//     dV, dK, dQ (t)  once Pᵀ (t) and dS (t) are written,
// so the tensor cores compute the next tile's scores while the softmax warps turn
// tile t's into Pᵀ and dS (warp 10 issues the scores, warp 9 the products). The dQ
// of a tile is read out one iteration later, through a staging area of its own.
// Warp 11 is idle: it completes the control warpgroup (8-11), whose registers go to
// the compute warps by setmaxnreg.
//
// Persistent: one CTA per SM walks work items (b, h, 128-key tile) round-robin;
// under the causal masks a unit pairs key tile k with key tile nkb-1-k of the same
// head (the one with most query tiles with the one with fewest), so that units
// cost the same. K and V are double-buffered, so the next item's keys load during
// the current item's last tiles, and its first scores are computed while the
// softmax warps write the current item's dK and dV out. Barrier phases run on
// per-CTA tile and item counters.
//   Tensor memory: Sᵀ [0,128), dPᵀ [128,256), dV [256,320), dK [320,384),
//   dQ [384,448), Pᵀ [448,512).
struct LayoutPipe {
    static constexpr int D = 64;
    static constexpr int TILE = CHUNK_BYTES;                 // a 128 x 64 bf16 tile
    static constexpr int NUM_THREADS = 384;                  // warp 11 idle: completes the control warpgroup
    static constexpr int COMPUTE_THREADS = 256;
    static constexpr int WARP_TMA = 8;
    static constexpr int WARP_MMA = 9;                       // issues the products, owns the tensor memory
    static constexpr int WARP_MMA_S = 10;                    // issues the scores
    // registers per thread: the launch's share, then re-balanced by setmaxnreg from
    // the control warpgroup (warps 8-11) to the two compute warpgroups
    static constexpr uint32_t REG_LAUNCH = 65536 / NUM_THREADS / 8 * 8;
    static constexpr uint32_t REG_CTRL = 72;
    static constexpr uint32_t REG_COMPUTE = (REG_LAUNCH * NUM_THREADS - REG_CTRL * 128) / 256 / 8 * 8;
    static_assert(256 * REG_COMPUTE + 128 * REG_CTRL <= REG_LAUNCH * NUM_THREADS, "register split");
    static constexpr int QS = 2;                             // Q/dO/LSE/D ring depth
    static constexpr int KVS = 2;                            // K/V buffers
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + KVS * TILE;
    static constexpr int Q_OFF = V_OFF + KVS * TILE;
    static constexpr int DO_OFF = Q_OFF + QS * TILE;
    static constexpr int DS_OFF = DO_OFF + QS * TILE;      // dS: two 64-query chunks (row = key)
    static constexpr int DQ_OFF = DS_OFF + 2 * CHUNK_BYTES;  // dQ staging: two 32-column fp32 chunks
    static constexpr int LSE_OFF = DQ_OFF + 2 * CHUNK_BYTES;
    static constexpr int DD_OFF = LSE_OFF + QS * BM * 4;
    static constexpr int BAR_OFF = DD_OFF + QS * BM * 4;
    static constexpr int B_KVFULL = 0;
    static constexpr int B_KVEMPTY = B_KVFULL + KVS;
    static constexpr int B_QFULL = B_KVEMPTY + KVS;
    static constexpr int B_QEMPTY = B_QFULL + QS;
    static constexpr int B_SFULL = B_QEMPTY + QS;   // Sᵀ, dPᵀ computed                 (commit)
    static constexpr int B_RDONE = B_SFULL + 1;     // Sᵀ, dPᵀ loaded by the softmax     (256 arrivals)
    static constexpr int B_PFULL = B_RDONE + 1;     // Pᵀ and dS written                 (256 arrivals)
    static constexpr int B_BDONE = B_PFULL + 1;     // dV, dK, dQ of the tile done       (commit)
    static constexpr int B_DQFREE = B_BDONE + 1;    // dQ read out of tensor memory      (256 arrivals)
    static constexpr int B_DKVDONE = B_DQFREE + 1;  // an item's dV, dK complete         (commit)
    static constexpr int B_DKVFREE = B_DKVDONE + 1; // an item's dV, dK read out         (256 arrivals)
    static constexpr int B_DRAIN = B_DKVFREE + 1;   // [2] each issuing warp's last MMAs done
    static constexpr int B_NEVER = B_DRAIN + 2;
    static constexpr int NBARS = B_NEVER + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BYTES = MISC_OFF + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 320, DQ_COL = 384, P_COL = 448;
    static_assert(BYTES <= 232448, "shared memory budget");
};

// One work item: a 128-key tile of one (b, h) pair and the query tiles that see it.
struct BwdItem {
    int bh, k0, kv_len, qb_lo, nt;   // nt = 0: no query sees these keys (zero gradients)
    int off;                         // query row i sits at key position i + off
};

template <int MASK>
__device__ __forceinline__ int bwd_units_per_head(const BwdParams& p)
{
    return mask_is_causal(MASK) ? (p.num_kblocks + 1) / 2 : p.num_kblocks;
}

template <int MASK>
__device__ __forceinline__ int bwd_items_of_unit(int u, const BwdParams& p)
{
    if (!mask_is_causal(MASK)) return 1;
    const int k = u % bwd_units_per_head<MASK>(p);
    return (k == p.num_kblocks - 1 - k) ? 1 : 2;
}

template <int MASK>
__device__ __forceinline__ BwdItem bwd_item(int u, int iu, const BwdParams& p)
{
    const int uph = bwd_units_per_head<MASK>(p);
    BwdItem w;
    w.bh = u / uph;
    const int k = u % uph;
    const int kb = (mask_is_causal(MASK) && iu == 1) ? p.num_kblocks - 1 - k : k;
    w.k0 = kb * BN;
    w.kv_len = p.m;
    if (mask_has_lengths(MASK)) {
        const int len = __ldg(p.key_lengths + w.bh / p.H);
        w.kv_len = len < 0 ? 0 : (len > p.m ? p.m : len);
    }
    w.qb_lo = 0;
    w.off = causal_offset(MASK, p.causal_off, w.kv_len, p.n);
    if (mask_is_causal(MASK)) {
        const int first_q = w.k0 - w.off;            // first row that sees key k0
        w.qb_lo = first_q <= 0 ? 0 : first_q / BM;
    }
    const int nqb = (p.n + BM - 1) / BM;
    w.nt = w.k0 >= w.kv_len ? 0 : nqb - w.qb_lo;
    return w;
}

// Walks the tiles of this CTA's items in order, skipping items without queries.
template <int MASK>
struct BwdCursor {
    int u, iu, t;
    BwdItem w;
    bool valid;
    __device__ void settle(const BwdParams& p, int num_units)
    {
        while (u < num_units) {
            w = bwd_item<MASK>(u, iu, p);
            if (t < w.nt) {
                valid = true;
                return;
            }
            t = 0;
            if (++iu >= bwd_items_of_unit<MASK>(u, p)) {
                iu = 0;
                u += static_cast<int>(gridDim.x);
            }
        }
        valid = false;
    }
    __device__ void start(const BwdParams& p, int num_units)
    {
        u = static_cast<int>(blockIdx.x);
        iu = 0;
        t = 0;
        settle(p, num_units);
    }
    __device__ void next(const BwdParams& p, int num_units)
    {
        ++t;
        settle(p, num_units);
    }
};

template <int MASK, bool BIAS>
__global__ void __launch_bounds__(LayoutPipe::NUM_THREADS, 1)
attn_bwd_pipe_kernel(const __grid_constant__ BwdMaps maps, const BwdParams p)
{
    using L = LayoutPipe;
    constexpr int D = 64;
    const int num_units = p.B * p.H * bwd_units_per_head<MASK>(p);

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
        for (int s = 0; s < L::KVS; ++s) {
            mbar_init(bar(L::B_KVFULL + s), 1);
            mbar_init(bar(L::B_KVEMPTY + s), 1);
        }
        for (int s = 0; s < L::QS; ++s) {
            mbar_init(bar(L::B_QFULL + s), 1);
            mbar_init(bar(L::B_QEMPTY + s), 1);
        }
        mbar_init(bar(L::B_SFULL), 1);
        mbar_init(bar(L::B_RDONE), L::COMPUTE_THREADS);
        mbar_init(bar(L::B_PFULL), L::COMPUTE_THREADS);
        mbar_init(bar(L::B_BDONE), 1);
        mbar_init(bar(L::B_DQFREE), L::COMPUTE_THREADS);
        mbar_init(bar(L::B_DKVDONE), 1);
        mbar_init(bar(L::B_DKVFREE), L::COMPUTE_THREADS);
        mbar_init(bar(L::B_DRAIN), 1);
        mbar_init(bar(L::B_DRAIN + 1), 1);
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
    griddep_wait();   // nothing above reads global memory; the preparation kernel's outputs come after

    const uint32_t sK = sbase + L::K_OFF;
    const uint32_t sV = sbase + L::V_OFF;
    const uint32_t sQ = sbase + L::Q_OFF;
    const uint32_t sdO = sbase + L::DO_OFF;
    const uint32_t sdS = sbase + L::DS_OFF;
    const uint32_t sdQ = sbase + L::DQ_OFF;

    if (warp >= L::WARP_TMA) {
        regs_dec<L::REG_CTRL>();
        if (warp == L::WARP_TMA && lane == 0) {
            // ================================================== TMA producer
            BwdCursor<MASK> cur;
            cur.start(p, num_units);
            int gt = 0, it = 0;          // tiles and items so far
            int kv_issued = 0;           // K/V loads issued
            bool ok = true;
            while (ok && cur.valid) {
                if (cur.t == 0) {
                    const int ks = it % L::KVS;
                    if (it >= L::KVS &&
                        !mbar_wait(bar(L::B_KVEMPTY + ks), static_cast<uint32_t>(it / L::KVS - 1) & 1u, abort_word,
                                   p.status, STATUS_TMA_WAIT, limit)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(L::B_KVFULL + ks), 2 * L::TILE);
                    tma_load_3d(sK + ks * L::TILE, &maps.k, bar(L::B_KVFULL + ks), 0, cur.w.k0, cur.w.bh);
                    tma_load_3d(sV + ks * L::TILE, &maps.v, bar(L::B_KVFULL + ks), 0, cur.w.k0, cur.w.bh);
                    ++kv_issued;
                }
                const int s = gt % L::QS;
                if (gt >= L::QS &&
                    !mbar_wait(bar(L::B_QEMPTY + s), static_cast<uint32_t>(gt / L::QS - 1) & 1u, abort_word,
                               p.status, STATUS_TMA_WAIT, limit)) {
                    ok = false;
                    break;
                }
                const int q0 = (cur.w.qb_lo + cur.t) * BM;
                mbar_arrive_expect_tx(bar(L::B_QFULL + s), 2 * L::TILE + 2 * BM * 4);
                tma_load_3d(sQ + s * L::TILE, &maps.q, bar(L::B_QFULL + s), 0, q0, cur.w.bh);
                tma_load_3d(sdO + s * L::TILE, &maps.dout, bar(L::B_QFULL + s), 0, q0, cur.w.bh);
                const int64_t row0 = static_cast<int64_t>(cur.w.bh) * p.n_pad + q0;
                bulk_load(sbase + L::LSE_OFF + s * BM * 4, p.lse2 + row0, BM * 4, bar(L::B_QFULL + s));
                bulk_load(sbase + L::DD_OFF + s * BM * 4, p.dd + row0, BM * 4, bar(L::B_QFULL + s));
                if (cur.t == cur.w.nt - 1) ++it;
                ++gt;
                cur.next(p, num_units);
            }
            // land every copy still in flight (only possible after an abort)
            for (int i = kv_issued - 1; i >= 0 && i >= kv_issued - L::KVS; --i)
                drain(bar(L::B_KVFULL + i % L::KVS), static_cast<uint32_t>(i / L::KVS) & 1u, 100000000ull);
            for (int i = gt - 1; i >= 0 && i >= gt - L::QS; --i)
                drain(bar(L::B_QFULL + i % L::QS), static_cast<uint32_t>(i / L::QS) & 1u, 100000000ull);
        } else if (warp == L::WARP_MMA || warp == L::WARP_MMA_S) {
            // ================================================== MMA issuers (whole warp, one elected lane)
            // Warp 10 issues each tile's scores as soon as the softmax warps hold the
            // previous tile's; warp 9 issues the products. Their MMAs touch disjoint
            // tensor-memory columns, and every dependence between them passes through
            // the softmax warps' barriers (B_RDONE, B_PFULL).
            constexpr uint32_t ID_S = idesc_bf16_f32(BN, BM, false, false);   // M = keys, N = queries
            constexpr uint32_t ID_KV = idesc_bf16_f32(BN, D, false, true);    // M = keys, N = d
            constexpr uint32_t ID_DQ = idesc_bf16_f32(BM, D, true, true);     // M = queries, N = d
            const uint64_t dS_mn = sdesc_sw128(sdS, CHUNK_BYTES, 1024);
            const uint64_t dS_k = sdesc_sw128(sdS, 16, 1024);
            auto wait = [&](int b, uint32_t parity) -> bool {
                const bool r = mbar_wait(bar(b), parity, abort_word, p.status, STATUS_MMA_WAIT, limit);
                return __all_sync(0xffffffffu, r);
            };
            // Sᵀ = K Qᵀ and dPᵀ = V dOᵀ of the tile in Q buffer qs, keys in K/V buffer ks
            auto issue_A = [&](int qs, int ks) {
                const uint64_t dK_k = sdesc_sw128(sK + ks * L::TILE, 16, 1024);
                const uint64_t dV_k = sdesc_sw128(sV + ks * L::TILE, 16, 1024);
                const uint64_t dQ_k = sdesc_sw128(sQ + qs * L::TILE, 16, 1024);
                const uint64_t dO_k = sdesc_sw128(sdO + qs * L::TILE, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                    mma_ss_warp(tmem + L::S_COL, dK_k + off, dQ_k + off, ID_S, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                    mma_ss_warp(tmem + L::DP_COL, dV_k + off, dO_k + off, ID_S, kk > 0 ? 1u : 0u);
                }
                mma_commit_warp(bar(L::B_SFULL));
            };
            BwdCursor<MASK> cur;
            cur.start(p, num_units);
            bool ok = true;
            int gt = 0, it = 0;
            if (warp == L::WARP_MMA_S) {
                if (cur.valid) {
                    ok = wait(L::B_KVFULL, 0) && wait(L::B_QFULL, 0);
                    if (ok) {
                        tc_fence_after();
                        issue_A(0, 0);
                    }
                }
                while (ok && cur.valid) {
                    BwdCursor<MASK> nx = cur;
                    nx.next(p, num_units);
                    if (!nx.valid) break;
                    // the next tile's scores as soon as the softmax warps hold this tile's
                    const bool new_item = nx.t == 0;
                    const int nks = (it + (new_item ? 1 : 0)) % L::KVS;
                    ok = wait(L::B_QFULL + (gt + 1) % L::QS, static_cast<uint32_t>((gt + 1) / L::QS) & 1u) &&
                         (!new_item || wait(L::B_KVFULL + nks, static_cast<uint32_t>((it + 1) / L::KVS) & 1u)) &&
                         wait(L::B_RDONE, static_cast<uint32_t>(gt) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    issue_A((gt + 1) % L::QS, nks);
                    if (new_item) ++it;
                    ++gt;
                    cur = nx;
                }
                mma_commit_warp(bar(L::B_DRAIN + 1));
                drain(bar(L::B_DRAIN + 1), 0, 100000000ull);
            }
            while (warp == L::WARP_MMA && ok && cur.valid) {
                const int s = gt % L::QS;
                const int ks = it % L::KVS;
                const uint32_t parity = static_cast<uint32_t>(gt) & 1u;
                ok = wait(L::B_PFULL, parity);
                // this item's first dV, dK overwrite the accumulators of the previous item
                if (ok && cur.t == 0 && it > 0) ok = wait(L::B_DKVFREE, static_cast<uint32_t>(it - 1) & 1u);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dO_mn = sdesc_sw128(sdO + s * L::TILE, CHUNK_BYTES, 1024);
                const uint64_t dQ_mn = sdesc_sw128(sQ + s * L::TILE, CHUNK_BYTES, 1024);
                const uint64_t dK_mn = sdesc_sw128(sK + ks * L::TILE, CHUNK_BYTES, 1024);
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>((kk * 2048) >> 4);
                    mma_ts_warp(tmem + L::DV_COL, tmem + L::P_COL + kk * 8, dO_mn + off, ID_KV,
                                (cur.t > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk) {
                    const uint64_t aoff = static_cast<uint64_t>(((kk / 4) * CHUNK_BYTES + (kk % 4) * 32) >> 4);
                    const uint64_t boff = static_cast<uint64_t>((kk * 2048) >> 4);
                    mma_ss_warp(tmem + L::DK_COL, dS_k + aoff, dQ_mn + boff, ID_KV,
                                (cur.t > 0 || kk > 0) ? 1u : 0u);
                }
                // the last reads of this tile's Q and dO are issued: the producer may
                // refill the slot (dQ = dS K below reads neither)
                mma_commit_warp(bar(L::B_QEMPTY + s));
                // the item's dV and dK are final after its last tile's products above
                // (its epilogue stages them outside the dS area, which dQ still reads)
                if (cur.t == cur.w.nt - 1) mma_commit_warp(bar(L::B_DKVDONE));
                // the previous tile's dQ must have left its columns
                if (gt > 0 && !wait(L::B_DQFREE, parity ^ 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>((kk * 2048) >> 4);
                    mma_ss_warp(tmem + L::DQ_COL, dS_mn + off, dK_mn + off, ID_DQ, kk > 0 ? 1u : 0u);
                }
                mma_commit_warp(bar(L::B_BDONE));
                if (cur.t == cur.w.nt - 1) {
                    mma_commit_warp(bar(L::B_KVEMPTY + ks));
                    ++it;
                }
                ++gt;
                cur.next(p, num_units);
            }
            if (warp == L::WARP_MMA) {
                mma_commit_warp(bar(L::B_DRAIN));
                drain(bar(L::B_DRAIN), 0, 100000000ull);
            }
        }
        __syncwarp();
    } else {
        // ================================================== Pᵀ / dS, dQ read-out, epilogue
        regs_inc<L::REG_COMPUTE>();
        const int wq = warp % 4;                      // lane quadrant
        const int half = warp / 4;                    // column half
        const int r = 32 * wq + lane;                 // TMEM lane: a key here, a query row for dQ
        const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;
        const float sl2 = p.scale_log2;
        bool ok = true;
        bool bulk_pending = false;   // this warp has committed bulk groups (reduce-adds, stores)
        int gt = 0, it = 0;
        int prev_q0 = 0, prev_bh = 0;
        bool has_prev = false;       // a tile whose dQ is still to be read out
        auto wait_bulk_read = [&]() {
            if (bulk_pending && lane == 0) bulk_wait_group_read0();
            __syncwarp();
        };

        if (p.debug_flags & DEBUG_FORCE_TIMEOUT) {
            ok = mbar_wait(bar(L::B_NEVER), 0, abort_word, p.status, STATUS_FORCED, 20000000ull);
            ok = __all_sync(0xffffffffu, ok);
        }
        // dQ of the previous tile (in tensor memory once its B_BDONE completed): this
        // warpgroup's 32 columns -> its staging chunk -> TMA reduce-add
        auto dq_out = [&]() {
            uint32_t a[32];
            tmem_ld32(tmem + lane_base + L::DQ_COL + 32 * half, a);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(L::B_DQFREE));
            wait_bulk_read();
            const uint32_t row_base = sdQ + half * CHUNK_BYTES + r * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t addr = row_base + ((static_cast<uint32_t>(q) ^ static_cast<uint32_t>(r & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a[4 * q]),
                             "r"(a[4 * q + 1]), "r"(a[4 * q + 2]), "r"(a[4 * q + 3])
                             : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && prev_q0 + 32 * wq < p.n) {
                dq_reduce_add(&maps.dq_acc, sdQ + half * CHUNK_BYTES + wq * 32 * 128, 32 * half, prev_q0 + 32 * wq,
                              prev_bh);
                bulk_commit_group();
                bulk_pending = true;
            }
            __syncwarp();
            has_prev = false;
        };

        for (int u = static_cast<int>(blockIdx.x); ok && u < num_units; u += static_cast<int>(gridDim.x)) {
            const int n_items = bwd_items_of_unit<MASK>(u, p);
            for (int iu = 0; ok && iu < n_items; ++iu) {
                const BwdItem w = bwd_item<MASK>(u, iu, p);
                if (w.nt == 0) {
                    // no query sees these keys: their gradients are zero
                    if (w.k0 < p.m) {
                        const int rows = min(BN, p.m - w.k0);
                        const int64_t base = (static_cast<int64_t>(w.bh) * p.m + w.k0) * D;
                        uint4* gk = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dK) + base);
                        uint4* gv = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dV) + base);
                        for (int i = threadIdx.x; i < rows * D / 8; i += L::COMPUTE_THREADS) {
                            gk[i] = make_uint4(0u, 0u, 0u, 0u);
                            gv[i] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    continue;
                }
                const int key = w.k0 + r;
                const float sb = BIAS ? __ldg(p.slopes + w.bh % p.H) * 1.44269504088896341f : 0.f;   // log2 domain
                for (int t = 0; ok && t < w.nt; ++t) {
                    const int s = gt % L::QS;
                    const uint32_t parity = static_cast<uint32_t>(gt) & 1u;
                    const int q0 = (w.qb_lo + t) * BM;
                    ok = mbar_wait_suspend(bar(L::B_QFULL + s), static_cast<uint32_t>(gt / L::QS) & 1u, abort_word, p.status,
                                   STATUS_SOFTMAX_WAIT, limit, 2000u) &&
                         mbar_wait_suspend(bar(L::B_SFULL), parity, abort_word, p.status, STATUS_SOFTMAX_WAIT, limit, 2000u);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    const int c0 = 64 * half;         // this warpgroup's first query column
                    uint32_t sr[64], dr[64];
                    tmem_ld32(tmem + lane_base + L::S_COL + c0, sr);
                    tmem_ld32(tmem + lane_base + L::S_COL + c0 + 32, sr + 32);
                    tmem_ld32(tmem + lane_base + L::DP_COL + c0, dr);
                    tmem_ld32(tmem + lane_base + L::DP_COL + c0 + 32, dr + 32);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(bar(L::B_RDONE));    // the MMA warp may compute the next Sᵀ, dPᵀ
                    const uint32_t lse_s = sbase + L::LSE_OFF + (s * BM + c0) * 4;
                    const uint32_t dd_s = sbase + L::DD_OFF + (s * BM + c0) * 4;
                    const float d1 = static_cast<float>(q0 + c0 + w.off - key);
                    const bool need_mask =
                        __any_sync(0xffffffffu, key >= w.kv_len || q0 + c0 + 63 >= p.n ||
                                                    (mask_is_causal(MASK) && key > q0 + c0 + w.off));
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        float lz[32];
#pragma unroll
                        for (int v = 0; v < 8; ++v) lds_v4f(lse_s + (32 * c + 4 * v) * 4, lz + 4 * v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int j = 32 * c + i;
                            // with the distance bias −sb |i' − key| of query column j under BIAS
                            const float z = BIAS ? fmaf(-sb, fabsf(d1 + static_cast<float>(j)), -lz[i]) : -lz[i];
                            sr[j] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(sr[j]), sl2, z)));
                        }
                    }
                    if (need_mask) {
                        const int q_first =
                            key >= w.kv_len ? INT32_MAX : (mask_is_causal(MASK) ? key - w.off : 0);
                        const int j_lo = q_first == INT32_MAX ? BM : max(q_first - q0, 0) - c0;
                        const int j_hi = min(p.n - q0, BM) - c0;
#pragma unroll
                        for (int j = 0; j < 64; ++j)
                            if (j < j_lo || j >= j_hi) sr[j] = 0u;
                    }
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        float dz[32];
#pragma unroll
                        for (int v = 0; v < 8; ++v) lds_v4f(dd_s + (32 * c + 4 * v) * 4, dz + 4 * v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int j = 32 * c + i;
                            dr[j] = __float_as_uint(__uint_as_float(sr[j]) * (__uint_as_float(dr[j]) - dz[i]));
                        }
                    }
                    // the previous tile's dV, dK, dQ have consumed Pᵀ and dS
                    if (gt > 0) {
                        ok = mbar_wait_suspend(bar(L::B_BDONE), parity ^ 1u, abort_word, p.status, STATUS_SOFTMAX_WAIT,
                                       limit, 2000u);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    {
                        uint32_t pk[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            pk[i] = pack_bf16x2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]));
                        tmem_st32(tmem + lane_base + L::P_COL + 32 * half, pk);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            pk[i] = pack_bf16x2(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1]));
                        const uint32_t row_base = sdS + half * CHUNK_BYTES + r * 128;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const uint32_t addr =
                                row_base + ((static_cast<uint32_t>(q) ^ static_cast<uint32_t>(r & 7)) << 4);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * q]),
                                         "r"(pk[4 * q + 1]), "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                                         : "memory");
                        }
                    }
                    tmem_wait_st();
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(L::B_PFULL));
                    if (has_prev) dq_out();           // B_BDONE of the previous tile was waited for above
                    prev_q0 = q0;
                    prev_bh = w.bh;
                    has_prev = true;
                    ++gt;
                }
                if (!ok) break;

                // ---------------------------------------- this item's dV and dK (x scale)
                // Warpgroup 0 takes dV, warpgroup 1 dK: each warp reads its 32 rows, all
                // 64 columns, out of tensor memory (the next item's first dV, dK may then
                // overwrite them), stages them in its own dQ staging chunk (the last
                // tile's dQ = dS K may still be reading the dS area) once its earlier
                // reduce-adds have read it, and stores them with one TMA store.
                ok = mbar_wait_suspend(bar(L::B_DKVDONE), static_cast<uint32_t>(it) & 1u, abort_word, p.status,
                               STATUS_SOFTMAX_WAIT, limit, 2000u);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t o[64];
                const uint32_t col = half == 0 ? L::DV_COL : L::DK_COL;
                tmem_ld32(tmem + lane_base + col, o);
                tmem_ld32(tmem + lane_base + col + 32, o + 32);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(L::B_DKVFREE));
                const float mul = half == 0 ? 1.f : p.scale;
                wait_bulk_read();
                const uint32_t chunk_base = sdQ + half * CHUNK_BYTES + r * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    uint32_t v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        v[e] = pack_bf16x2(__uint_as_float(o[8 * q + 2 * e]) * mul,
                                           __uint_as_float(o[8 * q + 2 * e + 1]) * mul);
                    const uint32_t addr = chunk_base + ((static_cast<uint32_t>(q) ^ static_cast<uint32_t>(r & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]),
                                 "r"(v[2]), "r"(v[3])
                                 : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && w.k0 + 32 * wq < p.m) {
                    tma_store_3d(half == 0 ? &maps.dv : &maps.dk, sdQ + half * CHUNK_BYTES + wq * 32 * 128, 0,
                                 w.k0 + 32 * wq, w.bh);
                    bulk_commit_group();
                    bulk_pending = true;
                }
                __syncwarp();
                ++it;
            }
        }
        if (ok && has_prev) {
            // the last tile's dQ
            ok = mbar_wait_suspend(bar(L::B_BDONE), static_cast<uint32_t>(gt - 1) & 1u, abort_word, p.status,
                           STATUS_SOFTMAX_WAIT, limit, 2000u);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after();
                dq_out();
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

template <int DK, int DV, int MASK, bool BIAS = false>
cudaError_t launch(const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    constexpr bool PIPE = DK == 64 && DV == 64;
    using L = typename std::conditional<PIPE, LayoutPipe, Layout<DK, DV>>::type;
    auto kern = PIPE ? attn_bwd_pipe_kernel<MASK, BIAS> : attn_bwd_kernel<DK, DV, MASK, BIAS>;
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
    int64_t grid = static_cast<int64_t>(p.B) * p.H * p.num_kblocks;
    if (PIPE) {
        // persistent: one CTA per SM over units of one or two key tiles
        const int64_t units = static_cast<int64_t>(p.B) * p.H *
                              (mask_is_causal(MASK) ? (p.num_kblocks + 1) / 2 : p.num_kblocks);
        grid = units < p.num_sms ? units : p.num_sms;
    }
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(L::NUM_THREADS), L::BYTES, stream, maps, p);
}

}  // namespace bwd
}  // namespace attn
