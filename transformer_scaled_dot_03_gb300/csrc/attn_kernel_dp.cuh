// attn_kernel_dp.cuh -- sm_103a attention forward: persistent CTAs, 128-row query
// tiles, P held apart from S in tensor memory ("decoupled P").
//
// Computes the scaled dot-product attention of "Transformer 详解" §4.1-§4.2
// (scores = Q Kᵀ / sqrt(d_k), the causal mask of §5.3, the key-padding mask of
// §3.4 or both at once, row softmax, weights x V) with an online softmax over
// 128-key tiles, per (batch, head) pair. Under the causal mask query row i sees
// keys j <= i + (m - n): the n queries are the last n of the m positions.
//
// Schedule. A work unit is one (b, h) pair and one 128-row query tile (two
// tiles, longest with shortest, under the causal mask); each CTA takes units
// blockIdx.x, blockIdx.x + gridDim.x, ... Within a tile, P (bf16) has its own
// tensor-memory columns, so the softmax warps release the score tile S as soon
// as they have loaded it and the MMA warp computes S_{j+1} = Q K_{j+1}ᵀ while the
// softmax of key tile j is still running; O += P_j V_j runs behind. Across
// tiles, the next tile's Q is loaded early and its first S runs while the
// softmax warps write O out, so set-up and epilogue overlap neighbouring tiles.
// At d = 128 the S MMA takes Q from tensor memory (the softmax warps copy each
// tile's Q there from shared memory), so only K is read from shared memory;
// with both operands in shared memory the S MMA is bound by its bandwidth.
//
//   warps 0-3   softmax + epilogue (TMEM lanes 0-127 = the tile's query rows)
//   warp  4     TMA producer: Q, then a K ring and a V ring (K runs one tile ahead)
//   warp  5     tcgen05.mma issuer, owns the TMEM allocation
//   warps 6-7   idle (complete the control warpgroup for setmaxnreg)
// Tensor memory: S [0,128), P [128,192), O [192,192+d_v), at d_k = 128 also two
// Q buffers of 64 columns after O.
//   d_k = d_v = 64: 256 columns, 96 KB shared memory -> two CTAs per SM
//   otherwise     : 512 columns, up to 224 KB shared memory -> one CTA per SM
// O leaves through a shared-memory staging tile and per-warp TMA stores that
// are only waited for before the staging tile is reused.
//
// BIAS adds the linear distance bias of "第2章：完整的 Transformer 架构" §5.3
// (ALiBi): every scaled score gets -m_h |i' - j|, i' = i + (m - n) the query's
// position among the keys and m_h the slope of the head. The softmax warps form
// x = s * scale*log2e + bias first (a ramp in the column when the whole tile lies
// on one side of a warp's diagonal, the distance itself on the tiles that
// straddle it) and take the row maximum and the exponentials of x.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "attn_softmax.cuh"
#include "sm103a.cuh"

namespace attn {

using namespace sm103a;

namespace dp {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int CHUNK_BYTES = BM * 64 * 2;
constexpr float LN2 = 0.693147180559945309f;
constexpr float LOG2E = smx::LOG2E;

// Q and K tiles are 128 x d_k, V and O tiles 128 x d_v, each stored as 64-column
// chunks of 16 KB (128-byte rows, 128-byte swizzle).
template <int DK, int DV>
struct Layout {
    static constexpr int CHK = DK / 64;
    static constexpr int CHV = DV / 64;
    static constexpr int TILE_K = CHK * CHUNK_BYTES;   // a Q or K tile
    static constexpr int TILE_V = CHV * CHUNK_BYTES;   // a V or O tile
    static constexpr int NUM_THREADS = 256;
    static constexpr int WARP_TMA = 4;
    static constexpr int WARP_MMA = 5;
    static constexpr bool SMALL = DK == 64 && DV == 64;
    static constexpr int CTAS_PER_SM = SMALL ? 2 : 1;
    static constexpr bool Q_IN_TMEM = DK == 128;
    static constexpr int KS = SMALL ? 2 : 3;           // K ring depth
    static constexpr int VS = 2;                       // V ring depth
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + TILE_K;
    static constexpr int V_OFF = K_OFF + KS * TILE_K;
    static constexpr int OST_OFF = V_OFF + VS * TILE_V;  // O staging tile
    static constexpr int BAR_OFF = OST_OFF + TILE_V;
    static constexpr int B_QFULL = 0;               // Q of a tile loaded               (tx)
    static constexpr int B_QFREE = 1;               // Q buffer may be refilled
    static constexpr int B_QREADY = 2;              // Q copied into tensor memory      (128 arrivals)
    static constexpr int B_KFULL = 3;
    static constexpr int B_KEMPTY = B_KFULL + KS;
    static constexpr int B_VFULL = B_KEMPTY + KS;
    static constexpr int B_VEMPTY = B_VFULL + VS;
    static constexpr int B_SFULL = B_VEMPTY + VS;   // S computed               (commit)
    static constexpr int B_SFREE = B_SFULL + 1;     // S loaded by the softmax  (128 arrivals)
    static constexpr int B_PFULL = B_SFREE + 1;     // P written                (128 arrivals)
    static constexpr int B_PVDONE = B_PFULL + 1;    // O += P V completed       (commit)
    static constexpr int B_DRAIN = B_PVDONE + 1;
    static constexpr int B_NEVER = B_DRAIN + 1;
    static constexpr int NBARS = B_NEVER + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BYTES = MISC_OFF + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = SMALL ? 256 : 512;
    static constexpr uint32_t S_COL = 0, P_COL = 128, O_COL = 192, QT_COL = 192 + DV;
    static constexpr uint32_t REG_LAUNCH = (65536 / (NUM_THREADS * CTAS_PER_SM)) / 8 * 8;
    static constexpr uint32_t REG_CTRL = 72;
    static constexpr uint32_t REG_SOFTMAX_FIT = ((REG_LAUNCH * NUM_THREADS - REG_CTRL * 128) / 128) / 8 * 8;
    static constexpr uint32_t REG_SOFTMAX = REG_SOFTMAX_FIT > 248 ? 248 : REG_SOFTMAX_FIT;
    static_assert(128 * REG_SOFTMAX + 128 * REG_CTRL <= REG_LAUNCH * NUM_THREADS, "register split");
    static_assert((Q_IN_TMEM ? QT_COL + DK : O_COL + DV) <= TMEM_COLS, "tensor memory layout");
    static_assert(BYTES <= (CTAS_PER_SM == 2 ? 115712 : 232448), "shared memory budget");
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_test(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

// One query tile of work: (b, h) pair, first query row, key tiles to visit.
struct Unit {
    int bh, q0, kv_len, nkv;
    int off;   // query row i sits at key position i + off (the causal masks' diagonal)
};

// Work units are numbered head-major so that concurrently running units share
// K/V in L2. Without a causal mask a unit is one 128-row query tile. With it,
// a unit pairs query tile k with tile nqb-1-k of the same head (the longest with
// the shortest), so that every unit visits the same number of key tiles and a
// plain round-robin over units balances the CTAs.
__host__ __device__ inline int units_per_head(int num_qblocks, int mask)
{
    return mask_is_causal(mask) ? (num_qblocks + 1) / 2 : num_qblocks;
}

template <int MASK>
__device__ __forceinline__ int tiles_of_unit(int u, const FwdParams& p)
{
    if (!mask_is_causal(MASK)) return 1;
    const int k = u % units_per_head(p.num_qblocks, MASK);
    return (k == p.num_qblocks - 1 - k) ? 1 : 2;
}

template <int MASK>
__device__ __forceinline__ Unit tile_of(int u, int i, const FwdParams& p)
{
    Unit w;
    const int uph = units_per_head(p.num_qblocks, MASK);
    w.bh = u / uph;
    const int k = u % uph;
    const int qb = mask_is_causal(MASK) ? (i == 0 ? p.num_qblocks - 1 - k : k) : k;
    w.q0 = qb * BM;
    w.kv_len = p.m;
    if (mask_has_lengths(MASK)) {
        const int len = __ldg(p.key_lengths + w.bh / p.H);
        w.kv_len = len < 0 ? 0 : (len > p.m ? p.m : len);
    }
    w.nkv = (w.kv_len + BN - 1) / BN;
    w.off = causal_offset(MASK, p.causal_off, w.kv_len, p.n);
    if (mask_is_causal(MASK)) {
        // the last key visible to the tile's last row; none if it is negative
        const int last = min(w.q0 + BM - 1, p.n - 1) + w.off;
        w.nkv = last < 0 ? 0 : min(last / BN + 1, w.nkv);
    }
    return w;
}

// Position in this CTA's sequence of tiles: unit u, tile ti of that unit.
struct TilePos {
    int u, ti;
};

template <int MASK>
__device__ __forceinline__ void advance(TilePos& t, int u_step, const FwdParams& p)
{
    if (++t.ti >= tiles_of_unit<MASK>(t.u, p)) {
        t.ti = 0;
        t.u += u_step;
    }
}

template <int DK, int DV, int MASK, bool BIAS>
__global__ void __launch_bounds__(Layout<DK, DV>::NUM_THREADS, Layout<DK, DV>::CTAS_PER_SM)
attn_fwd_dp_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const FwdParams p)
{
    using L = Layout<DK, DV>;
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
    const int u_step = static_cast<int>(gridDim.x);
    const TilePos first_tile{static_cast<int>(blockIdx.x), 0};

    if (threadIdx.x == 0) {
        mbar_init(bar(L::B_QFULL), 1);
        mbar_init(bar(L::B_QFREE), L::Q_IN_TMEM ? BM : 1);
        mbar_init(bar(L::B_QREADY), BM);
        for (int s = 0; s < L::KS; ++s) {
            mbar_init(bar(L::B_KFULL + s), 1);
            mbar_init(bar(L::B_KEMPTY + s), 1);
        }
        for (int s = 0; s < L::VS; ++s) {
            mbar_init(bar(L::B_VFULL + s), 1);
            mbar_init(bar(L::B_VEMPTY + s), 1);
        }
        mbar_init(bar(L::B_SFULL), 1);
        mbar_init(bar(L::B_SFREE), BM);
        mbar_init(bar(L::B_PFULL), BM);
        mbar_init(bar(L::B_PVDONE), 1);
        mbar_init(bar(L::B_DRAIN), 1);
        mbar_init(bar(L::B_NEVER), 1);
        *abort_word = 0u;
        fence_mbar_init();
    }
    if (warp == L::WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == L::WARP_TMA && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Everything above touches no global memory: under a programmatic dependent
    // launch it may run before the previous grid in the stream has finished,
    // whose results (Q, K, V, the key lengths) are read only after this wait.
    // (Explicit triggers for the next grid, at a CTA's start or at its last
    // unit, measured slower than the implicit one at this grid's completion.)
    griddep_wait();

    const uint32_t sQ = sbase + L::Q_OFF;
    const uint32_t sK = sbase + L::K_OFF;
    const uint32_t sV = sbase + L::V_OFF;
    const uint32_t sO = sbase + L::OST_OFF;

    if (warp >= 4) {
        regs_dec<L::REG_CTRL>();
        if (warp == L::WARP_TMA && lane == 0) {
            // ================================================== TMA producer
            // Running counts over all tiles of this CTA give every ring slot's phase.
            int qc = 0, kc = 0, vc = 0;
            bool ok = true;
            auto load_K = [&](int bh, int j) -> bool {
                const int s = kc % L::KS;
                if (kc >= L::KS &&
                    !mbar_wait_suspend(bar(L::B_KEMPTY + s), static_cast<uint32_t>(kc / L::KS - 1) & 1u,
                               abort_word, p.status, STATUS_TMA_WAIT, limit, 2000u))
                    return false;
                mbar_arrive_expect_tx(bar(L::B_KFULL + s), L::TILE_K);
                for (int c = 0; c < L::CHK; ++c)
                    tma_load_3d(sK + s * L::TILE_K + c * CHUNK_BYTES, &tmK, bar(L::B_KFULL + s), c * 64,
                                j * BN, bh);
                ++kc;
                return true;
            };
            auto load_V = [&](int bh, int j) -> bool {
                const int s = vc % L::VS;
                if (vc >= L::VS &&
                    !mbar_wait_suspend(bar(L::B_VEMPTY + s), static_cast<uint32_t>(vc / L::VS - 1) & 1u,
                               abort_word, p.status, STATUS_TMA_WAIT, limit, 2000u))
                    return false;
                mbar_arrive_expect_tx(bar(L::B_VFULL + s), L::TILE_V);
                for (int c = 0; c < L::CHV; ++c)
                    tma_load_3d(sV + s * L::TILE_V + c * CHUNK_BYTES, &tmV, bar(L::B_VFULL + s), c * 64,
                                j * BN, bh);
                ++vc;
                return true;
            };
            for (TilePos t = first_tile; ok && t.u < p.num_units; advance<MASK>(t, u_step, p)) {
                const Unit w = tile_of<MASK>(t.u, t.ti, p);
                if (w.nkv == 0) continue;
                // the previous tile's Q must have left the buffer
                if (qc > 0 && !mbar_wait_suspend(bar(L::B_QFREE), static_cast<uint32_t>(qc - 1) & 1u, abort_word,
                                         p.status, STATUS_TMA_WAIT, limit, 2000u)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(L::B_QFULL), L::TILE_K);
                for (int c = 0; c < L::CHK; ++c)
                    tma_load_3d(sQ + c * CHUNK_BYTES, &tmQ, bar(L::B_QFULL), c * 64, w.q0, w.bh);
                ++qc;
                // K(j+1) is issued before V(j): S(j+1) needs it while P(j) is computed
                ok = load_K(w.bh, 0);
                for (int j = 0; ok && j < w.nkv; ++j) {
                    if (j + 1 < w.nkv) ok = load_K(w.bh, j + 1);
                    if (ok) ok = load_V(w.bh, j);
                }
            }
            // land every copy still in flight (only possible after an abort)
            if (qc > 0) drain_wait(bar(L::B_QFULL), static_cast<uint32_t>(qc - 1) & 1u, 100000000ull);
            for (int i = kc - 1; i >= 0 && i >= kc - L::KS; --i)
                drain_wait(bar(L::B_KFULL + i % L::KS), static_cast<uint32_t>(i / L::KS) & 1u, 100000000ull);
            for (int i = vc - 1; i >= 0 && i >= vc - L::VS; --i)
                drain_wait(bar(L::B_VFULL + i % L::VS), static_cast<uint32_t>(i / L::VS) & 1u, 100000000ull);
        } else if (warp == L::WARP_MMA) {
            // ================================================== MMA issuer
            // The whole warp runs this loop with warp-uniform values; one elected
            // lane issues each tcgen05 instruction. Descriptors are formed once per
            // buffer and advanced by adding the encoded byte offset (address >> 4).
            constexpr uint32_t ID_S = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t ID_PV = idesc_bf16_f32(BM, DV, false, true);
            const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
            const uint64_t dK0 = sdesc_sw128(sK, 16, 1024);
            const uint64_t dV0 = sdesc_sw128(sV, CHUNK_BYTES, 1024);
            int qc = 0, kc = 0, vc = 0, g = 0;   // g: key-tile steps over all tiles
            auto wait = [&](int b, uint32_t parity) -> bool {
                const bool r = mbar_wait_suspend(bar(b), parity, abort_word, p.status, STATUS_MMA_WAIT, limit, 2000u);
                return __all_sync(0xffffffffu, r);
            };
            auto issue_S = [&](int s) {
                const uint64_t dK = dK0 + static_cast<uint64_t>((s * L::TILE_K) >> 4);
                const uint32_t qt = tmem + L::QT_COL + static_cast<uint32_t>((qc - 1) & 1) * (DK / 2);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk / 4) * CHUNK_BYTES + (kk % 4) * 32) >> 4);
                    if (L::Q_IN_TMEM)
                        mma_ts_warp(tmem + L::S_COL, qt + kk * 8, dK + off, ID_S, kk > 0 ? 1u : 0u);
                    else
                        mma_ss_warp(tmem + L::S_COL, dQ + off, dK + off, ID_S, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_PV = [&](int s, bool acc) {
                const uint64_t dV = dV0 + static_cast<uint64_t>((s * L::TILE_V) >> 4);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts_warp(tmem + L::O_COL, tmem + L::P_COL + kk * 8, dV + static_cast<uint64_t>((kk * 2048) >> 4),
                                ID_PV, (acc || kk > 0) ? 1u : 0u);
            };
            bool ok = true;
            // S(g) for the key tile in ring slot kc; waits for the data and for the
            // softmax to have loaded S(g-1) out of the S columns.
            auto next_S = [&](bool last_of_tile) -> bool {
                const int s = kc % L::KS;
                if (!wait(L::B_KFULL + s, static_cast<uint32_t>(kc / L::KS) & 1u)) return false;
                if (g > 0 && !wait(L::B_SFREE, static_cast<uint32_t>(g - 1) & 1u)) return false;
                tc_fence_after();
                issue_S(s);
                mma_commit_warp(bar(L::B_SFULL));
                mma_commit_warp(bar(L::B_KEMPTY + s));
                if (last_of_tile && !L::Q_IN_TMEM) mma_commit_warp(bar(L::B_QFREE));
                ++kc;
                ++g;
                return true;
            };
            for (TilePos t = first_tile; ok && t.u < p.num_units; advance<MASK>(t, u_step, p)) {
                const Unit w = tile_of<MASK>(t.u, t.ti, p);
                if (w.nkv == 0) continue;
                ok = wait(L::Q_IN_TMEM ? L::B_QREADY : L::B_QFULL, static_cast<uint32_t>(qc) & 1u);
                ++qc;
                if (ok) ok = next_S(w.nkv == 1);
                for (int j = 0; ok && j < w.nkv; ++j) {
                    if (j + 1 < w.nkv) {
                        ok = next_S(j + 2 == w.nkv);
                        if (!ok) break;
                    }
                    const int sv = vc % L::VS;
                    const int step = g - (j + 1 < w.nkv ? 2 : 1);   // this tile's step j
                    ok = wait(L::B_VFULL + sv, static_cast<uint32_t>(vc / L::VS) & 1u) &&
                         wait(L::B_PFULL, static_cast<uint32_t>(step) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    issue_PV(sv, j > 0);
                    mma_commit_warp(bar(L::B_PVDONE));
                    mma_commit_warp(bar(L::B_VEMPTY + sv));
                    ++vc;
                }
            }
            mma_commit_warp(bar(L::B_DRAIN));
            drain_wait(bar(L::B_DRAIN), 0, 100000000ull);
        }
        __syncwarp();
    } else {
        // ================================================== softmax + epilogue
        regs_inc<L::REG_SOFTMAX>();
        const int r = 32 * warp + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        const uint32_t tS = tmem + lane_base + L::S_COL;
        const uint32_t tP = tmem + lane_base + L::P_COL;
        const uint32_t tO = tmem + lane_base + L::O_COL;
        const float sl2 = p.scale_log2;
        bool ok = true;
        int g = 0;        // key-tile steps over all tiles
        int qc = 0;       // tiles whose Q went into tensor memory
        TilePos q_done{-1, 0};   // last tile whose Q was copied
        bool store_pending = false;

        if (p.debug_flags & DEBUG_FORCE_TIMEOUT) {
            ok = mbar_wait(bar(L::B_NEVER), 0, abort_word, p.status, STATUS_FORCED, 20000000ull);
            ok = __all_sync(0xffffffffu, ok);
        }

        // Copy a tile's Q row from shared memory (128-byte swizzle) into the
        // tensor-memory Q buffer the S MMA reads, then free the shared buffer.
        auto copy_q = [&]() -> bool {
            bool w_ok = mbar_wait_suspend(bar(L::B_QFULL), static_cast<uint32_t>(qc) & 1u, abort_word, p.status,
                                  STATUS_SOFTMAX_WAIT, limit, 2000u);
            w_ok = __all_sync(0xffffffffu, w_ok);
            if (!w_ok) return false;
            const uint32_t qt = tmem + lane_base + L::QT_COL + static_cast<uint32_t>(qc & 1) * (DK / 2);
#pragma unroll
            for (int c = 0; c < L::CHK; ++c) {
                uint32_t q[32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t addr = sQ + c * CHUNK_BYTES + r * 128 +
                                          ((static_cast<uint32_t>(k) ^ static_cast<uint32_t>(r & 7)) << 4);
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(q[4 * k]), "=r"(q[4 * k + 1]), "=r"(q[4 * k + 2]), "=r"(q[4 * k + 3])
                                 : "r"(addr)
                                 : "memory");
                }
                tmem_st32(qt + 32 * c, q);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(L::B_QFREE));
            mbar_arrive(bar(L::B_QREADY));
            ++qc;
            return true;
        };

        for (TilePos t = first_tile; ok && t.u < p.num_units; advance<MASK>(t, u_step, p)) {
            const Unit w = tile_of<MASK>(t.u, t.ti, p);
            const int qrow = w.q0 + r;
            const int qlim = qrow + w.off;   // the row's key position: last key it sees under the causal mask
            // distance-bias slope of the head, log2 domain
            const float sb = BIAS ? __ldg(p.slopes + w.bh % p.H) * LOG2E : 0.f;
            float m_ref = -INFINITY;
            float l_run = 0.f;
            if (L::Q_IN_TMEM && w.nkv > 0 && !(q_done.u == t.u && q_done.ti == t.ti)) {
                ok = copy_q();
                if (!ok) break;
                q_done = t;
            }

            for (int j = 0; j < w.nkv; ++j, ++g) {
                ok = mbar_wait_suspend(bar(L::B_SFULL), static_cast<uint32_t>(g) & 1u, abort_word, p.status,
                               STATUS_SOFTMAX_WAIT, limit, 2000u);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();

                uint32_t sr[BN];
                tmem_ld32(tS + 0, sr + 0);
                tmem_ld32(tS + 32, sr + 32);
                tmem_ld32(tS + 64, sr + 64);
                tmem_ld32(tS + 96, sr + 96);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(L::B_SFREE));      // S may now be overwritten by the next S

                float s[BN];
#pragma unroll
                for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c]);
                uint32_t pk[BN / 2];
                const float alpha = smx::tile_step<MASK, BIAS>(s, j * BN, w.kv_len, qlim, sl2, sb, m_ref, l_run, pk);

                if (g > 0) {
                    // the previous O += P V must be complete: it reads the P columns,
                    // and O is rescaled below
                    ok = mbar_wait_suspend(bar(L::B_PVDONE), static_cast<uint32_t>(g - 1) & 1u, abort_word, p.status,
                                   STATUS_SOFTMAX_WAIT, limit, 2000u);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                }
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int cc = 0; cc < DV / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32 * cc, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + 32 * cc, o);
                    }
                }
                tmem_st32(tP + 0, pk);
                tmem_st32(tP + 32, pk + 32);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(L::B_PFULL));
            }
            if (!ok) break;

            // ---------------------------------------------- epilogue of this tile
            if (w.nkv > 0) {
                ok = mbar_wait_suspend(bar(L::B_PVDONE), static_cast<uint32_t>(g - 1) & 1u, abort_word, p.status,
                               STATUS_SOFTMAX_WAIT, limit, 2000u);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
            }
            if (L::Q_IN_TMEM) {
                // hand the next loaded tile's Q to the tensor core before writing O out,
                // so that its first S overlaps this epilogue (every MMA of this and the
                // previous tile is complete, so the Q buffer being overwritten is free)
                TilePos nt = t;
                advance<MASK>(nt, u_step, p);
                while (nt.u < p.num_units && tile_of<MASK>(nt.u, nt.ti, p).nkv == 0) advance<MASK>(nt, u_step, p);
                // (a tile without keys between two with keys finds its successor's Q
                // already copied by the tile before it)
                if (nt.u < p.num_units && !(q_done.u == nt.u && q_done.ti == nt.ti)) {
                    ok = copy_q();
                    if (!ok) break;
                    q_done = nt;
                }
            }
            const bool any = l_run > 0.f;
            const float inv_l = any ? 1.f / l_run : 0.f;
            if (p.LSE != nullptr && qrow < p.n)
                p.LSE[static_cast<int64_t>(w.bh) * p.n + qrow] = any ? (m_ref + __log2f(l_run)) * LN2 : -INFINITY;
            // the previous TMA store from this warp's staging rows must have read them
            if (store_pending && lane == 0) bulk_wait_group_read0();
            __syncwarp();
#pragma unroll
            for (int cc = 0; cc < DV / 32; ++cc) {
                uint32_t o[32];
                if (w.nkv > 0) {
                    tmem_ld32(tO + 32 * cc, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                const uint32_t chunk_base = sO + (cc / 2) * CHUNK_BYTES + r * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        v[e] = pack_bf16x2(__uint_as_float(o[8 * q + 2 * e]) * inv_l,
                                           __uint_as_float(o[8 * q + 2 * e + 1]) * inv_l);
                    const uint32_t piece = static_cast<uint32_t>((cc % 2) * 4 + q);
                    const uint32_t addr = chunk_base + ((piece ^ static_cast<uint32_t>(r & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]),
                                 "r"(v[2]), "r"(v[3])
                                 : "memory");
                }
            }
            // O has been read out of tensor memory: the next tile's first O += P V may
            // overwrite it (it waits for this warpgroup's next P, written after this).
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && w.q0 + 32 * warp < p.n) {
                for (int c = 0; c < L::CHV; ++c)
                    tma_store_3d(&tmO, sO + c * CHUNK_BYTES + warp * 32 * 128, c * 64, w.q0 + 32 * warp, w.bh);
                bulk_commit_group();
                store_pending = true;
            }
            __syncwarp();
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
cudaError_t launch(const TensorMaps& maps, const FwdParams& p, int num_sms, cudaStream_t stream)
{
    using L = Layout<DK, DV>;
    auto kern = attn_fwd_dp_kernel<DK, DV, MASK, BIAS>;
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
    const int64_t slots = static_cast<int64_t>(num_sms) * L::CTAS_PER_SM;
    const int64_t grid = p.num_units < slots ? p.num_units : slots;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(L::NUM_THREADS), L::BYTES, stream, maps.q,
                      maps.k, maps.v, maps.o, p);
}

}  // namespace dp
}  // namespace attn
