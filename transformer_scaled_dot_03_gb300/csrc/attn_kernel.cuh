// attn_kernel.cuh -- sm_103a attention forward kernel (one template per head
// dim, mask kind and number of query tiles per CTA).
//
// What it computes is the scaled dot-product attention of "Transformer 详解"
// §4.1 (scores = Q Kᵀ / sqrt(d_k), mask, row softmax, weights x V), per head
// ("Transformer 详解" §4.2), with the causal mask of §5.3 or the key-padding
// mask of §3.4. The n x m score matrix only ever lives in tensor memory: the
// row softmax is computed online over 128-key tiles (running row maximum and
// row sum, earlier partial sums rescaled when the maximum grows), which gives
// the same result as the plain definition up to rounding.
//
// CTA = one (batch, head) pair x NT query tiles of 128 rows (NT = 1 or 2).
//   warps 0 .. 4NT-1   softmax + epilogue, one warpgroup per query tile
//   warp  4NT          TMA producer (Q once, K/V ring)
//   warp  4NT+1        tcgen05.mma issuer; also owns the TMEM allocation
//   warps 4NT+2, +3    idle (complete the control warpgroup for setmaxnreg)
// Tensor memory (lane = query row of a tile):
//   [t*128, t*128+128)          S/P of tile t
//   [NT*128 + t*D, +D)          O of tile t
// Per key tile j and query tile t the MMA warp issues S_t = Q_t K_jᵀ
// (SS, fp32 in TMEM), the softmax warps turn S_t into P_t (bf16, written back
// over S_t) and rescale O_t when the row maximum has grown by more than 2^8,
// then the MMA warp issues O_t += P_t V_j (TS: P from TMEM, V from shared
// memory). With NT = 2 the two tiles alternate on the tensor core; with NT = 1
// two CTAs share an SM and interleave the same way.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "sm103a.cuh"

namespace attn {

using namespace sm103a;

constexpr int BM = 128;                    // query rows per tile (TMEM lanes)
constexpr int BN = 128;                    // keys per K/V stage
constexpr int CHUNK_BYTES = BM * 64 * 2;   // [128 rows][64 bf16] = 16 KB, one TMA box
constexpr float LN2 = 0.693147180559945309f;
// The reference maximum of a row is only raised when a new score exceeds it by
// more than this many powers of two; until then exp2(x - m_ref) <= 2^8, which
// bf16 P and the fp32 sums hold exactly as well as values <= 1.
constexpr float RESCALE_LOG2 = 8.0f;

template <int D, int NT>
struct Layout {
    static constexpr int CH = D / 64;                 // 64-column chunks per row
    static constexpr int TILE = CH * CHUNK_BYTES;     // one [128][D] bf16 tile
    static constexpr int NUM_THREADS = NT * 128 + 128;
    static constexpr int WARP_TMA = NT * 4;
    static constexpr int WARP_MMA = NT * 4 + 1;
    static constexpr int CTAS_PER_SM = (NT == 1 && D == 64) ? 2 : 1;
    static constexpr int STAGES = (D == 64) ? (NT == 2 ? 4 : 2) : 2;   // K/V ring depth
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + NT * TILE;
    static constexpr int V_OFF = K_OFF + STAGES * TILE;
    static constexpr int BAR_OFF = V_OFF + STAGES * TILE;
    // barrier indices
    static constexpr int B_Q = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_VFULL = B_KFULL + STAGES;
    static constexpr int B_KVEMPTY = B_VFULL + STAGES;
    static constexpr int B_SFULL = B_KVEMPTY + STAGES;
    static constexpr int B_PFULL = B_SFULL + NT;
    static constexpr int B_OFULL = B_PFULL + NT;
    static constexpr int B_DRAIN = B_OFULL + NT;
    static constexpr int B_NEVER = B_DRAIN + 1;
    static constexpr int NBARS = B_NEVER + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;   // tmem slot, abort word
    static constexpr int BYTES = MISC_OFF + 16 + 1024;    // + slack for 1024-byte alignment
    static constexpr uint32_t TMEM_COLS = (NT * 128 + NT * D) <= 256 ? 256 : 512;
    static constexpr uint32_t O_COL = NT * 128;
    // Register split (setmaxnreg): the launch gives every thread REG_LAUNCH
    // registers; the control warpgroup drops to REG_CTRL and the softmax
    // warpgroups rise to REG_SOFTMAX, within the block's launch total.
    static constexpr uint32_t REG_LAUNCH = (65536 / (NUM_THREADS * CTAS_PER_SM)) / 8 * 8;
    static constexpr uint32_t REG_CTRL = 56;
    static constexpr uint32_t REG_SOFTMAX_FIT =
        ((REG_LAUNCH * NUM_THREADS - REG_CTRL * 128) / (NT * 128)) / 8 * 8;
    static constexpr uint32_t REG_SOFTMAX = REG_SOFTMAX_FIT > 248 ? 248 : REG_SOFTMAX_FIT;
    static_assert(NT * 128 * REG_SOFTMAX + 128 * REG_CTRL <= REG_LAUNCH * NUM_THREADS,
                  "register split exceeds the launch allocation");
};

// Wait that ignores the abort word (used to drain in-flight copies / MMAs).
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_test(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

template <int D, int MASK, int NT>
__global__ void __launch_bounds__(Layout<D, NT>::NUM_THREADS, Layout<D, NT>::CTAS_PER_SM)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                const FwdParams p)
{
    using L = Layout<D, NT>;
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

    // ---- work unit: (b, h) pair and NT*128-row query block; heavy causal blocks first
    const int bh = static_cast<int>(blockIdx.x / static_cast<uint32_t>(p.num_qblocks));
    int qb = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.num_qblocks));
    if (MASK == MASK_CAUSAL) qb = p.num_qblocks - 1 - qb;
    const int b = bh / p.H;
    const int q0 = qb * NT * BM;

    int kv_len = p.m;
    if (MASK == MASK_KEY_PADDING) {
        const int len = __ldg(p.key_lengths + b);
        kv_len = len < 0 ? 0 : (len > p.m ? p.m : len);
    }
    int nkv[NT];
    int nkv_max = 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int first = q0 + t * BM;
        if (first >= p.n) {
            nkv[t] = 0;
        } else if (MASK == MASK_CAUSAL) {
            const int last = min(first + BM - 1, p.n - 1);
            nkv[t] = min(last / BN + 1, (kv_len + BN - 1) / BN);
        } else {
            nkv[t] = (kv_len + BN - 1) / BN;
        }
        nkv_max = max(nkv_max, nkv[t]);
    }
    const uint64_t limit = p.watchdog_ns;

    // ---- set-up: barriers, TMEM
    if (threadIdx.x == 0) {
        mbar_init(bar(L::B_Q), 1);
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(bar(L::B_KFULL + s), 1);
            mbar_init(bar(L::B_VFULL + s), 1);
            mbar_init(bar(L::B_KVEMPTY + s), 1);
        }
        for (int t = 0; t < NT; ++t) {
            mbar_init(bar(L::B_SFULL + t), 1);
            mbar_init(bar(L::B_PFULL + t), BM);
            mbar_init(bar(L::B_OFULL + t), 1);
        }
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

    const uint32_t sQ = sbase + L::Q_OFF;
    const uint32_t sK = sbase + L::K_OFF;
    const uint32_t sV = sbase + L::V_OFF;

    if (warp >= NT * 4) {
        regs_dec<L::REG_CTRL>();
        if (warp == L::WARP_TMA) {
            // ================================================== TMA producer
            if (lane == 0 && nkv_max > 0) {
                uint32_t qbytes = 0;
                for (int t = 0; t < NT; ++t) qbytes += nkv[t] > 0 ? L::TILE : 0;
                mbar_arrive_expect_tx(bar(L::B_Q), qbytes);
                for (int t = 0; t < NT; ++t) {
                    if (nkv[t] == 0) continue;
                    for (int c = 0; c < L::CH; ++c)
                        tma_load_3d(sQ + t * L::TILE + c * CHUNK_BYTES, &tmQ, bar(L::B_Q), c * 64,
                                    q0 + t * BM, bh);
                }
                int issued = 0;
                for (int j = 0; j < nkv_max; ++j) {
                    const int s = j % L::STAGES;
                    const uint32_t use = static_cast<uint32_t>(j / L::STAGES);
                    if (j >= L::STAGES &&
                        !mbar_wait(bar(L::B_KVEMPTY + s), (use - 1u) & 1u, abort_word, p.status,
                                   STATUS_TMA_WAIT, limit))
                        break;
                    mbar_arrive_expect_tx(bar(L::B_KFULL + s), L::TILE);
                    for (int c = 0; c < L::CH; ++c)
                        tma_load_3d(sK + s * L::TILE + c * CHUNK_BYTES, &tmK, bar(L::B_KFULL + s),
                                    c * 64, j * BN, bh);
                    mbar_arrive_expect_tx(bar(L::B_VFULL + s), L::TILE);
                    for (int c = 0; c < L::CH; ++c)
                        tma_load_3d(sV + s * L::TILE + c * CHUNK_BYTES, &tmV, bar(L::B_VFULL + s),
                                    c * 64, j * BN, bh);
                    issued = j + 1;
                }
                // Every copy still in flight (possible only after an abort) must land
                // before shared memory is released; completed phases return at once.
                drain_wait(bar(L::B_Q), 0, 100000000ull);
                for (int j = issued - 1; j >= 0 && j >= issued - L::STAGES; --j) {
                    const int s = j % L::STAGES;
                    const uint32_t ph = static_cast<uint32_t>(j / L::STAGES) & 1u;
                    drain_wait(bar(L::B_KFULL + s), ph, 100000000ull);
                    drain_wait(bar(L::B_VFULL + s), ph, 100000000ull);
                }
            }
        } else if (warp == L::WARP_MMA) {
            // ================================================== MMA issuer
            if (lane == 0 && nkv_max > 0) {
                constexpr uint32_t ID_S = idesc_bf16_f32(BM, BN, false, false);
                constexpr uint32_t ID_PV = idesc_bf16_f32(BM, D, false, true);
                // S_t = Q_t K_sᵀ : D/16 MMAs of K = 16 (32 bytes along each 128-byte row)
                auto issue_S = [&](int t, int s) {
                    const uint32_t a0 = sQ + t * L::TILE, b0 = sK + s * L::TILE;
                    const uint32_t dcol = tmem + t * 128;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk / 4) * CHUNK_BYTES + (kk % 4) * 32;
                        mma_ss(dcol, sdesc_sw128(a0 + off, 16, 1024), sdesc_sw128(b0 + off, 16, 1024),
                               ID_S, kk > 0 ? 1u : 0u);
                    }
                };
                // O_t += P_t V_s : 8 MMAs of K = 16 keys; P from TMEM (8 columns per step),
                // V MN-major: 16 keys = two 8-row atoms (2048 bytes), 64-column chunks 16 KB apart
                auto issue_PV = [&](int t, int s, bool acc) {
                    const uint32_t v0 = sV + s * L::TILE;
                    const uint32_t pcol = tmem + t * 128;
                    const uint32_t dcol = tmem + L::O_COL + t * D;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ts(dcol, pcol + kk * 8, sdesc_sw128(v0 + kk * 2048, CHUNK_BYTES, 1024),
                               ID_PV, (acc || kk > 0) ? 1u : 0u);
                };

                bool ok = mbar_wait(bar(L::B_Q), 0, abort_word, p.status, STATUS_MMA_WAIT, limit) &&
                          mbar_wait(bar(L::B_KFULL + 0), 0, abort_word, p.status, STATUS_MMA_WAIT, limit);
                tc_fence_after();
                if (ok) {
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        if (nkv[t] == 0) continue;
                        issue_S(t, 0);
                        mma_commit(bar(L::B_SFULL + t));
                    }
                }
                for (int j = 0; ok && j < nkv_max; ++j) {
                    const int s = j % L::STAGES;
                    const uint32_t ph = static_cast<uint32_t>(j / L::STAGES) & 1u;
                    ok = mbar_wait(bar(L::B_VFULL + s), ph, abort_word, p.status, STATUS_MMA_WAIT, limit);
                    if (!ok) break;
                    bool knext = false;
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        if (!ok || j >= nkv[t]) continue;
                        ok = mbar_wait(bar(L::B_PFULL + t), static_cast<uint32_t>(j) & 1u, abort_word,
                                       p.status, STATUS_MMA_WAIT, limit);
                        if (!ok) continue;
                        tc_fence_after();
                        issue_PV(t, s, j > 0);
                        if (j + 1 < nkv[t]) {
                            const int s1 = (j + 1) % L::STAGES;
                            if (!knext) {
                                ok = mbar_wait(bar(L::B_KFULL + s1),
                                               static_cast<uint32_t>((j + 1) / L::STAGES) & 1u,
                                               abort_word, p.status, STATUS_MMA_WAIT, limit);
                                if (!ok) continue;
                                tc_fence_after();
                                knext = true;
                            }
                            issue_S(t, s1);
                            mma_commit(bar(L::B_SFULL + t));
                        } else {
                            mma_commit(bar(L::B_OFULL + t));
                        }
                    }
                    if (ok) mma_commit(bar(L::B_KVEMPTY + s));
                }
                // nothing may be in flight when TMEM is released
                mma_commit(bar(L::B_DRAIN));
                drain_wait(bar(L::B_DRAIN), 0, 100000000ull);
            }
        }
        __syncwarp();
    } else {
        // ================================================== softmax + epilogue
        regs_inc<L::REG_SOFTMAX>();
        const int t = warp / 4;
        const int wq = warp % 4;                       // TMEM lane quadrant
        const int r = 32 * wq + lane;                  // row within the tile
        const int qrow = q0 + t * BM + r;              // query row within the head
        const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;
        const uint32_t tS = tmem + lane_base + t * 128;
        const uint32_t tO = tmem + lane_base + L::O_COL + t * D;
        const float sl2 = p.scale_log2;
        const bool tile_active = q0 + t * BM < p.n;
        int my_nkv = nkv[0];
#pragma unroll
        for (int u = 1; u < NT; ++u)
            if (t == u) my_nkv = nkv[u];

        float m_ref = -INFINITY;   // reference max of scaled scores (log2 units)
        float l_run = 0.f;         // running sum of exp2(x - m_ref)
        bool ok = true;

        if (p.debug_flags & DEBUG_FORCE_TIMEOUT) {
            ok = mbar_wait(bar(L::B_NEVER), 0, abort_word, p.status, STATUS_FORCED, 20000000ull);
            ok = __all_sync(0xffffffffu, ok);
        }

        for (int j = 0; ok && j < my_nkv; ++j) {
            ok = mbar_wait(bar(L::B_SFULL + t), static_cast<uint32_t>(j) & 1u, abort_word, p.status,
                           STATUS_SOFTMAX_WAIT, limit);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();

            uint32_t sr[BN];
            tmem_ld32(tS + 0, sr + 0);
            tmem_ld32(tS + 32, sr + 32);
            tmem_ld32(tS + 64, sr + 64);
            tmem_ld32(tS + 96, sr + 96);
            tmem_wait_ld();
            float s[BN];
#pragma unroll
            for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c]);

            // mask: keys past the valid length, and keys after the query row (causal)
            const int key0 = j * BN;
            const bool need_mask =
                (key0 + BN > kv_len) || (MASK == MASK_CAUSAL && key0 + BN - 1 > qrow);
            if (need_mask) {
#pragma unroll
                for (int c = 0; c < BN; ++c) {
                    const int key = key0 + c;
                    if (key >= kv_len || (MASK == MASK_CAUSAL && key > qrow)) s[c] = -INFINITY;
                }
            }
            // row maximum: eight independent chains
            float mx[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = s[k];
#pragma unroll
            for (int c = 8; c < BN; c += 8)
#pragma unroll
                for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], s[c + k]);
            const float tile_max =
                fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                      fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
            // raise the reference only when the new maximum exceeds it by > 2^8
            const bool raise = tile_max > m_ref + RESCALE_LOG2;
            const float m_new = raise ? tile_max : m_ref;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = raise ? ex2_approx(m_ref - m_use) : 1.f;   // 0 on the first raise

            uint32_t pk[BN / 2];
            float rs[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) rs[k] = 0.f;
#pragma unroll
            for (int c = 0; c < BN / 2; ++c) {
                const float p0 = ex2_approx(fmaf(s[2 * c], sl2, -m_use));
                const float p1 = ex2_approx(fmaf(s[2 * c + 1], sl2, -m_use));
                rs[c % 8] += p0 + p1;
                pk[c] = pack_bf16x2(p0, p1);
            }
            const float tile_sum =
                ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
            l_run = l_run * alpha + tile_sum;

            // earlier partial output of this row: O *= alpha (warp-uniform decision)
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * cc, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tO + 32 * cc, o);
                }
            }
            m_ref = m_new;

            // P (bf16 pairs) over the first 64 columns of this tile's S
            tmem_st32(tS + 0, pk);
            tmem_st32(tS + 32, pk + 32);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(L::B_PFULL + t));
        }

        // ---------------------------------------------- epilogue
        const bool have_o = my_nkv > 0;
        if (ok && have_o) {
            ok = mbar_wait(bar(L::B_OFULL + t), 0, abort_word, p.status, STATUS_SOFTMAX_WAIT, limit);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
        }
        if (ok && tile_active) {
            const bool any = l_run > 0.f;
            const float inv_l = any ? 1.f / l_run : 0.f;
            if (p.LSE != nullptr && qrow < p.n)
                p.LSE[static_cast<int64_t>(bh) * p.n + qrow] =
                    any ? (m_ref + __log2f(l_run)) * LN2 : -INFINITY;

            // stage O (bf16, 128-byte swizzle) in this tile's Q buffer, then TMA-store it.
            // All MMAs reading Q_t have completed (OFULL covers them).
            const uint32_t stage = sQ + t * L::TILE;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                if (have_o) {
                    tmem_ld32(tO + 32 * cc, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                const uint32_t chunk_base = stage + (cc / 2) * CHUNK_BYTES + r * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_bf16x2(__uint_as_float(o[8 * q + 2 * e]) * inv_l,
                                           __uint_as_float(o[8 * q + 2 * e + 1]) * inv_l);
                    const uint32_t piece = static_cast<uint32_t>((cc % 2) * 4 + q);
                    const uint32_t addr = chunk_base + ((piece ^ static_cast<uint32_t>(r & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]),
                                 "r"(w[1]), "r"(w[2]), "r"(w[3])
                                 : "memory");
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && q0 + t * BM + 32 * wq < p.n) {
                for (int c = 0; c < L::CH; ++c)
                    tma_store_3d(&tmO, stage + c * CHUNK_BYTES + wq * 32 * 128, c * 64,
                                 q0 + t * BM + 32 * wq, bh);
                bulk_commit_group();
                bulk_wait_group0();
            }
            __syncwarp();
        }
    }

    // ---- teardown: every role has drained its async work
    tc_fence_before();
    __syncthreads();
    if (warp == L::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

template <int D, int MASK, int NT>
cudaError_t launch_fwd(const TensorMaps& maps, const FwdParams& p, int64_t num_ctas, cudaStream_t stream)
{
    using L = Layout<D, NT>;
    auto kern = attn_fwd_kernel<D, MASK, NT>;
    // The shared-memory opt-in is set once per device, so that a launch inside
    // stream capture issues nothing but the launch itself.
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
    kern<<<static_cast<unsigned>(num_ctas), L::NUM_THREADS, L::BYTES, stream>>>(maps.q, maps.k, maps.v,
                                                                               maps.o, p);
    return cudaGetLastError();
}

}  // namespace attn
