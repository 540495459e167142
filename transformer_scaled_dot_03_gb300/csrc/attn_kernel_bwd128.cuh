// attn_kernel_bwd128.cuh -- sm_103a attention backward at d_k = d_v = 128:
// persistent CTAs over 128-key tiles, 64-query steps, the scores of step g + 1
// computed by the tensor cores while the compute warps work on step g.
//
// Computes the same gradients as attn_kernel_bwd.cuh ("Transformer 详解"
// §4.1-§4.2 with the masks of §3.4 and §5.3; P recomputed from the saved LSE):
//   dV = Pᵀ dO,  dS = P ∘ (dP - D),  dK = scale * dSᵀ Q,  dQ = scale * dS K.
// At d = 128 the accumulators dV and dK take 256 of the 512 tensor-memory
// columns. The other 256 hold two step buffers of 128 columns, so that one step's
// Sᵀ = K Qᵀ and dPᵀ = V dOᵀ (64 queries each) can be computed while the previous
// step's are still in use. Within a buffer, Pᵀ (bf16) is written over Sᵀ once it
// has been read, and the step's dQ is computed transposed,
// dQᵀ = Kᵀ dSᵀ (128 head dims x 64 queries), into the columns of dPᵀ, which the
// compute warps have read before they write Pᵀ. dS goes to shared memory (row =
// key, the step's 64 queries contiguous), where it is the K-major A operand of
// dK += dSᵀ Q and the MN-major B operand of dQᵀ.
//
// Two warps issue the MMAs: one every step's scores, the other every step's
// products (dQᵀ first, so that its read-out overlaps dV and dK and the buffer frees
// early, then dV, then dK). The scores of step g + 2 go to step g's buffer once step
// g's dQᵀ and dV are complete and its dQᵀ has been read out.
//
//   warps 0-7   thread = key: Pᵀ = exp2(Sᵀ·c - LSE₂), dS = Pᵀ ∘ (dPᵀ - D) for the
//               step's 64 queries, warp w taking tensor-memory lanes 32(w % 4)..
//               and queries 32(w / 4)..
//   warps 8-11  thread = head dim: each step's dQᵀ as soon as its products are
//               done -> staging -> TMA reduce-add into the fp32 dQ accumulator,
//               which frees the step buffer for the step after next; thread = key
//               for the item's dV and dK (read out, scaled, stored)
//   warp  12    TMA producer: K and V per item, Q, dO, LSE, D per step (3 slots)
//   warp  13    tcgen05.mma issuer of the scores, owns the tensor-memory allocation
//   warp  14    tcgen05.mma issuer of the products
//   warp  15    idle
// Tensor memory: buffer b (b = step % 2) at columns [128b, 128b + 128): Sᵀ in
// [128b, 128b + 64), each query half's Pᵀ (16 columns) over the first 16 of its own
// 32 Sᵀ columns (so no warp writes columns another warp may still be reading);
// dPᵀ then dQᵀ in [128b + 64, 128b + 128); dV [256, 384), dK [384, 512).
#pragma once

#include <climits>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "attn_kernel_bwd.cuh"
#include "sm103a.cuh"

namespace attn {

using namespace sm103a;

namespace bwd128 {

constexpr int D = 128;
constexpr int BK = 128;                    // keys per item
constexpr int BQ = 64;                     // queries per step
constexpr int KV_CHUNK = 128 * 64 * 2;     // 128 rows x 64 bf16 (128-byte rows, 128-byte swizzle)
constexpr int Q_CHUNK = BQ * 64 * 2;       // 64 rows x 64 bf16
constexpr int DQ_BLOCK = 32 * 32 * 4;      // 32 queries x 32 head dims fp32
constexpr uint32_t kWaitHintNs = 2000;     // suspend bound of the compute and read-out warps' waits

struct Layout {
    static constexpr int NUM_THREADS = 512;
    static constexpr int COMPUTE_THREADS = 256;
    static constexpr int DQ_THREADS = 128;            // warps 8-11
    static constexpr int WARP_DQ = 8;
    static constexpr int WARP_TMA = 12;
    static constexpr int WARP_MMA = 13;               // issues the scores, owns the tensor memory
    static constexpr int WARP_MMA_B = 14;             // issues the products
    static constexpr int QS = 3;                      // Q/dO/LSE/D ring depth
    static constexpr int TILE_KV = 2 * KV_CHUNK;      // a 128 x 128 K or V tile
    static constexpr int TILE_Q = 2 * Q_CHUNK;        // a 64 x 128 Q or dO tile
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + TILE_KV;
    static constexpr int Q_OFF = V_OFF + TILE_KV;
    static constexpr int DO_OFF = Q_OFF + QS * TILE_Q;
    static constexpr int DS_OFF = DO_OFF + QS * TILE_Q;     // dS bf16: 128 keys x 64 queries
    static constexpr int DQ_OFF = DS_OFF + KV_CHUNK;        // dQᵀ staging: 32 x 32 blocks, two per read-out warp
    static constexpr int LSE_OFF = DQ_OFF + 8 * DQ_BLOCK;
    static constexpr int DD_OFF = LSE_OFF + QS * BQ * 4;
    static constexpr int BAR_OFF = DD_OFF + QS * BQ * 4;
    static constexpr int B_KVFULL = 0;
    static constexpr int B_KVEMPTY = 1;
    static constexpr int B_QFULL = 2;
    static constexpr int B_QEMPTY = B_QFULL + QS;
    static constexpr int B_SFULL = B_QEMPTY + QS;   // [2] Sᵀ, dPᵀ of a step in buffer b       (commit)
    static constexpr int B_PFULL = B_SFULL + 2;     // Pᵀ and dS of a step written              (256 arrivals)
    static constexpr int B_DQDONE = B_PFULL + 1;    // [2] dQᵀ of a step in buffer b done       (commit)
    static constexpr int B_BDONE = B_DQDONE + 2;    // [2] all products of a step in buffer b   (commit)
    static constexpr int B_PUSED = B_BDONE + 2;     // [2] Pᵀ of buffer b consumed (dQᵀ, dV)    (commit)
    static constexpr int B_DQFREE = B_PUSED + 2;    // [2] dQᵀ of buffer b read out             (128 arrivals)
    static constexpr int B_DKVDONE = B_DQFREE + 2;  // an item's dV, dK complete                (commit)
    static constexpr int B_DKVFREE = B_DKVDONE + 1; // an item's dV, dK read out                (128 arrivals)
    static constexpr int B_DRAIN = B_DKVFREE + 1;   // [2] each issuing warp's last MMAs done
    static constexpr int B_NEVER = B_DRAIN + 2;
    static constexpr int NBARS = B_NEVER + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BYTES = MISC_OFF + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t DV_COL = 256, DK_COL = 384;
    static_assert(DS_OFF % 1024 == 0 && DQ_OFF % 1024 == 0 && Q_OFF % 1024 == 0 && DO_OFF % 1024 == 0,
                  "swizzled tiles start on 1024-byte boundaries");
    static_assert(BYTES <= 232448, "shared memory budget");
};

// One work item: a 128-key tile of one (b, h) pair and the 64-query steps that see it.
struct Item {
    int bh, k0, kv_len, s_lo, ns;   // steps s_lo .. s_lo + ns - 1; ns = 0: no query sees these keys
    int off;                        // query row i sits at key position i + off
};

template <int MASK>
__device__ __forceinline__ Item item_of(int u, int iu, const BwdParams& p)
{
    const int uph = bwd::bwd_units_per_head<MASK>(p);
    Item w;
    w.bh = u / uph;
    const int k = u % uph;
    const int kb = (mask_is_causal(MASK) && iu == 1) ? p.num_kblocks - 1 - k : k;
    w.k0 = kb * BK;
    w.kv_len = p.m;
    if (mask_has_lengths(MASK)) {
        const int len = __ldg(p.key_lengths + w.bh / p.H);
        w.kv_len = len < 0 ? 0 : (len > p.m ? p.m : len);
    }
    w.off = causal_offset(MASK, p.causal_off, w.kv_len, p.n);
    w.s_lo = 0;
    if (mask_is_causal(MASK)) {
        const int first_q = w.k0 - w.off;            // first row that sees key k0
        w.s_lo = first_q <= 0 ? 0 : first_q / BQ;
    }
    const int nsteps = (p.n + BQ - 1) / BQ;
    w.ns = (w.k0 >= w.kv_len || w.s_lo >= nsteps) ? 0 : nsteps - w.s_lo;
    return w;
}

// Walks the steps of this CTA's items in order, skipping items without queries.
template <int MASK>
struct Cursor {
    int u, iu, t;
    int item;   // items with steps entered so far, minus one: this step's item number
    Item w;
    bool valid;
    __device__ void settle(const BwdParams& p, int num_units)
    {
        while (u < num_units) {
            w = item_of<MASK>(u, iu, p);
            if (t < w.ns) {
                valid = true;
                return;
            }
            t = 0;
            if (++iu >= bwd::bwd_items_of_unit<MASK>(u, p)) {
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
        item = 0;
        settle(p, num_units);
    }
    __device__ void next(const BwdParams& p, int num_units)
    {
        if (++t < w.ns) return;   // the same item: nothing to recompute
        settle(p, num_units);
        if (valid && t == 0) ++item;
    }
};

template <int MASK, bool BIAS>
__global__ void __launch_bounds__(Layout::NUM_THREADS, 1)
attn_bwd_pipe128_kernel(const __grid_constant__ BwdMaps maps, const BwdParams p)
{
    using L = Layout;
    const int num_units = p.B * p.H * bwd::bwd_units_per_head<MASK>(p);

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
        mbar_init(bar(L::B_KVEMPTY), 1);
        for (int s = 0; s < L::QS; ++s) {
            mbar_init(bar(L::B_QFULL + s), 1);
            mbar_init(bar(L::B_QEMPTY + s), 1);
        }
        mbar_init(bar(L::B_SFULL), 1);
        mbar_init(bar(L::B_SFULL + 1), 1);
        mbar_init(bar(L::B_PFULL), L::COMPUTE_THREADS);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::B_DQDONE + b), 1);
            mbar_init(bar(L::B_BDONE + b), 1);
            mbar_init(bar(L::B_PUSED + b), 1);
            mbar_init(bar(L::B_DQFREE + b), L::DQ_THREADS);
            mbar_init(bar(L::B_DRAIN + b), 1);
        }
        mbar_init(bar(L::B_DKVDONE), 1);
        mbar_init(bar(L::B_DKVFREE), L::DQ_THREADS);
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
        if (warp == L::WARP_TMA && lane == 0) {
            // ================================================== TMA producer
            Cursor<MASK> cur;
            cur.start(p, num_units);
            int gt = 0, it = 0;          // steps and items so far
            int kv_issued = 0;           // K/V loads issued
            bool ok = true;
            while (ok && cur.valid) {
                if (cur.t == 0) {
                    // the previous item's last products must have read K and V
                    if (it > 0 && !mbar_wait(bar(L::B_KVEMPTY), static_cast<uint32_t>(it - 1) & 1u, abort_word,
                                             p.status, STATUS_TMA_WAIT, limit)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(L::B_KVFULL), 2 * L::TILE_KV);
                    for (int c = 0; c < 2; ++c) {
                        tma_load_3d(sK + c * KV_CHUNK, &maps.k, bar(L::B_KVFULL), c * 64, cur.w.k0, cur.w.bh);
                        tma_load_3d(sV + c * KV_CHUNK, &maps.v, bar(L::B_KVFULL), c * 64, cur.w.k0, cur.w.bh);
                    }
                    ++kv_issued;
                }
                const int s = gt % L::QS;
                if (gt >= L::QS &&
                    !mbar_wait(bar(L::B_QEMPTY + s), static_cast<uint32_t>(gt / L::QS - 1) & 1u, abort_word,
                               p.status, STATUS_TMA_WAIT, limit)) {
                    ok = false;
                    break;
                }
                const int q0 = (cur.w.s_lo + cur.t) * BQ;
                mbar_arrive_expect_tx(bar(L::B_QFULL + s), 2 * L::TILE_Q + 2 * BQ * 4);
                for (int c = 0; c < 2; ++c) {
                    tma_load_3d(sQ + s * L::TILE_Q + c * Q_CHUNK, &maps.q, bar(L::B_QFULL + s), c * 64, q0, cur.w.bh);
                    tma_load_3d(sdO + s * L::TILE_Q + c * Q_CHUNK, &maps.dout, bar(L::B_QFULL + s), c * 64, q0,
                                cur.w.bh);
                }
                const int64_t row0 = static_cast<int64_t>(cur.w.bh) * p.n_pad + q0;
                bulk_load(sbase + L::LSE_OFF + s * BQ * 4, p.lse2 + row0, BQ * 4, bar(L::B_QFULL + s));
                bulk_load(sbase + L::DD_OFF + s * BQ * 4, p.dd + row0, BQ * 4, bar(L::B_QFULL + s));
                if (cur.t == cur.w.ns - 1) ++it;
                ++gt;
                cur.next(p, num_units);
            }
            // land every copy still in flight (only possible after an abort)
            if (kv_issued > 0) bwd::drain(bar(L::B_KVFULL), static_cast<uint32_t>(kv_issued - 1) & 1u, 100000000ull);
            for (int i = gt - 1; i >= 0 && i >= gt - L::QS; --i)
                bwd::drain(bar(L::B_QFULL + i % L::QS), static_cast<uint32_t>(i / L::QS) & 1u, 100000000ull);
        } else if (warp == L::WARP_MMA || warp == L::WARP_MMA_B) {
            // ================================================== MMA issuers (whole warp, one elected lane)
            // Warp 13 issues every step's scores, warp 14 every step's products, so
            // that one warp's bookkeeping and waits overlap the other's issue. Issue
            // order between the two is not an order on the tensor pipe: step h's
            // scores go to the buffer of step h - 2 only once that step's dQᵀ and dV
            // (the products that use the buffer) are complete (B_PUSED) and its dQᵀ
            // has been read out (B_DQFREE).
            constexpr uint32_t ID_S = idesc_bf16_f32(BK, BQ, false, false);   // M = keys, N = queries
            constexpr uint32_t ID_KV = idesc_bf16_f32(BK, D, false, true);    // M = keys, N = head dims
            constexpr uint32_t ID_DQ = idesc_bf16_f32(D, BQ, true, true);     // M = head dims, N = queries
            const uint64_t dK_k = sdesc_sw128(sK, 16, 1024);
            const uint64_t dV_k = sdesc_sw128(sV, 16, 1024);
            const uint64_t dK_mn = sdesc_sw128(sK, KV_CHUNK, 1024);
            const uint64_t dS_k = sdesc_sw128(sdS, 16, 1024);
            const uint64_t dS_mn = sdesc_sw128(sdS, KV_CHUNK, 1024);
            // (a phase that has already completed is seen by a non-blocking probe,
            // which returns sooner than a potentially suspending one)
            auto wait = [&](int b, uint32_t parity) -> bool {
                if (__all_sync(0xffffffffu, mbar_test_now(bar(b), parity))) return true;
                const bool r = mbar_wait(bar(b), parity, abort_word, p.status, STATUS_MMA_WAIT, limit);
                return __all_sync(0xffffffffu, r);
            };
            Cursor<MASK> cur;
            cur.start(p, num_units);
            bool ok = true;
            int g = 0;      // step
            int s = 0;      // its Q slot
            if (warp == L::WARP_MMA) {
                while (ok && cur.valid) {
                    const int b = g & 1;
                    const uint32_t rp = static_cast<uint32_t>((g - 2) >> 1) & 1u;   // step g - 2's phase
                    ok = (g < 2 || (wait(L::B_PUSED + b, rp) && wait(L::B_DQFREE + b, rp))) &&
                         // an item's keys (loaded once the previous item's products are done)
                         (cur.t != 0 || wait(L::B_KVFULL, static_cast<uint32_t>(cur.item) & 1u)) &&
                         wait(L::B_QFULL + s, static_cast<uint32_t>(g / L::QS) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    // Sᵀ = K Qᵀ and dPᵀ = V dOᵀ into buffer b, the two chains interleaved
                    const uint64_t dQ_k = sdesc_sw128(sQ + s * L::TILE_Q, 16, 1024);
                    const uint64_t dO_k = sdesc_sw128(sdO + s * L::TILE_Q, 16, 1024);
                    const uint32_t col = tmem + 128u * static_cast<uint32_t>(b);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t aoff = static_cast<uint64_t>(((kk / 4) * KV_CHUNK + (kk % 4) * 32) >> 4);
                        const uint64_t boff = static_cast<uint64_t>(((kk / 4) * Q_CHUNK + (kk % 4) * 32) >> 4);
                        mma_ss_warp(col, dK_k + aoff, dQ_k + boff, ID_S, kk > 0 ? 1u : 0u);
                        mma_ss_warp(col + 64, dV_k + aoff, dO_k + boff, ID_S, kk > 0 ? 1u : 0u);
                    }
                    mma_commit_warp(bar(L::B_SFULL + b));
                    ++g;
                    s = s == L::QS - 1 ? 0 : s + 1;
                    cur.next(p, num_units);
                }
            } else {
                while (ok && cur.valid) {
                    const int b = g & 1;
                    const uint32_t bcol = tmem + 128u * static_cast<uint32_t>(b);
                    const bool last = cur.t == cur.w.ns - 1;
                    const int item = cur.item;
                    const uint32_t acc0 = cur.t > 0 ? 1u : 0u;
                    const uint64_t dO_mn = sdesc_sw128(sdO + s * L::TILE_Q, Q_CHUNK, 1024);
                    const uint64_t dQ_mn = sdesc_sw128(sQ + s * L::TILE_Q, Q_CHUNK, 1024);
                    ok = wait(L::B_PFULL, static_cast<uint32_t>(g) & 1u);
                    // this item's first dV, dK overwrite the accumulators of the previous item
                    if (ok && cur.t == 0 && item > 0) ok = wait(L::B_DKVFREE, static_cast<uint32_t>(item - 1) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    // dQᵀ = Kᵀ dSᵀ into the dPᵀ columns (read by now), first, so that its
                    // read-out overlaps dV and dK
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t off = static_cast<uint64_t>((kk * 2048) >> 4);
                        mma_ss_warp(bcol + 64, dK_mn + off, dS_mn + off, ID_DQ, kk > 0 ? 1u : 0u);
                    }
                    mma_commit_warp(bar(L::B_DQDONE + b));
                    // dV += Pᵀ dO, the last product that uses the step's buffer
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk) {
                        const uint64_t off = static_cast<uint64_t>((kk * 2048) >> 4);
                        // Pᵀ of queries 16kk.. : the query half kk / 2, its (kk % 2)-th 8 columns
                        mma_ts_warp(tmem + L::DV_COL, bcol + (kk >> 1) * 32 + (kk & 1) * 8, dO_mn + off, ID_KV,
                                    (acc0 | kk) ? 1u : 0u);
                    }
                    mma_commit_warp(bar(L::B_PUSED + b));
                    // dK += dSᵀ Q (shared memory only)
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk) {
                        const uint64_t off = static_cast<uint64_t>((kk * 2048) >> 4);
                        mma_ss_warp(tmem + L::DK_COL, dS_k + static_cast<uint64_t>((kk * 32) >> 4), dQ_mn + off,
                                    ID_KV, (acc0 | kk) ? 1u : 0u);
                    }
                    // the last reads of this step's Q and dO are issued
                    mma_commit_warp(bar(L::B_QEMPTY + s));
                    if (last) mma_commit_warp(bar(L::B_DKVDONE));
                    mma_commit_warp(bar(L::B_BDONE + b));
                    // an item's keys are read for the last time by its last products
                    // (its last scores are complete: their P came before)
                    if (last) mma_commit_warp(bar(L::B_KVEMPTY));
                    ++g;
                    s = s == L::QS - 1 ? 0 : s + 1;
                    cur.next(p, num_units);
                }
            }
            const int dr = warp == L::WARP_MMA ? 0 : 1;
            mma_commit_warp(bar(L::B_DRAIN + dr));
            bwd::drain(bar(L::B_DRAIN + dr), 0, 100000000ull);
        }
        __syncwarp();
    } else if (warp >= L::WARP_DQ) {
        // ================================================== dQᵀ read-out, dV / dK epilogue
        const int wq = warp % 4;                      // lane quadrant
        const int r = 32 * wq + lane;                 // TMEM lane: a head dim for dQᵀ, a key for dV, dK
        const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;
        bool ok = true;
        bool bulk_pending = false;   // this warp has committed reduce-adds
        int gt = 0, it = 0;
        const uint32_t chunk = static_cast<uint32_t>(lane >> 2);
        const uint32_t word = static_cast<uint32_t>(lane & 3) << 2;
        for (int u = static_cast<int>(blockIdx.x); ok && u < num_units; u += static_cast<int>(gridDim.x)) {
            const int n_items = bwd::bwd_items_of_unit<MASK>(u, p);
            for (int iu = 0; ok && iu < n_items; ++iu) {
                const Item w = item_of<MASK>(u, iu, p);
                if (w.ns == 0) {
                    // no query sees these keys: their gradients are zero
                    if (w.k0 < p.m) {
                        const int rows = min(BK, p.m - w.k0);
                        const int64_t base = (static_cast<int64_t>(w.bh) * p.m + w.k0) * D;
                        uint4* gk = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dK) + base);
                        uint4* gv = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dV) + base);
                        for (int i = r; i < rows * D / 8; i += L::DQ_THREADS) {
                            gk[i] = make_uint4(0u, 0u, 0u, 0u);
                            gv[i] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    continue;
                }
                for (int t = 0; ok && t < w.ns; ++t) {
                    const int q0 = (w.s_lo + t) * BQ;
                    ok = mbar_wait_suspend(bar(L::B_DQDONE + (gt & 1)), static_cast<uint32_t>(gt >> 1) & 1u, abort_word, p.status,
                                   STATUS_SOFTMAX_WAIT, limit, kWaitHintNs);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    // this warp's 32 head dims x the step's 64 queries
                    uint32_t a[64];
                    const uint32_t col = 128u * static_cast<uint32_t>(gt & 1) + 64u;
                    tmem_ld32(tmem + lane_base + col, a);
                    tmem_ld32(tmem + lane_base + col + 32, a + 32);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(bar(L::B_DQFREE + (gt & 1)));
                    // the reduce-adds of the previous step must have read the staging blocks
                    if (bulk_pending && lane == 0) bulk_wait_group_read0();
                    __syncwarp();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t block = sdQ + static_cast<uint32_t>(h * 4 + wq) * DQ_BLOCK;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            // row = query 32h + i, 128-byte swizzle of the fp32 box
                            const uint32_t addr = block + i * 128 + ((chunk ^ static_cast<uint32_t>(i & 7)) << 4) + word;
                            asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(a[32 * h + i]) : "memory");
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        for (int h = 0; h < 2; ++h) {
                            if (q0 + 32 * h >= p.n) break;
                            bwd::dq_reduce_add(&maps.dq_acc, sdQ + static_cast<uint32_t>(h * 4 + wq) * DQ_BLOCK, 32 * wq,
                                               q0 + 32 * h, w.bh);
                        }
                        bulk_commit_group();
                        bulk_pending = true;
                    }
                    __syncwarp();
                    ++gt;
                }
                if (!ok) break;

                // ---------------------------------------- this item's dV and dK (x scale)
                // Each thread reads its key's 128 columns of dV, then of dK, 32 at a time,
                // and stores each piece (64 bytes) straight to global memory; the last
                // read releases the accumulators to the next item.
                ok = mbar_wait_suspend(bar(L::B_DKVDONE), static_cast<uint32_t>(it) & 1u, abort_word, p.status,
                               STATUS_SOFTMAX_WAIT, limit, kWaitHintNs);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const int key = w.k0 + r;
#pragma unroll 1
                for (int g2 = 0; g2 < 8; ++g2) {
                    const bool dk = g2 >= 4;
                    const int c = g2 % 4;
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_base + (dk ? L::DK_COL : L::DV_COL) + 32 * c, o);
                    tmem_wait_ld();
                    if (g2 == 7) {
                        tc_fence_before();
                        mbar_arrive(bar(L::B_DKVFREE));
                    }
                    if (key < p.m) {
                        const float mul = dk ? p.scale : 1.f;
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dk ? p.dK : p.dV) +
                                                              (static_cast<int64_t>(w.bh) * p.m + key) * D + 32 * c);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * mul, __uint_as_float(o[8 * q + 1]) * mul);
                            v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * mul, __uint_as_float(o[8 * q + 3]) * mul);
                            v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * mul, __uint_as_float(o[8 * q + 5]) * mul);
                            v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * mul, __uint_as_float(o[8 * q + 7]) * mul);
                            dst[q] = v;
                        }
                    }
                }
                ++it;
            }
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    } else {
        // ================================================== Pᵀ / dS
        const int wq = warp % 4;                      // lane quadrant
        const int half = warp / 4;                    // query half of a step
        const int r = 32 * wq + lane;                 // TMEM lane: a key
        const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;
        const float sl2 = p.scale_log2;
        bool ok = true;
        int gt = 0;

        if (p.debug_flags & DEBUG_FORCE_TIMEOUT) {
            ok = mbar_wait(bar(L::B_NEVER), 0, abort_word, p.status, STATUS_FORCED, 20000000ull);
            ok = __all_sync(0xffffffffu, ok);
        }
        for (int u = static_cast<int>(blockIdx.x); ok && u < num_units; u += static_cast<int>(gridDim.x)) {
            const int n_items = bwd::bwd_items_of_unit<MASK>(u, p);
            for (int iu = 0; ok && iu < n_items; ++iu) {
                const Item w = item_of<MASK>(u, iu, p);
                const int key = w.k0 + r;
                const float sb = BIAS ? __ldg(p.slopes + w.bh % p.H) * 1.44269504088896341f : 0.f;   // log2 domain
                for (int t = 0; ok && t < w.ns; ++t) {
                    const int s = gt % L::QS;
                    const int b = gt & 1;
                    const int q0 = (w.s_lo + t) * BQ;
                    ok = mbar_wait_suspend(bar(L::B_QFULL + s), static_cast<uint32_t>(gt / L::QS) & 1u, abort_word, p.status,
                                   STATUS_SOFTMAX_WAIT, limit, kWaitHintNs) &&
                         mbar_wait_suspend(bar(L::B_SFULL + b), static_cast<uint32_t>(gt >> 1) & 1u, abort_word, p.status,
                                   STATUS_SOFTMAX_WAIT, limit, kWaitHintNs);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    const int c0 = 32 * half;         // this warp's first query column of the step
                    const uint32_t bcol = 128u * static_cast<uint32_t>(b);
                    uint32_t sr[32], dr[32];
                    tmem_ld32(tmem + lane_base + bcol + c0, sr);
                    tmem_wait_ld();
                    const uint32_t lse_s = sbase + L::LSE_OFF + (s * BQ + c0) * 4;
                    const uint32_t dd_s = sbase + L::DD_OFF + (s * BQ + c0) * 4;
                    const float d1 = static_cast<float>(q0 + c0 + w.off - key);
                    const bool need_mask =
                        __any_sync(0xffffffffu, key >= w.kv_len || q0 + c0 + 31 >= p.n ||
                                                    (mask_is_causal(MASK) && key > q0 + c0 + w.off));
                    {
                        float lz[32];
#pragma unroll
                        for (int v = 0; v < 8; ++v) lds_v4f(lse_s + 16 * v, lz + 4 * v);
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            // with the distance bias −sb |i' − key| of query column j under BIAS
                            const float z = BIAS ? fmaf(-sb, fabsf(d1 + static_cast<float>(j)), -lz[j]) : -lz[j];
                            sr[j] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(sr[j]), sl2, z)));
                        }
                    }
                    if (need_mask) {
                        const int q_first =
                            key >= w.kv_len ? INT_MAX : (mask_is_causal(MASK) ? key - w.off : 0);
                        const int j_lo = q_first == INT_MAX ? BQ : max(q_first - q0, 0) - c0;
                        const int j_hi = min(p.n - q0, BQ) - c0;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < j_lo || j >= j_hi) sr[j] = 0u;
                    }
                    tmem_ld32(tmem + lane_base + bcol + 64 + c0, dr);
                    tmem_wait_ld();
                    {
                        float dz[32];
#pragma unroll
                        for (int v = 0; v < 8; ++v) lds_v4f(dd_s + 16 * v, dz + 4 * v);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            dr[j] = __float_as_uint(__uint_as_float(sr[j]) * (__uint_as_float(dr[j]) - dz[j]));
                    }
                    // the previous step's dQᵀ, dV and dK have read dS (B_BDONE follows them)
                    if (gt > 0) {
                        ok = mbar_wait_suspend(bar(L::B_BDONE + ((gt - 1) & 1)), static_cast<uint32_t>((gt - 1) >> 1) & 1u, abort_word, p.status,
                                       STATUS_SOFTMAX_WAIT, limit, kWaitHintNs);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16x2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]));
                        tmem_st16(tmem + lane_base + bcol + c0, pk);   // over this warp's own Sᵀ columns
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16x2(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1]));
                        const uint32_t row_base = sdS + r * 128;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t piece = static_cast<uint32_t>(4 * half + q);
                            const uint32_t addr = row_base + ((piece ^ static_cast<uint32_t>(r & 7)) << 4);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * q]),
                                         "r"(pk[4 * q + 1]), "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                                         : "memory");
                        }
                    }
                    tmem_wait_st();
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(L::B_PFULL));
                    ++gt;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == L::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

template <int MASK, bool BIAS = false>
cudaError_t launch(const BwdMaps& maps, const BwdParams& p, cudaStream_t stream)
{
    using L = Layout;
    auto kern = attn_bwd_pipe128_kernel<MASK, BIAS>;
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
    // persistent: one CTA per SM over units of one or two key tiles
    const int64_t units = static_cast<int64_t>(p.B) * p.H *
                          (mask_is_causal(MASK) ? (p.num_kblocks + 1) / 2 : p.num_kblocks);
    const int64_t grid = units < p.num_sms ? units : p.num_sms;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(L::NUM_THREADS), L::BYTES, stream, maps, p);
}

}  // namespace bwd128
}  // namespace attn
