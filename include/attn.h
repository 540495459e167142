/*
 * attn.h -- C ABI of the GB300 (sm_103a) multi-head scaled dot-product
 * attention forward pass.
 *
 * Operation ("Transformer 详解" §4.1-§4.2 and §5.3-§5.4; "从 RNN 到 Transformer
 * （二）" §4.9; "第2章：完整的 Transformer 架构" §2.2, §6, §7): for every batch
 * entry b, head h and query row i, independently per head,
 *
 *     O[b,h,i,:] = sum_j softmax_j( scale * q_i . k_j + M_bij ) v_j
 *     LSE[b,h,i] = ln sum_{j : M_bij = 0} exp( scale * q_i . k_j )
 *
 * where M_bij is 0 for a visible key and -inf for a masked one:
 *     ATTN_MASK_NONE         every key is visible (encoder self-attention,
 *                            cross-attention without padding);
 *     ATTN_MASK_CAUSAL       key j is visible to query i iff j <= i + (m - n)
 *                            (decoder self-attention, "Transformer 详解" §5.3,
 *                            which prints the square case n = m; for n != m
 *                            the n queries are the last n of the m positions,
 *                            as when new queries attend to a cache of m keys,
 *                            so with n > m the first n - m rows see no key);
 *     ATTN_MASK_KEY_PADDING  key j is visible iff j < key_lengths[b], for all
 *                            query rows (the [batch,1,1,seq] pad mask of
 *                            "Transformer 详解" §3.4 for tail-padded batches);
 *     ATTN_MASK_CAUSAL_KEY_PADDING
 *                            both conditions at once (the decoder target mask
 *                            of "Transformer 详解" §5.3: pad mask AND
 *                            subsequent mask).
 *     ATTN_MASK_CAUSAL_CACHE causal inside a partly filled key/value cache: m
 *                            slots of which key_lengths[b] are filled, the n
 *                            queries being the last n filled positions, so key
 *                            j is visible to query i iff j < key_lengths[b] and
 *                            j <= i + (key_lengths[b] - n) (the cache of fixed
 *                            size with batched entries of the transformer wiki
 *                            page's KV cache section; with key_lengths[b] = m
 *                            it is ATTN_MASK_CAUSAL).
 * A row that sees no key gets O = 0 and LSE = -inf.
 * The n x m score matrix is never written to memory. LSE is the per-row
 * natural-log normaliser (not printed on the pages; a standard by-product
 * needed to merge or differentiate attention).
 *
 * Conventions common to every entry point:
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     owned by the caller. The library neither frees nor retains them.
 *   - Layouts are contiguous row-major: Q [B,H,n,d_k], K [B,H,m,d_k],
 *     V [B,H,m,d_v], O [B,H,n,d_v] in bf16 (IEEE bfloat16, 2 bytes); LSE
 *     [B,H,n] fp32; key_lengths int32 [B].
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronise the host. The return value is the
 *     enqueue status. Faults inside a kernel surface later from the CUDA
 *     runtime; a device-side watchdog expiry is reported by
 *     attn_get_device_status().
 *   - Memory: the library allocates one 4-byte device status word per device
 *     on the first call on that device and nothing else. The exception is
 *     attn_fwd_noalloc, which allocates nothing (its status word sits in a
 *     fixed array inside the library; see its comment).
 *   - Thread safety: concurrent calls on distinct streams are safe. The status
 *     words are shared by every call on a device, so attn_get_device_status
 *     reports a timeout of any call on the device, whichever stream it ran on.
 */
#ifndef ATTN_SM103A_H
#define ATTN_SM103A_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_MASK_NONE = 0,
    ATTN_MASK_CAUSAL = 1,
    ATTN_MASK_KEY_PADDING = 2,
    ATTN_MASK_CAUSAL_KEY_PADDING = 3,
    ATTN_MASK_CAUSAL_CACHE = 4
} attn_mask_kind_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad mask kind,
                                  a key-padding mask without lengths */
    ATTN_ERR_UNSUPPORTED = -2, /* a head dim outside {64, 128}, n or m above
                                  2^30, or B*H*ceil(n/128) beyond int range */
    ATTN_ERR_MISALIGNED = -3,  /* Q, K, V or O not 16-byte aligned; LSE or
                                  key_lengths not 4-byte aligned */
    ATTN_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed (message in
                                  attn_last_error()) */
    ATTN_ERR_TIMEOUT = -5      /* a device-side bounded wait expired (watchdog) */
} attn_status_t;

/*
 * Attention forward. See the file comment for the operation and layouts.
 *   B, H, n, m   batch, heads, query rows, key/value rows. B, H or n equal to 0
 *                is a no-op; m = 0 writes O = 0 and LSE = -inf.
 *   d_k, d_v     head dims, each 64 or 128 (d_k != d_v allowed).
 *   mask_kind    attn_mask_kind_t.
 *   key_lengths  device int32 [B]; required for KEY_PADDING,
 *                CAUSAL_KEY_PADDING and CAUSAL_CACHE, ignored otherwise.
 *                Values are read on the device and clamped to [0, m]; a length
 *                of 0 gives O = 0 and LSE = -inf for every row of that entry.
 *   scale        multiplies q.k; a value <= 0, NaN or inf selects 1/sqrt(d_k)
 *                ("从 RNN 到 Transformer（二）" §4.4).
 *   O            bf16 output [B,H,n,d_v] (round to nearest even).
 *   LSE          fp32 output [B,H,n], or NULL to skip it.
 *   stream       cudaStream_t to enqueue on.
 * Returns ATTN_OK or a negative attn_status_t; on error nothing is enqueued.
 */
int attn_fwd(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d_k,
             int d_v, int mask_kind, const int32_t* key_lengths, float scale, void* O,
             float* LSE, void* stream);

/*
 * Attention forward with a linear distance bias ("第2章：完整的 Transformer 架构"
 * §5.3, ALiBi): every scaled score gets a bias proportional to the distance
 * between the query and the key, with a slope of its own for each head,
 *
 *     O = softmax(Q Kᵀ * scale - slope_h * D + M) V,   D_ij = |i + (m - n) - j|,
 *
 * i + (m - n) being the query's position among the keys (the n queries are the
 * last n of the m positions, as for the causal mask; |i - j| when n = m). The
 * masks combine with the bias as in attn_fwd, and LSE is the natural log of the
 * masked sum of exp of the biased scaled scores.
 *   slopes       device fp32 [H], caller-owned, 4-byte aligned: the slope of
 *                every head in the units of the scaled scores (natural-log
 *                domain). Any finite values; 0 is no bias.
 *   other arguments as in attn_fwd (d_k, d_v each 64 or 128).
 * Returns ATTN_OK or a negative attn_status_t (INVALID_ARG when slopes is NULL);
 * on error nothing is enqueued. Its decoding
 * form is attn_decode_alibi, its backward attn_bwd_alibi.
 */
int attn_fwd_alibi(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d_k,
                   int d_v, int mask_kind, const int32_t* key_lengths, const float* slopes, float scale,
                   void* O, float* LSE, void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * words: the one attn_fwd and the other entry points use, and the one inside
 * the array of attn_fwd_noalloc. Returns ATTN_ERR_TIMEOUT if any kernel since
 * the last call gave up on a bounded wait (its outputs are then undefined),
 * ATTN_ERR_CUDA if the synchronisation or the read failed, else ATTN_OK. It
 * allocates no device memory (a word that no call has created yet reads as
 * zero). Kernels still running on other streams may set a bit after the read;
 * synchronise them first for a complete report.
 */
int attn_get_device_status(void* stream);

/*
 * The raw status bits (which kind of wait gave up) that the calling thread's
 * last attn_get_device_status read; 0 if it reported ATTN_OK.
 */
uint32_t attn_last_status_detail(void);

/*
 * Watchdog settings for subsequent calls from any thread: `limit_ns` is the
 * wall-clock limit of one device-side wait (0 restores the default, 2 s).
 * `debug_flags` bit 0 makes the warps that consume each kernel's results (the
 * softmax warps of the forward, the compute warps of the backward, the consumer
 * warps of the few-row decode kernel, the epilogue warps of the projections) wait
 * on a barrier that nothing completes, with a 20 ms limit, so that tests can
 * exercise the timeout path without a fault. Not meant to be changed while other threads launch.
 */
void attn_set_watchdog(uint64_t limit_ns, uint32_t debug_flags);

/*
 * attn_fwd without device memory allocation. The pages have no counterpart to
 * this entry point. It is for callers that may not call cudaMalloc: code that
 * runs while another component owns every device allocation (a pooled or
 * caching allocator with a fixed budget), or code that must not add device
 * allocations once it is running.
 *
 * Arguments, layouts, results and status codes are those of attn_fwd. The only
 * difference is where the kernel's scratch memory lives. attn_fwd allocates
 * its 4-byte device status word on its first call on a device; this entry
 * point uses the first word of a fixed 256-byte device array inside the
 * library instead (every GPU that loads the library holds the array until the
 * process exits). One call needs those 4 bytes whatever the problem sizes, so
 * no size is refused for want of scratch. No call allocates or frees device
 * memory, and neither does attn_get_device_status.
 *
 *   - The first call on each device looks up the array's device address with
 *     cudaGetSymbolAddress on that device. Make that first call before any
 *     stream capture on the device.
 *   - All calls share the array. The kernel only sets bits in the status word
 *     and never reads it, so the word needs no reset between calls: it is zero
 *     when the library loads, and attn_get_device_status reads and clears it
 *     together with attn_fwd's word. Calls that overlap on the GPU (different
 *     streams, no ordering between them) race on this word: a timeout in one
 *     is reported for all of them, and a clear issued while one is running can
 *     drop its bit.
 */
int attn_fwd_noalloc(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d_k,
                     int d_v, int mask_kind, const int32_t* key_lengths, float scale, void* O,
                     float* LSE, void* stream);

/*
 * Attention backward: the gradients of the forward above for an upstream
 * gradient dO. The pages print the forward only; the backward is the chain
 * rule through it (training is the pages' motivation): with P the attention
 * weights (0 where masked),
 *
 *     dV = Pᵀ dO,   dS = P ∘ (dO Vᵀ - D),  D_i = dO_i · O_i,
 *     dQ = scale * dS K,   dK = scale * dSᵀ Q.
 *
 * P is recomputed from Q, K and the forward's LSE; D from the forward's O.
 *   Q, K, V      the forward's inputs (bf16, layouts as in attn_fwd).
 *   O, LSE       the forward's outputs for these inputs (bf16 [B,H,n,d_v],
 *                fp32 [B,H,n]); LSE may not be NULL.
 *   dO           bf16 [B,H,n,d_v], the gradient of the loss with respect to O.
 *   B..scale     as in attn_fwd; d_k, d_v each 64 or 128 (d_k != d_v allowed).
 *   dQ, dK, dV   bf16 outputs [B,H,n,d_k], [B,H,m,d_k], [B,H,m,d_v]. Keys that
 *                no query sees (masked for every row) get exactly 0. n = 0
 *                writes dK = dV = 0; m = 0 writes dQ = 0.
 *   workspace    device scratch owned by the caller, 256-byte aligned, at least
 *                attn_bwd_workspace_size(...) bytes (an fp32 dQ accumulator and
 *                two fp32 per-row vectors); its contents on entry do not
 *                matter. Not needed (may be NULL) when n = 0 or m = 0.
 * Three kernels run on `stream`: a preparation kernel (D, LSE·log2 e, zeroing the
 * accumulator), the main kernel (one CTA per (b, h, 128-key tile)), and the
 * conversion of dQ to bf16. The dQ accumulation order across key tiles is not
 * fixed, so dQ may differ in its last bits between runs; dK and dV do not.
 * Returns ATTN_OK or a negative attn_status_t (ATTN_ERR_INVALID_ARG also for a
 * workspace that is too small); on error nothing is enqueued.
 */
size_t attn_bwd_workspace_size(int B, int H, int n, int m, int d_k, int d_v);

int attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
             const float* LSE, int B, int H, int n, int m, int d_k, int d_v, int mask_kind,
             const int32_t* key_lengths, float scale, void* dQ, void* dK, void* dV,
             void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd for the forward with the linear distance bias (attn_fwd_alibi,
 * "第2章：完整的 Transformer 架构" §5.3): P is recomputed from the biased scores
 * and the biased forward's LSE; the bias depends on neither Q nor K, so the
 * formulas for dQ, dK and dV are those of attn_bwd. `slopes` as in
 * attn_fwd_alibi (device fp32 [H], 4-byte aligned); O and LSE must come from
 * attn_fwd_alibi with the same slopes. Workspace, results and status codes as in
 * attn_bwd; ATTN_ERR_INVALID_ARG when slopes is NULL.
 */
int attn_bwd_alibi(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                   const float* LSE, int B, int H, int n, int m, int d_k, int d_v, int mask_kind,
                   const int32_t* key_lengths, const float* slopes, float scale, void* dQ, void* dK,
                   void* dV, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Attention forward for a few query rows against a long key/value sequence:
 * the decoding step of a model that keeps its keys and values in a cache
 * (each new token's query attends to every cached position). Same operation,
 * masks, layouts and results as attn_fwd (any n <= 8 gives the same O and LSE
 * up to rounding). With few (b, h) pairs for the GPU (B*H below four per CTA
 * slot: 4 x SMs at d = 128, 8 x SMs at d = 64) it streams K and V once with a
 * split over the keys and merges the chunks; with more pairs it runs the
 * tensor-core kernel of attn_fwd, which then streams K and V at the memory
 * system's rate without a merge.
 *   n            query rows per (b, h); 0 is a no-op. Up to 8 rows take the
 *                split kernel described below; more always take the
 *                tensor-core kernel of attn_fwd (no workspace).
 *   d_k, d_v     each 64 or 128 (d_k != d_v allowed).
 *   key_lengths  for the key-padding masks: the valid cache length per batch
 *                entry (as in attn_fwd).
 *   workspace    device scratch for the per-chunk partial results, owned by the
 *                caller, 256-byte aligned, at least
 *                attn_decode_workspace_size(...) bytes. The size covers the
 *                largest chunk count any device may use; it is 0 when the keys of
 *                a (b, h) pair are never split (B*H >= 2048 or m <= 256), and the
 *                pointer may then be NULL. The chunk count itself is chosen per
 *                launch from the device's SM count.
 * Kernels on `stream`: the split kernel, then (if the keys were split) a merge
 * kernel. Returns ATTN_OK or a negative attn_status_t; on error nothing is
 * enqueued.
 */
size_t attn_decode_workspace_size(int B, int H, int n, int m, int d_k, int d_v);

int attn_decode(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d_k,
                int d_v, int mask_kind, const int32_t* key_lengths, float scale, void* O, float* LSE,
                void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode with the linear distance bias of attn_fwd_alibi ("第2章：完整的
 * Transformer 架构" §5.3, ALiBi): score of row i and key j minus
 * slopes[h] * |i + (m - n) - j|, i + (m - n) being the new token's position in
 * the cache. `slopes` is a device fp32 [H] array (4-byte aligned, caller-owned);
 * everything else as in attn_decode, including the workspace (the same size).
 * ATTN_ERR_INVALID_ARG when slopes is NULL.
 */
int attn_decode_alibi(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d_k,
                      int d_v, int mask_kind, const int32_t* key_lengths, const float* slopes, float scale,
                      void* O, float* LSE, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The projections around the attention ("从 RNN 到 Transformer（二）" §4.6,
 * "Transformer 详解" §4.2): Q = W_Q(x).view(B, n, h, d).transpose(1, 2) (and K, V
 * likewise) before it, and Y = W_O(out.transpose(1, 2).reshape(B, n, h d)) after
 * it. Weights are in nn.Linear layout [out_features, in_features] (y = x Wᵀ + b);
 * the bias is optional (NULL: none). bf16 in and out, fp32 accumulation, one
 * persistent tensor-core GEMM whose loads and stores do the head split and merge.
 *
 * attn_proj_heads: X bf16 [B, n, d_model]; W bf16 [num_out*d_model, d_model]
 *   (the weights of num_out projections stacked, e.g. W_Q, W_K, W_V); bias bf16
 *   [num_out*d_model] or NULL; out0..out{num_out-1} bf16 [B, H, n, d_model/H]
 *   receive column blocks 0..num_out-1 split per head. num_out is 1..3 (3: self-
 *   attention's Q, K, V; 1 and 2: cross-attention's Q from the decoder and K, V
 *   from the encoder).
 * attn_merge_proj: O bf16 [B, H, n, d] (an attention output); W_o bf16
 *   [d_out, H*d]; bias bf16 [d_out] or NULL; Y bf16 [B, n, d_out].
 * Supported: d_model/H (resp. d) in {64, 128}; n a multiple of 32; d_out a
 * multiple of 64 (else ATTN_ERR_UNSUPPORTED). Pointers 16-byte aligned.
 * Returns ATTN_OK or a negative attn_status_t; on error nothing is enqueued.
 */
int attn_proj_heads(const void* X, const void* W, const void* bias, int B, int n, int d_model, int H,
                    int num_out, void* out0, void* out1, void* out2, void* stream);

int attn_merge_proj(const void* O, const void* W_o, const void* bias, int B, int n, int H, int d,
                    int d_out, void* Y, void* stream);

/* Human-readable name of a status code. */
const char* attn_status_string(int status);

/* Message of the last ATTN_ERR_CUDA on the calling thread ("" if none). */
const char* attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_SM103A_H */
