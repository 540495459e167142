// attn_api.cu -- C ABI of the sm_103a attention forward (declared in
// include/attn.h): argument validation, TMA tensor maps, the per-device
// status word and the kernel launch.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/attn.h"
#include "attn_internal.h"
#include "sm103a.cuh"

namespace {

constexpr uint64_t kDefaultWatchdogNs = 2000000000ull;   // 2 s per device-side wait
constexpr int kMaxDevices = 64;
constexpr int kMaxSeq = 1 << 30;   // n, m: row indices plus a tile stay within int

std::mutex g_mu;
uint32_t* g_status[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
uint64_t g_watchdog_ns = kDefaultWatchdogNs;
uint32_t g_debug_flags = 0;
thread_local char g_last_error[256] = "";
thread_local uint32_t g_last_detail = 0;   // bits read by this thread's last attn_get_device_status

int fail_cuda(const char* what, cudaError_t e)
{
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, cudaGetErrorString(e));
    return ATTN_ERR_CUDA;
}

int fail_msg(const char* what)
{
    snprintf(g_last_error, sizeof(g_last_error), "%s", what);
    return ATTN_ERR_CUDA;
}

// The device status word of the current device, created on first use.
int status_word(uint32_t** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) return fail_msg("device index out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_status[dev] == nullptr) {
        uint32_t* p = nullptr;
        e = cudaMalloc(&p, sizeof(uint32_t));
        if (e != cudaSuccess) return fail_cuda("cudaMalloc(status word)", e);
        e = cudaMemset(p, 0, sizeof(uint32_t));
        if (e != cudaSuccess) return fail_cuda("cudaMemset(status word)", e);
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return fail_cuda("cudaDeviceSynchronize", e);
        g_status[dev] = p;
    }
    *out = g_status[dev];
    return ATTN_OK;
}

// The current device's status word if it exists (no allocation); null otherwise.
int existing_status_word(uint32_t** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) return fail_msg("device index out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    *out = g_status[dev];
    return ATTN_OK;
}

int encoder(PFN_cuTensorMapEncodeTiled_v12000* out)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return fail_cuda("cudaGetDriverEntryPointByVersion", e);
        if (fn == nullptr || q != cudaDriverEntryPointSuccess)
            return fail_msg("cuTensorMapEncodeTiled not available");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return ATTN_OK;
}

// 3-D bf16 map over [bh][rows][d] with a {64, box_rows, 1} box and 128-byte swizzle.
int make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* base, int64_t bh,
             int64_t rows, int64_t d, uint32_t box_rows)
{
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(bh)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * 2), static_cast<cuuint64_t>(rows * d * 2)};
    cuuint32_t box[3] = {64u, box_rows, 1u};
    cuuint32_t es[3] = {1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed (%d)",
                 static_cast<int>(r));
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

// 3-D fp32 map over [bh][rows][d] with a {32, 32, 1} box and 128-byte swizzle
// (the backward's dQ accumulator, written by TMA reduce-add).
int make_map_f32(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, void* base, int64_t bh,
                 int64_t rows, int64_t d)
{
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(bh)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * 4), static_cast<cuuint64_t>(rows * d * 4)};
    cuuint32_t box[3] = {32u, 32u, 1u};
    cuuint32_t es[3] = {1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled (f32) failed (%d)",
                 static_cast<int>(r));
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

__global__ void fill_no_keys_kernel(uint16_t* O, int64_t o_elems, float* LSE, int64_t rows)
{
    sm103a::griddep_wait();   // earlier kernels' reads and writes of O and LSE come first
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    for (int64_t i = i0; i < o_elems; i += stride) O[i] = 0;
    if (LSE != nullptr)
        for (int64_t i = i0; i < rows; i += stride) LSE[i] = -INFINITY;
}

// Number of SMs of the current device (cached per device).
int sm_count(int* out)
{
    static int cached[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) return fail_msg("device index out of range");
    if (cached[dev] == 0) {
        int v = 0;
        e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail_cuda("cudaDeviceGetAttribute", e);
        cached[dev] = v;
    }
    *out = cached[dev];
    return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool head_dim_ok(int d) { return d == 64 || d == 128; }

// Host-side checks shared by both entry points.
int validate(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d_k, int d_v,
             int mask_kind, const int32_t* key_lengths, void* O, float* LSE)
{
    if (B < 0 || H < 0 || n < 0 || m < 0) return ATTN_ERR_INVALID_ARG;
    if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_CAUSAL_CACHE) return ATTN_ERR_INVALID_ARG;
    if (attn::mask_has_lengths(mask_kind) && key_lengths == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!head_dim_ok(d_k) || !head_dim_ok(d_v)) return ATTN_ERR_UNSUPPORTED;
    if (n > kMaxSeq || m > kMaxSeq) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || n == 0) return ATTN_OK;   // nothing to compute
    if (O == nullptr || (m > 0 && (Q == nullptr || K == nullptr || V == nullptr)))
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(O, 16) || !aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16))
        return ATTN_ERR_MISALIGNED;
    if ((LSE != nullptr && !aligned(LSE, 4)) || (key_lengths != nullptr && !aligned(key_lengths, 4)))
        return ATTN_ERR_MISALIGNED;
    const int64_t bh = static_cast<int64_t>(B) * H;
    const int64_t num_qblocks = (static_cast<int64_t>(n) + 127) / 128;
    if (bh > INT32_MAX || bh * num_qblocks > INT32_MAX) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// m = 0: no keys at all, every row gets O = 0 and LSE = -inf.
int fill_no_keys(int64_t bh, int n, int d_v, void* O, float* LSE, cudaStream_t st)
{
    const int64_t rows = bh * n;
    const int64_t elems = rows * d_v;
    const int64_t blocks = std::min<int64_t>((elems + 255) / 256, 152 * 8);
    const cudaError_t e = attn::launch_pdl(fill_no_keys_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                                           static_cast<uint16_t*>(O), elems, LSE, rows);
    return e == cudaSuccess ? ATTN_OK : fail_cuda("fill kernel launch", e);
}

// Tensor maps, parameters and the launch of the attention kernel (m >= 1),
// with `status` as the kernel's device status word; `slopes` (device fp32 [H])
// selects the kernel with the linear distance bias, null the plain one.
int launch_attention(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d_k,
                     int d_v, int mask_kind, const int32_t* key_lengths, float scale, void* O, float* LSE,
                     uint32_t* status, cudaStream_t st, const float* slopes = nullptr)
{
    const int64_t bh = static_cast<int64_t>(B) * H;
    const int64_t num_qblocks = (static_cast<int64_t>(n) + 127) / 128;

    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    int rc = encoder(&enc);
    if (rc != ATTN_OK) return rc;
    attn::TensorMaps maps;
    if ((rc = make_map(enc, &maps.q, Q, bh, n, d_k, 128)) != ATTN_OK) return rc;
    if ((rc = make_map(enc, &maps.k, K, bh, m, d_k, 128)) != ATTN_OK) return rc;
    if ((rc = make_map(enc, &maps.v, V, bh, m, d_v, 128)) != ATTN_OK) return rc;
    if ((rc = make_map(enc, &maps.o, O, bh, n, d_v, 32)) != ATTN_OK) return rc;

    const double sc = (scale > 0.f && std::isfinite(scale)) ? static_cast<double>(scale)
                                                             : 1.0 / std::sqrt(static_cast<double>(d_k));
    const bool paired = attn::mask_is_causal(mask_kind);   // causal units pair two query tiles
    attn::FwdParams p;
    p.B = B;
    p.H = H;
    p.n = n;
    p.m = m;
    p.causal_off = m - n;
    p.num_qblocks = static_cast<int>(num_qblocks);
    p.num_units = static_cast<int>(bh * (paired ? (num_qblocks + 1) / 2 : num_qblocks));
    p.O = O;
    p.key_lengths = attn::mask_has_lengths(mask_kind) ? key_lengths : nullptr;
    p.scale_log2 = static_cast<float>(sc * 1.4426950408889634074);
    p.LSE = LSE;
    p.slopes = slopes;
    p.status = status;
    p.watchdog_ns = g_watchdog_ns;
    p.debug_flags = g_debug_flags;

    int num_sms = 0;
    if ((rc = sm_count(&num_sms)) != ATTN_OK) return rc;
    cudaError_t e;
    if (slopes != nullptr)
        e = attn::launch_fwd_alibi(d_k, d_v, mask_kind, maps, p, num_sms, st);
    else if (d_k != d_v)
        e = attn::launch_fwd_dmix(d_k, d_v, mask_kind, maps, p, num_sms, st);
    else if (d_k == 64)
        e = attn::launch_fwd_d64(mask_kind, maps, p, num_sms, st);
    else
        e = attn::launch_fwd_d128(mask_kind, maps, p, num_sms, st);
    return e == cudaSuccess ? ATTN_OK : fail_cuda("attention kernel launch", e);
}

// ---------------------------------------------------------------------------
// Entry point for callers that may not allocate device memory.
//
// attn_fwd keeps its device status word (the kernel's only scratch memory) in
// a 4-byte cudaMalloc made on the first call on each device. Some callers
// cannot allow that: code that runs while another component owns every
// allocation (a caching or pooled allocator, a fixed memory budget), or code
// that must not add device allocations after start-up. attn_fwd_noalloc runs
// the same kernel with its scratch taken from this file-scope device array.

// The array's stated size. One call uses its first word as the kernel's status
// word, whatever the problem sizes (the forward kernel needs no other scratch).
constexpr size_t kNoAllocScratchBytes = 256;
constexpr size_t kNoAllocStatusBytes = sizeof(uint32_t);
static_assert(kNoAllocStatusBytes <= kNoAllocScratchBytes, "scratch layout");

static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(uint32_t)];

std::mutex g_noalloc_mu;
uint32_t* g_noalloc_addr[kMaxDevices] = {};   // device address of the array, per device

// Device address of the scratch array on the current device, looked up once
// per device. In host code the array's name is only a host-side stand-in.
int noalloc_scratch(uint32_t** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) return fail_msg("device index out of range");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return fail_cuda("cudaGetSymbolAddress(no-allocation scratch)", e);
        if (ptr == nullptr) return fail_msg("no-allocation scratch has no device address");
        g_noalloc_addr[dev] = static_cast<uint32_t*>(ptr);
    }
    *out = g_noalloc_addr[dev];
    return ATTN_OK;
}

// The array's device address on the current device if a call has looked it up
// there already; null otherwise.
int existing_noalloc_scratch(uint32_t** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) return fail_msg("device index out of range");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    *out = g_noalloc_addr[dev];
    return ATTN_OK;
}

// Reads a device status word and, if it is non-zero, clears it on `st`.
int read_and_clear(uint32_t* word, cudaStream_t st, uint32_t* value)
{
    uint32_t v = 0;
    cudaError_t e = cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda("cudaMemcpy(status word)", e);
    if (v != 0) {
        e = cudaMemsetAsync(word, 0, sizeof(uint32_t), st);
        if (e != cudaSuccess) return fail_cuda("cudaMemsetAsync(status word)", e);
        e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return fail_cuda("cudaStreamSynchronize", e);
    }
    *value = v;
    return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d_k,
             int d_v, int mask_kind, const int32_t* key_lengths, float scale, void* O, float* LSE,
             void* stream)
{
    int rc = validate(Q, K, V, B, H, n, m, d_k, d_v, mask_kind, key_lengths, O, LSE);
    if (rc != ATTN_OK || B == 0 || H == 0 || n == 0) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (m == 0) return fill_no_keys(static_cast<int64_t>(B) * H, n, d_v, O, LSE, st);
    uint32_t* status = nullptr;
    if ((rc = status_word(&status)) != ATTN_OK) return rc;
    return launch_attention(Q, K, V, B, H, n, m, d_k, d_v, mask_kind, key_lengths, scale, O, LSE, status, st);
}

int attn_fwd_alibi(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d_k,
                   int d_v, int mask_kind, const int32_t* key_lengths, const float* slopes, float scale,
                   void* O, float* LSE, void* stream)
{
    int rc = validate(Q, K, V, B, H, n, m, d_k, d_v, mask_kind, key_lengths, O, LSE);
    if (rc != ATTN_OK || B == 0 || H == 0 || n == 0) return rc;
    if (slopes == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned(slopes, 4)) return ATTN_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (m == 0) return fill_no_keys(static_cast<int64_t>(B) * H, n, d_v, O, LSE, st);
    uint32_t* status = nullptr;
    if ((rc = status_word(&status)) != ATTN_OK) return rc;
    return launch_attention(Q, K, V, B, H, n, m, d_k, d_v, mask_kind, key_lengths, scale, O, LSE, status, st,
                            slopes);
}

int attn_get_device_status(void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    g_last_detail = 0;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail_cuda("cudaStreamSynchronize", e);
    // attn_fwd's word (absent until a call created it) and the word in the
    // no-allocation entry point's array (known once a call looked it up)
    uint32_t* words[2] = {nullptr, nullptr};
    int rc = existing_status_word(&words[0]);
    if (rc == ATTN_OK) rc = existing_noalloc_scratch(&words[1]);
    if (rc != ATTN_OK) return rc;
    uint32_t bits = 0;
    for (uint32_t* w : words) {
        if (w == nullptr) continue;
        uint32_t v = 0;
        if ((rc = read_and_clear(w, st, &v)) != ATTN_OK) return rc;
        bits |= v;
    }
    g_last_detail = bits;
    return bits != 0 ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

uint32_t attn_last_status_detail(void) { return g_last_detail; }

void attn_set_watchdog(uint64_t limit_ns, uint32_t debug_flags)
{
    g_watchdog_ns = limit_ns == 0 ? kDefaultWatchdogNs : limit_ns;
    g_debug_flags = debug_flags;
}

const char* attn_status_string(int status)
{
    switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    default: return "ATTN_ERR_UNKNOWN";
    }
}

const char* attn_last_error(void) { return g_last_error; }

}  // extern "C"

extern "C" int attn_fwd_noalloc(const void* Q, const void* K, const void* V, int B, int H, int n, int m,
                                int d_k, int d_v, int mask_kind, const int32_t* key_lengths, float scale,
                                void* O, float* LSE, void* stream)
{
    int rc = validate(Q, K, V, B, H, n, m, d_k, d_v, mask_kind, key_lengths, O, LSE);
    if (rc != ATTN_OK || B == 0 || H == 0 || n == 0) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (m == 0) return fill_no_keys(static_cast<int64_t>(B) * H, n, d_v, O, LSE, st);
    uint32_t* scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch)) != ATTN_OK) return rc;
    // The kernel only ORs bits into its status word and never reads it back, so the
    // word needs no reset before a call: it starts at zero when the module loads and
    // attn_get_device_status clears it once it has read it (like attn_fwd's word).
    return launch_attention(Q, K, V, B, H, n, m, d_k, d_v, mask_kind, key_lengths, scale, O, LSE, scratch, st);
}

// ---------------------------------------------------------------------------
// Backward.
namespace {

constexpr size_t kWsAlign = 256;
constexpr float kLog2e = 1.4426950408889634074f;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: dQ accumulator fp32 [B*H, n, d_k], then LSE*log2(e) and D, each fp32
// [B*H, n_pad] with n_pad = n rounded up to whole 128-row query tiles.
struct BwdWorkspace {
    size_t lse_off, dd_off, total;
    int64_t n_pad;
};

BwdWorkspace bwd_workspace(int64_t bh, int64_t n, int64_t d_k)
{
    BwdWorkspace w;
    w.n_pad = (n + 127) / 128 * 128;
    const size_t dq = round_up(static_cast<size_t>(bh * n * d_k) * 4, kWsAlign);
    const size_t row = round_up(static_cast<size_t>(bh * w.n_pad) * 4, kWsAlign);
    w.lse_off = dq;
    w.dd_off = dq + row;
    w.total = dq + 2 * row;
    return w;
}

// D_i = sum_c dO_ic O_ic (fp32 from the bf16 tensors) and LSE_i * log2(e) for every
// row of the padded layout (0 in the padding), and the row's d_k accumulator
// entries zeroed, in one pass over the rows, so that the reads of O and dO and the
// zero writes stream together. A group of G = d_v / 8 lanes takes a row (16 bytes
// of O and of dO per lane, d_k / (4 G) float4 of zeros); a warp takes two sets of
// 32 / G rows per iteration, so that every lane has four 16-byte loads in flight.
__global__ void bwd_prep_kernel(const uint16_t* __restrict__ O, const uint16_t* __restrict__ dO,
                                const float* __restrict__ LSE, int64_t bh_count, int n, int64_t n_pad, int d_k,
                                int d_v, float* __restrict__ lse2, float* __restrict__ dd, float4* __restrict__ dq_acc)
{
    sm103a::griddep_wait();   // O, dO and LSE of the earlier kernels are visible
    const int G = d_v / 8;                       // lanes per row: 8 or 16
    const int lane = threadIdx.x % 32;
    const int g = lane % G;
    const int zq = d_k / 4;                      // float4 per accumulator row
    const int64_t total = bh_count * n_pad;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x / 32 * (32 / G);   // rows per sweep
    const uint64_t keep = sm103a::l2_policy_evict_last();   // the accumulator is added into and read back next
    for (int64_t base = warp_id * (32 / G); base < total; base += 2 * step) {
        uint4 a[2], b[2];
        float lz[2];
        bool valid[2];
        int64_t row[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            row[u] = base + u * step + lane / G;
            const int64_t bh = row[u] / n_pad;
            const int64_t q = row[u] - bh * n_pad;
            valid[u] = row[u] < total && q < n;
            a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
            lz[u] = 0.f;
            if (valid[u]) {
                const int64_t r = bh * n + q;
                a[u] = *reinterpret_cast<const uint4*>(O + r * d_v + 8 * g);
                b[u] = *reinterpret_cast<const uint4*>(dO + r * d_v + 8 * g);
                if (g == 0) lz[u] = LSE[r];
                for (int i = g; i < zq; i += G)
                    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %1, %1, %1}, %2;" ::"l"(dq_acc + r * zq + i),
                                 "f"(0.f), "l"(keep)
                                 : "memory");
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const uint32_t av[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
            const uint32_t bv[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc = fmaf(__uint_as_float(av[k] << 16), __uint_as_float(bv[k] << 16), acc);
                acc = fmaf(__uint_as_float(av[k] & 0xFFFF0000u), __uint_as_float(bv[k] & 0xFFFF0000u), acc);
            }
            for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (g == 0 && row[u] < total) {
                dd[row[u]] = valid[u] ? acc : 0.f;
                lse2[row[u]] = valid[u] ? lz[u] * kLog2e : 0.f;
            }
        }
    }
}

// dQ = bf16(scale * accumulator), four elements per step.
__global__ void bwd_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ dQ, int64_t vec, float scale)
{
    sm103a::griddep_wait();   // the main kernel's reduce-adds into the accumulator are complete
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < vec; i += stride) {
        const float4 a = acc[i];
        const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * scale, a.y * scale);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * scale, a.w * scale);
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t*>(&lo);
        o.y = *reinterpret_cast<const uint32_t*>(&hi);
        dQ[i] = o;
    }
}

int64_t grid_for(int64_t work, int64_t per_block)
{
    return std::max<int64_t>(1, std::min<int64_t>((work + per_block - 1) / per_block, 152 * 8));
}

}  // namespace

extern "C" size_t attn_bwd_workspace_size(int B, int H, int n, int m, int d_k, int d_v)
{
    (void)m;
    (void)d_v;
    if (B <= 0 || H <= 0 || n <= 0 || d_k <= 0) return 0;
    return bwd_workspace(static_cast<int64_t>(B) * H, n, d_k).total;
}

namespace {

// The backward; `slopes` (device fp32 [H]) for the forward with the linear distance bias, null without.
int bwd_impl(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE, int B,
             int H, int n, int m, int d_k, int d_v, int mask_kind, const int32_t* key_lengths, const float* slopes,
             float scale, void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes, void* stream)
{
    if (B < 0 || H < 0 || n < 0 || m < 0) return ATTN_ERR_INVALID_ARG;
    if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_CAUSAL_CACHE) return ATTN_ERR_INVALID_ARG;
    if (attn::mask_has_lengths(mask_kind) && key_lengths == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!head_dim_ok(d_k) || !head_dim_ok(d_v)) return ATTN_ERR_UNSUPPORTED;
    if (n > kMaxSeq || m > kMaxSeq) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0) return ATTN_OK;
    const int64_t bh = static_cast<int64_t>(B) * H;
    if (bh > INT32_MAX || bh * ((static_cast<int64_t>(m) + 127) / 128) > INT32_MAX) return ATTN_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool have_rows = n > 0, have_keys = m > 0;
    if ((have_rows && dQ == nullptr) || (have_keys && (dK == nullptr || dV == nullptr))) return ATTN_ERR_INVALID_ARG;
    if ((dQ && !aligned(dQ, 16)) || (dK && !aligned(dK, 16)) || (dV && !aligned(dV, 16)))
        return ATTN_ERR_MISALIGNED;
    if (!have_rows || !have_keys) {
        // no queries: dK = dV = 0; no keys: O = 0 is constant, dQ = 0
        cudaError_t e = cudaSuccess;
        if (!have_rows) {
            e = cudaMemsetAsync(dK, 0, static_cast<size_t>(bh) * m * d_k * 2, st);
            if (e == cudaSuccess) e = cudaMemsetAsync(dV, 0, static_cast<size_t>(bh) * m * d_v * 2, st);
        } else {
            e = cudaMemsetAsync(dQ, 0, static_cast<size_t>(bh) * n * d_k * 2, st);
        }
        return e == cudaSuccess ? ATTN_OK : fail_cuda("cudaMemsetAsync(empty gradient)", e);
    }
    if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr || dO == nullptr || LSE == nullptr ||
        workspace == nullptr)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(dO, 16) ||
        !aligned(LSE, 4) || !aligned(workspace, kWsAlign) || (key_lengths != nullptr && !aligned(key_lengths, 4)))
        return ATTN_ERR_MISALIGNED;
    const BwdWorkspace ws = bwd_workspace(bh, n, d_k);
    if (workspace_bytes < ws.total) return ATTN_ERR_INVALID_ARG;

    uint32_t* status = nullptr;
    int rc = status_word(&status);
    if (rc != ATTN_OK) return rc;
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if ((rc = encoder(&enc)) != ATTN_OK) return rc;
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    float* dq_acc = reinterpret_cast<float*>(wsb);
    float* lse2 = reinterpret_cast<float*>(wsb + ws.lse_off);
    float* dd = reinterpret_cast<float*>(wsb + ws.dd_off);

    attn::BwdMaps maps;
    // the d_k = d_v = 128 kernel walks the queries in 64-row steps
    const uint32_t q_box = (d_k == 128 && d_v == 128) ? 64u : 128u;
    if ((rc = make_map(enc, &maps.q, Q, bh, n, d_k, q_box)) != ATTN_OK) return rc;
    if ((rc = make_map(enc, &maps.k, K, bh, m, d_k, 128)) != ATTN_OK) return rc;
    if ((rc = make_map(enc, &maps.v, V, bh, m, d_v, 128)) != ATTN_OK) return rc;
    if ((rc = make_map(enc, &maps.dout, dO, bh, n, d_v, q_box)) != ATTN_OK) return rc;
    if ((rc = make_map(enc, &maps.dk, dK, bh, m, d_k, 32)) != ATTN_OK) return rc;
    if ((rc = make_map(enc, &maps.dv, dV, bh, m, d_v, 32)) != ATTN_OK) return rc;
    if ((rc = make_map_f32(enc, &maps.dq_acc, dq_acc, bh, n, d_k)) != ATTN_OK) return rc;

    const double sc = (scale > 0.f && std::isfinite(scale)) ? static_cast<double>(scale)
                                                             : 1.0 / std::sqrt(static_cast<double>(d_k));
    attn::BwdParams p;
    p.B = B;
    p.H = H;
    p.n = n;
    p.m = m;
    p.causal_off = m - n;
    p.num_kblocks = static_cast<int>((static_cast<int64_t>(m) + 127) / 128);
    if ((rc = sm_count(&p.num_sms)) != ATTN_OK) return rc;
    p.n_pad = static_cast<int>(ws.n_pad);
    p.key_lengths = attn::mask_has_lengths(mask_kind) ? key_lengths : nullptr;
    p.lse2 = lse2;
    p.dd = dd;
    p.dK = dK;
    p.dV = dV;
    p.scale_log2 = static_cast<float>(sc * 1.4426950408889634074);
    p.scale = static_cast<float>(sc);
    p.slopes = slopes;
    p.status = status;
    p.watchdog_ns = g_watchdog_ns;
    p.debug_flags = g_debug_flags;

    const int64_t dq_vec = bh * n * d_k / 4;
    const int64_t prep_threads = (bh * ws.n_pad * (d_v / 8) + 1) / 2;   // two rows per lane group
    cudaError_t e = attn::launch_pdl(bwd_prep_kernel, dim3(static_cast<unsigned>(grid_for(prep_threads, 256))), dim3(256),
                                     0, st, static_cast<const uint16_t*>(O), static_cast<const uint16_t*>(dO), LSE,
                                     bh, n, ws.n_pad, d_k, d_v, lse2, dd, reinterpret_cast<float4*>(dq_acc));
    if (e != cudaSuccess) return fail_cuda("backward preparation kernel launch", e);
    if (slopes != nullptr)
        e = attn::launch_bwd_alibi(d_k, d_v, mask_kind, maps, p, st);
    else if (d_k != d_v)
        e = attn::launch_bwd_dmix(d_k, d_v, mask_kind, maps, p, st);
    else
        e = d_k == 64 ? attn::launch_bwd_d64(mask_kind, maps, p, st) : attn::launch_bwd_d128(mask_kind, maps, p, st);
    if (e != cudaSuccess) return fail_cuda("backward kernel launch", e);
    e = attn::launch_pdl(bwd_convert_kernel, dim3(static_cast<unsigned>(grid_for(dq_vec, 256))), dim3(256), 0, st,
                         reinterpret_cast<const float4*>(dq_acc), static_cast<uint2*>(dQ), dq_vec, p.scale);
    return e == cudaSuccess ? ATTN_OK : fail_cuda("dQ conversion kernel launch", e);
}

}  // namespace

extern "C" int attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                        const float* LSE, int B, int H, int n, int m, int d_k, int d_v, int mask_kind,
                        const int32_t* key_lengths, float scale, void* dQ, void* dK, void* dV, void* workspace,
                        size_t workspace_bytes, void* stream)
{
    return bwd_impl(Q, K, V, O, dO, LSE, B, H, n, m, d_k, d_v, mask_kind, key_lengths, nullptr, scale, dQ, dK, dV,
                    workspace, workspace_bytes, stream);
}

extern "C" int attn_bwd_alibi(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                              const float* LSE, int B, int H, int n, int m, int d_k, int d_v, int mask_kind,
                              const int32_t* key_lengths, const float* slopes, float scale, void* dQ, void* dK,
                              void* dV, void* workspace, size_t workspace_bytes, void* stream)
{
    if (slopes == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned(slopes, 4)) return ATTN_ERR_MISALIGNED;
    return bwd_impl(Q, K, V, O, dO, LSE, B, H, n, m, d_k, d_v, mask_kind, key_lengths, slopes, scale, dQ, dK, dV,
                    workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// Few-row forward (decoding against a key/value cache).
namespace {

constexpr int kDecodeMaxRows = 8;
constexpr int64_t kDecodeMaxCtas = 2048;      // bound on B*H*chunks used to size the workspace
constexpr int64_t kDecodeCtaOverheadKeys = 256;

// Largest number of key chunks (of at least 256 keys) a launch may use for
// this shape; independent of the device so that the workspace size can be
// computed without one.
int64_t decode_split_cap(int64_t bh, int m)
{
    const int64_t by_keys = std::max<int64_t>(1, (m + 255) / 256);
    const int64_t by_ctas = std::max<int64_t>(1, (kDecodeMaxCtas + bh - 1) / bh);
    return std::min(by_keys, by_ctas);
}

// Chunk count for a launch on `slots` concurrent CTAs (SMs x CTAs per SM): the
// count in [1, cap] that minimises waves x (keys per CTA + a per-CTA overhead),
// the smaller one on ties. Chunks are whole 128-key tiles.
// attn_decode hands problems with at least this many (b, h) pairs per CTA slot to
// the forward kernel (measured with 1024 pairs on 152 slots, d = 128, 8192 keys:
// 452 against 510 us at n = 1, 470 against 937 us at n = 4).
constexpr int64_t kDecodeTileWaves = 4;

void decode_split(int64_t bh, int m, int64_t slots, int* split_len, int* num_splits)
{
    const int64_t cap = decode_split_cap(bh, m);
    int64_t best_s = 1, best_t = INT64_MAX;
    for (int64_t s = 1; s <= cap; ++s) {
        const int64_t len = ((m + s - 1) / s + 127) / 128 * 128;
        const int64_t used = (m + len - 1) / len;                 // chunks that hold keys
        if (used != s) continue;
        const int64_t waves = (bh * s + slots - 1) / slots;
        const int64_t t = waves * (len + kDecodeCtaOverheadKeys);
        if (t < best_t) {
            best_t = t;
            best_s = s;
        }
    }
    const int64_t len = ((m + best_s - 1) / best_s + 127) / 128 * 128;
    *split_len = static_cast<int>(len);
    *num_splits = static_cast<int>(best_s);
}

int decode_rows(int n) { return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : 8; }

}  // namespace

extern "C" size_t attn_decode_workspace_size(int B, int H, int n, int m, int d_k, int d_v)
{
    (void)d_k;
    if (B <= 0 || H <= 0 || n <= 0 || m <= 0 || d_v <= 0 || n > kDecodeMaxRows) return 0;
    const int64_t bh = static_cast<int64_t>(B) * H;
    const int64_t cap = decode_split_cap(bh, m);
    if (cap == 1) return 0;
    const size_t rows = static_cast<size_t>(bh) * cap * n;
    return round_up(rows * d_v * 4, kWsAlign) + round_up(rows * 2 * 4, kWsAlign);
}

namespace {

// The few-row forward; `slopes` (device fp32 [H]) adds the linear distance bias, null none.
int decode_impl(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d_k, int d_v,
                int mask_kind, const int32_t* key_lengths, const float* slopes, float scale, void* O, float* LSE,
                void* workspace, size_t workspace_bytes, void* stream)
{
    if (B < 0 || H < 0 || n < 0 || m < 0) return ATTN_ERR_INVALID_ARG;
    if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_CAUSAL_CACHE) return ATTN_ERR_INVALID_ARG;
    if (attn::mask_has_lengths(mask_kind) && key_lengths == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!head_dim_ok(d_k) || !head_dim_ok(d_v)) return ATTN_ERR_UNSUPPORTED;
    if (m > kMaxSeq) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || n == 0) return ATTN_OK;
    const int64_t bh = static_cast<int64_t>(B) * H;
    if (O == nullptr || (m > 0 && (Q == nullptr || K == nullptr || V == nullptr))) return ATTN_ERR_INVALID_ARG;
    if (!aligned(O, 16) || !aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16)) return ATTN_ERR_MISALIGNED;
    if ((LSE != nullptr && !aligned(LSE, 4)) || (key_lengths != nullptr && !aligned(key_lengths, 4)))
        return ATTN_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (m == 0) return fill_no_keys(bh, n, d_v, O, LSE, st);
    const size_t need = attn_decode_workspace_size(B, H, n, m, d_k, d_v);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return ATTN_ERR_INVALID_ARG;
    if (need > 0 && !aligned(workspace, kWsAlign)) return ATTN_ERR_MISALIGNED;
    if (bh * decode_split_cap(bh, m) > INT32_MAX) return ATTN_ERR_UNSUPPORTED;
    int num_sms = 0;
    int rc0 = sm_count(&num_sms);
    if (rc0 != ATTN_OK) return rc0;
    // the forward kernel's CTA slots decide the path; the split kernel's size the chunks
    const int64_t tile_slots = static_cast<int64_t>(num_sms) * (d_k == 64 && d_v == 64 ? 2 : 1);
    const int64_t slots = static_cast<int64_t>(num_sms) * attn::decode_ctas_per_sm(d_k, d_v, decode_rows(n));
    if (n > kDecodeMaxRows || bh >= kDecodeTileWaves * tile_slots) {
        // More rows than the split kernel holds, or enough (b, h) pairs to fill
        // every SM several times over: the tensor-core forward kernel streams each
        // pair's K and V once at the memory system's rate (its 128-row query tile
        // is mostly padding, which the tensor cores absorb), and no chunk merge is
        // needed.
        uint32_t* status = nullptr;
        int rc = status_word(&status);
        if (rc != ATTN_OK) return rc;
        return launch_attention(Q, K, V, B, H, n, m, d_k, d_v, mask_kind, key_lengths, scale, O, LSE, status, st,
                                slopes);
    }
    int split_len = 0, num_splits = 0;
    decode_split(bh, m, slots, &split_len, &num_splits);

    uint32_t* status = nullptr;
    int rc = status_word(&status);
    if (rc != ATTN_OK) return rc;
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if ((rc = encoder(&enc)) != ATTN_OK) return rc;
    CUtensorMap tmK, tmV;
    if ((rc = make_map(enc, &tmK, K, bh, m, d_k, 128)) != ATTN_OK) return rc;
    if ((rc = make_map(enc, &tmV, V, bh, m, d_v, 128)) != ATTN_OK) return rc;

    const double sc = (scale > 0.f && std::isfinite(scale)) ? static_cast<double>(scale)
                                                             : 1.0 / std::sqrt(static_cast<double>(d_k));
    attn::DecodeParams p;
    p.Q = static_cast<const uint16_t*>(Q);
    p.B = B;
    p.H = H;
    p.n = n;
    p.m = m;
    p.causal_off = m - n;
    p.mask = mask_kind;
    p.key_lengths = attn::mask_has_lengths(mask_kind) ? key_lengths : nullptr;
    p.scale_log2 = static_cast<float>(sc * 1.4426950408889634074);
    p.split_len = split_len;
    p.num_splits = num_splits;
    p.O = static_cast<uint16_t*>(O);
    p.LSE = LSE;
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    // partials laid out for the cap's chunk count; the launch uses num_splits <= cap of them
    const size_t prow = static_cast<size_t>(bh) * decode_split_cap(bh, m) * n;
    p.part_o = num_splits > 1 ? reinterpret_cast<float*>(wsb) : nullptr;
    p.part_ml = num_splits > 1 ? reinterpret_cast<float*>(wsb + round_up(prow * d_v * 4, kWsAlign)) : nullptr;
    p.slopes = slopes;
    p.status = status;
    p.watchdog_ns = g_watchdog_ns;
    p.debug_flags = g_debug_flags;
    cudaError_t e = attn::launch_decode(d_k, d_v, decode_rows(n), tmK, tmV, p, st);
    return e == cudaSuccess ? ATTN_OK : fail_cuda("decode kernel launch", e);
}

}  // namespace

extern "C" int attn_decode(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d_k,
                           int d_v, int mask_kind, const int32_t* key_lengths, float scale, void* O, float* LSE,
                           void* workspace, size_t workspace_bytes, void* stream)
{
    return decode_impl(Q, K, V, B, H, n, m, d_k, d_v, mask_kind, key_lengths, nullptr, scale, O, LSE, workspace,
                       workspace_bytes, stream);
}

extern "C" int attn_decode_alibi(const void* Q, const void* K, const void* V, int B, int H, int n, int m,
                                 int d_k, int d_v, int mask_kind, const int32_t* key_lengths, const float* slopes,
                                 float scale, void* O, float* LSE, void* workspace, size_t workspace_bytes,
                                 void* stream)
{
    if (slopes == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned(slopes, 4)) return ATTN_ERR_MISALIGNED;
    return decode_impl(Q, K, V, B, H, n, m, d_k, d_v, mask_kind, key_lengths, slopes, scale, O, LSE, workspace,
                       workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// Projections around the attention.
namespace {

// Any-rank tiled map with 128-byte swizzle; dims innermost first, strides in bytes
// for dims 1..rank-1.
int encode_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, CUtensorMapDataType type, uint32_t rank,
               const void* base, const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box)
{
    cuuint32_t es[5] = {1u, 1u, 1u, 1u, 1u};
    CUresult r = enc(map, type, rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled (rank %u) failed (%d)", rank,
                 static_cast<int>(r));
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

// [rows][cols] bf16 matrix as a 3-D map {cols, rows, 1} with a {64, box_rows, 1} box.
int matrix_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* base, int64_t rows,
               int64_t cols, uint32_t box_rows)
{
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols * 2), static_cast<cuuint64_t>(rows * cols * 2)};
    cuuint32_t box[3] = {64u, box_rows, 1u};
    return encode_map(enc, map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box);
}

// [B][H][n][d] bf16 head tensor as a 4-D map with a {64, box_rows, 1, 1} box.
int heads_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* base, int64_t B, int64_t H,
              int64_t n, int64_t d, uint32_t box_rows)
{
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d * 2), static_cast<cuuint64_t>(n * d * 2),
                             static_cast<cuuint64_t>(H * n * d * 2)};
    cuuint32_t box[4] = {64u, box_rows, 1u, 1u};
    return encode_map(enc, map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box);
}

int run_proj(bool heads_in, bool heads_out, attn::ProjMaps& maps, attn::ProjParams& p, cudaStream_t st)
{
    uint32_t* status = nullptr;
    int rc = status_word(&status);
    if (rc != ATTN_OK) return rc;
    int num_sms = 0;
    if ((rc = sm_count(&num_sms)) != ATTN_OK) return rc;
    p.tiles_m = (p.R + 127) / 128;
    p.tiles_n = (p.N + 255) / 256;
    p.status = status;
    p.watchdog_ns = g_watchdog_ns;
    p.debug_flags = g_debug_flags;
    cudaError_t e = attn::launch_proj(heads_in, heads_out, maps, p, num_sms, st);
    return e == cudaSuccess ? ATTN_OK : fail_cuda("projection kernel launch", e);
}

}  // namespace

extern "C" int attn_proj_heads(const void* X, const void* W, const void* bias, int B, int n, int d_model, int H,
                               int num_out, void* out0, void* out1, void* out2, void* stream)
{
    if (B < 0 || n < 0 || d_model < 1 || H < 1 || num_out < 1 || num_out > 3) return ATTN_ERR_INVALID_ARG;
    if (d_model % H != 0 || !head_dim_ok(d_model / H)) return ATTN_ERR_UNSUPPORTED;
    if (n % 32 != 0) return ATTN_ERR_UNSUPPORTED;
    const int64_t R = static_cast<int64_t>(B) * n;
    if (R > INT32_MAX / 2 || static_cast<int64_t>(num_out) * d_model > 65536) return ATTN_ERR_UNSUPPORTED;
    if (R == 0) return ATTN_OK;
    void* outs[3] = {out0, out1, out2};
    if (X == nullptr || W == nullptr) return ATTN_ERR_INVALID_ARG;
    for (int t = 0; t < num_out; ++t)
        if (outs[t] == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(W, 16) || (bias != nullptr && !aligned(bias, 16))) return ATTN_ERR_MISALIGNED;
    for (int t = 0; t < num_out; ++t)
        if (!aligned(outs[t], 16)) return ATTN_ERR_MISALIGNED;
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    int rc = encoder(&enc);
    if (rc != ATTN_OK) return rc;
    const int d = d_model / H;
    const int N = num_out * d_model;
    attn::ProjMaps maps;
    if ((rc = matrix_map(enc, &maps.a, X, R, d_model, 128)) != ATTN_OK) return rc;
    if ((rc = matrix_map(enc, &maps.w, W, N, d_model, 256)) != ATTN_OK) return rc;
    for (int t = 0; t < 3; ++t)
        if ((rc = heads_map(enc, &maps.c[t], outs[t < num_out ? t : 0], B, H, n, d, 32)) != ATTN_OK) return rc;
    attn::ProjParams p;
    p.R = static_cast<int>(R);
    p.N = N;
    p.K = d_model;
    p.n = n;
    p.H = H;
    p.d = d;
    p.d_block = d_model;
    p.a_box_rows = 128;
    p.bias = static_cast<const uint16_t*>(bias);
    return run_proj(false, true, maps, p, static_cast<cudaStream_t>(stream));
}

extern "C" int attn_merge_proj(const void* O, const void* W_o, const void* bias, int B, int n, int H, int d,
                               int d_out, void* Y, void* stream)
{
    if (B < 0 || n < 0 || H < 1 || d_out < 1) return ATTN_ERR_INVALID_ARG;
    if (!head_dim_ok(d) || d_out % 64 != 0 || n % 32 != 0) return ATTN_ERR_UNSUPPORTED;
    const int64_t R = static_cast<int64_t>(B) * n;
    if (R > INT32_MAX / 2 || static_cast<int64_t>(H) * d > 65536 || d_out > 65536) return ATTN_ERR_UNSUPPORTED;
    if (R == 0) return ATTN_OK;
    if (O == nullptr || W_o == nullptr || Y == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned(O, 16) || !aligned(W_o, 16) || !aligned(Y, 16) || (bias != nullptr && !aligned(bias, 16)))
        return ATTN_ERR_MISALIGNED;
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    int rc = encoder(&enc);
    if (rc != ATTN_OK) return rc;
    const int K = H * d;
    attn::ProjMaps maps;
    const uint32_t a_rows = n % 128 == 0 ? 128u : 32u;
    if ((rc = heads_map(enc, &maps.a, O, B, H, n, d, a_rows)) != ATTN_OK) return rc;
    if ((rc = matrix_map(enc, &maps.w, W_o, d_out, K, 256)) != ATTN_OK) return rc;
    if ((rc = matrix_map(enc, &maps.c[0], Y, R, d_out, 32)) != ATTN_OK) return rc;
    maps.c[1] = maps.c[0];
    maps.c[2] = maps.c[0];
    attn::ProjParams p;
    p.R = static_cast<int>(R);
    p.N = d_out;
    p.K = K;
    p.n = n;
    p.H = H;
    p.d = d;
    p.d_block = d_out;
    p.a_box_rows = static_cast<int>(a_rows);
    p.bias = static_cast<const uint16_t*>(bias);
    return run_proj(true, false, maps, p, static_cast<cudaStream_t>(stream));
}
