// Forward pass that allocates no device memory, for callers that cannot call
// cudaMalloc: code running where the allocator is owned by someone else (a
// framework's caching allocator that must see every allocation, an embedded
// runtime that fixes its memory budget at start-up) or code that must not
// allocate once it is up (a latency-critical serving loop, where a
// cudaMalloc would synchronise the device).  It runs the same three kernels
// as swin_wattn_forward (QKV GEMM with the roll+partition gather, window
// attention, projection GEMM with the reverse+roll scatter), but their
// intermediates live in one fixed array compiled into the library instead of
// a workspace the handle allocates.
#include <mutex>

#include "swin_wattn.h"
#include "swin_wattn_test.h"
#include "common.cuh"

using namespace swin;

namespace {

// The fixed scratch: 256 bytes of status word, then the q/k/v buffer
// [T, 3C] and the attention output [T, C], bf16.  Every GPU that loads the
// library holds this array until the process exits.
constexpr size_t kStatusBytes = 256;
constexpr size_t kScratchBytes = SWIN_WATTN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
// Per device: the device address of the array and the context it was looked
// up in.  A device reset (or the primary context released and created again)
// gives the device a new context, in which the library's device code -- and
// so the array -- is loaded again, possibly at another address: the address
// is looked up again whenever the current context differs.
void *g_scratch_on_device[kMaxDevices];
void *g_scratch_context[kMaxDevices];

// cuCtxGetCurrent through the runtime's driver entry point (the library does
// not link libcuda itself).
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
CtxGetCurrentFn ctx_get_current()
{
    static CtxGetCurrentFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(f);
    }();
    return fn;
}

// The device address of the scratch on the current device.  The first call on
// a device (and the first after its context changed) looks it up, which may
// load the library's device code on that device; later calls reuse it.
int scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SWIN_WATTN_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return SWIN_WATTN_EUNSUPPORTED;
    // (cudaGetSymbolAddress below makes the device's primary context current
    // if none is; the context is read after it)
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    CUcontext ctx = nullptr;
    CtxGetCurrentFn get = ctx_get_current();
    if (g_scratch_on_device[dev] && get && get(&ctx) == CUDA_SUCCESS && ctx == g_scratch_context[dev]) {
        *out = g_scratch_on_device[dev];
        return SWIN_WATTN_OK;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return SWIN_WATTN_ECUDA;
    }
    ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    g_scratch_on_device[dev] = p;
    g_scratch_context[dev] = ctx;   // null: looked up again on every call
    *out = p;
    return SWIN_WATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

} // namespace

extern "C" int swin_wattn_forward_noalloc(int C, int heads, int M, int shift, int mode, const void *x, int B, int H,
                                          int W, const void *Wqkv, const void *bqkv, const void *bias_table,
                                          const float *logit_scale, const void *Wproj, const void *bproj, void *out,
                                          swin_stream_t stream)
{
    // the block parameters, as swin_wattn_create checks them
    if (C <= 0 || heads <= 0 || M <= 0 || C % heads) return SWIN_WATTN_EINVAL;
    if (shift < 0 || shift >= M) return SWIN_WATTN_EINVAL;
    if (mode & ~(SWIN_WATTN_V2 | SWIN_WATTN_FP32)) return SWIN_WATTN_EINVAL;
    if ((mode & SWIN_WATTN_FP32) || C / heads != 32 || M > 64) return SWIN_WATTN_EUNSUPPORTED;
    // the call's arguments, as swin_wattn_forward checks them
    if (!x || !Wqkv || !bias_table || !Wproj || !out) return SWIN_WATTN_EINVAL;
    if ((mode & SWIN_WATTN_V2) && !logit_scale) return SWIN_WATTN_EINVAL;
    if (B < 0 || H <= 0 || W <= 0 || H % M || W % M) return SWIN_WATTN_EINVAL;
    const void *ptrs[] = {x, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj, out};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SWIN_WATTN_EINVAL;
    const size_t io = (size_t)B * H * W * C * 2;
    if (io && (const char *)x < (const char *)out + io && (const char *)out < (const char *)x + io)
        return SWIN_WATTN_EINVAL;
    if (B == 0) return SWIN_WATTN_OK;
    // q/k/v (6 bytes per channel per token) and attention output (2 bytes)
    const Geom g = make_geom(B, H, W, C, M, shift);
    const size_t qkv_bytes = (size_t)g.T * 3 * C * 2, attn_bytes = (size_t)g.T * C * 2;
    static_assert(kStatusBytes + SWIN_WATTN_NOALLOC_MAX_INTERMEDIATE_BYTES == kScratchBytes, "scratch layout");
    if (qkv_bytes + attn_bytes > SWIN_WATTN_NOALLOC_MAX_INTERMEDIATE_BYTES) return SWIN_WATTN_ESCRATCH;

    void *base = nullptr;
    int rc = scratch_address(&base);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    int *err = reinterpret_cast<int *>(base);
    bf16 *qkv = reinterpret_cast<bf16 *>((char *)base + kStatusBytes);
    bf16 *attn = reinterpret_cast<bf16 *>((char *)base + kStatusBytes + qkv_bytes);
    // the status word keeps the previous call's value: clear it
    if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return SWIN_WATTN_ECUDA;
    const DeviceStatus st{err, 2000000000ull};

    GemmArgs k1{};
    k1.A = (const bf16 *)x; k1.lda = C; k1.Bw = (const bf16 *)Wqkv; k1.bias = (const bf16 *)bqkv;
    k1.D = qkv; k1.ldd = 3 * C; k1.rows = g.T; k1.N = 3 * C; k1.K = C; k1.g = g;
    k1.norm_cols = (mode & SWIN_WATTN_V2) ? 2 * C : 0;
    if (launch_gemm(k1, LOAD_GATHER, STORE_PLAIN, st, s) != cudaSuccess) return SWIN_WATTN_ECUDA;
    AttnArgs k2{};
    k2.qkv = qkv; k2.attn = attn; k2.table = (const bf16 *)bias_table; k2.tau = logit_scale; k2.heads = heads;
    k2.mode = mode & SWIN_WATTN_V2; k2.g = g;
    if (launch_attention(k2, st, s) != cudaSuccess) return SWIN_WATTN_ECUDA;
    GemmArgs k3{};
    k3.A = attn; k3.lda = C; k3.Bw = (const bf16 *)Wproj; k3.bias = (const bf16 *)bproj;
    k3.D = (bf16 *)out; k3.ldd = C; k3.rows = g.T; k3.N = C; k3.K = C; k3.g = g;
    if (launch_gemm(k3, LOAD_PLAIN, STORE_SCATTER, st, s) != cudaSuccess) return SWIN_WATTN_ECUDA;
    return SWIN_WATTN_OK;
}

extern "C" int swin_wattn_noalloc_sync_status(swin_stream_t stream)
{
    void *base = nullptr;
    int rc = scratch_address(&base);
    if (rc) return rc;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SWIN_WATTN_ECUDA;
    int err = 0;
    if (cudaMemcpy(&err, base, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SWIN_WATTN_ECUDA;
    if (err) {
        if (cudaMemset(base, 0, sizeof(int)) != cudaSuccess) return SWIN_WATTN_ECUDA;
        if (err & ERR_TIMEOUT) return SWIN_WATTN_ETIMEOUT;
    }
    return SWIN_WATTN_OK;
}

extern "C" int swin_wattn_test_noalloc_watchdog(int64_t wait_limit_us, swin_stream_t stream)
{
    if (wait_limit_us <= 0 || wait_limit_us > 60000000) return SWIN_WATTN_EINVAL;
    void *base = nullptr;
    int rc = scratch_address(&base);
    if (rc) return rc;
    const DeviceStatus st{reinterpret_cast<int *>(base), (uint64_t)wait_limit_us * 1000ull};
    return launch_watchdog(st, (cudaStream_t)stream) == cudaSuccess ? SWIN_WATTN_OK : SWIN_WATTN_ECUDA;
}
