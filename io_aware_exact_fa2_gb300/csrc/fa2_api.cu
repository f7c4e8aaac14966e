// fa2_api.cu -- the C ABI declared in include/fa2.h: argument validation,
// device selection, the device error word, and dispatch by head dimension.
//
// The host-wrapper role follows Olowookere, "FlashAttention-2 from scratch
// with a custom Triton kernel", section "Host wrapper and kernel launch"
// (validate and read shapes, build the grid over query blocks x batch*head,
// launch; no attention logic here).  Unlike the page's wrapper this one
// allocates nothing: the caller owns O and LSE.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fa2_launch.cuh"

#define FA2_EXPORT extern "C" __attribute__((visibility("default")))

namespace fa2 {

// Written by a kernel when one of its bounded waits runs out (first code wins).
static __device__ int g_device_error;

// Device address of fa2_fwd_noalloc's fixed scratch on `dev` (fa2_noalloc.cu).
void *noalloc_scratch_ptr(int dev);

namespace {

constexpr int kMaxDevices = 64;
constexpr double kLog2e = 1.4426950408889634074;  // log2(e) = 1 / ln 2

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

unsigned long long wait_limit_ns()
{
    static unsigned long long limit = [] {
        const char *s = std::getenv("FA2_WAIT_LIMIT_MS");
        long long ms = s ? std::atoll(s) : 0;
        if (ms <= 0)
            ms = 1000;
        return static_cast<unsigned long long>(ms) * 1000000ull;
    }();
    return limit;
}

// Whether non-causal passes given a workspace cut their key-tile iterations
// into equal per-SM ranges: FA2_SPLIT=always / never overrides the cost model
// (read on every call, so a process can switch it between calls).
int split_policy()
{
    const char *s = std::getenv("FA2_SPLIT");
    if (s && std::strcmp(s, "always") == 0)
        return SPLIT_ALWAYS;
    if (s && std::strcmp(s, "never") == 0)
        return SPLIT_NEVER;
    return SPLIT_AUTO;
}

// Number of SMs of a device (looked up once per device).
int sm_count(int dev)
{
    static std::mutex mu;
    static int cache[kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < kMaxDevices && cache[dev] > 0)
        return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < kMaxDevices)
        cache[dev] = n;
    return n;
}

// Device address of g_device_error for the current device (looked up once per device).
int *device_error_ptr(int dev)
{
    static std::mutex mu;
    static int *cache[kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < kMaxDevices && cache[dev])
        return cache[dev];
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (dev >= 0 && dev < kMaxDevices)
        cache[dev] = static_cast<int *>(ptr);
    return static_cast<int *>(ptr);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Pure host-side checks (no CUDA call).
fa2_status validate(const void *q, const void *k, const void *v, const void *o, const float *lse, int B, int H,
                    int Lq, int Lk, int D, float scale)
{
    if (!q || !k || !v || !o || !lse)
        return FA2_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || Lq < 0 || Lk <= 0 || D <= 0)
        return FA2_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H > INT_MAX)
        return FA2_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f))
        return FA2_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
        return FA2_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256)
        return FA2_ERR_UNSUPPORTED;
    return FA2_OK;
}

// Make the device that owns `ptr` current for this library's runtime state.
fa2_status select_device_of(const void *ptr, int *dev_out)
{
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
        (void)cudaGetLastError();
        return FA2_ERR_CUDA;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return FA2_ERR_INVALID_ARG;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess)
        return FA2_ERR_CUDA;
    if (cur != attr.device && cudaSetDevice(attr.device) != cudaSuccess)
        return FA2_ERR_CUDA;
    *dev_out = attr.device;
    return FA2_OK;
}

fa2_status launch(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Lq,
                  int Lk, int D, int causal, float scale, cudaStream_t stream, void *workspace = nullptr,
                  size_t workspace_bytes = 0)
{
    int dev = 0;
    fa2_status st = select_device_of(q, &dev);
    if (st != FA2_OK)
        return st;
    LaunchArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.Lq = Lq;
    a.Lk = Lk;
    a.causal = causal;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
    a.err = device_error_ptr(dev);
    a.wait_limit_ns = wait_limit_ns();
    a.stream = stream;
    a.encode = encode_fn();
    a.device = dev;
    a.num_sms = sm_count(dev);
    a.split_policy = split_policy();
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    if (!a.err || !a.encode || a.num_sms <= 0)
        return FA2_ERR_CUDA;
    switch (D) {
    case 64: return launch_fwd_d64(a);
    case 128: return launch_fwd_d128(a);
    case 256: return launch_fwd_d256(a);
    default: return FA2_ERR_UNSUPPORTED;
    }
}

size_t workspace_bytes(int B, int H, int Lq, int Lk, int D, int causal, int num_sms)
{
    switch (D) {
    case 64: return workspace_bytes_d64(B, H, Lq, Lk, causal, num_sms, split_policy());
    case 128: return workspace_bytes_d128(B, H, Lq, Lk, causal, num_sms, split_policy());
    case 256: return workspace_bytes_d256(B, H, Lq, Lk, causal, num_sms, split_policy());
    default: return 0;
    }
}

}  // namespace
}  // namespace fa2

FA2_EXPORT fa2_status fa2_workspace_size(int B, int H, int Lq, int Lk, int D, int causal, int device,
                                         size_t *bytes)
{
    if (!bytes)
        return FA2_ERR_INVALID_ARG;
    *bytes = 0;
    if (B <= 0 || H <= 0 || Lq < 0 || Lk <= 0 || D <= 0 || device < 0)
        return FA2_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H > INT_MAX)
        return FA2_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256)
        return FA2_ERR_UNSUPPORTED;
    if (causal || Lq == 0)
        return FA2_OK;
    const int sms = fa2::sm_count(device);
    if (sms <= 0)
        return FA2_ERR_CUDA;
    *bytes = fa2::workspace_bytes(B, H, Lq, Lk, D, causal, sms);
    return FA2_OK;
}

FA2_EXPORT fa2_status fa2_fwd_ws(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                                 int Lq, int Lk, int D, int causal, float scale, void *workspace,
                                 size_t workspace_bytes, void *stream)
{
    fa2_status st = fa2::validate(q, k, v, o, lse, B, H, Lq, Lk, D, scale);
    if (st != FA2_OK || Lq == 0)
        return st;
    if (causal)   // the causal pass balances whole units and needs no workspace
        return fa2::launch(q, k, v, o, lse, B, H, Lq, Lk, D, causal, scale, static_cast<cudaStream_t>(stream));
    if (workspace && !fa2::aligned(workspace, 256))
        return FA2_ERR_INVALID_ARG;
    return fa2::launch(q, k, v, o, lse, B, H, Lq, Lk, D, causal, scale, static_cast<cudaStream_t>(stream),
                       workspace, workspace_bytes);
}

FA2_EXPORT fa2_status fa2_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                                      int H, int Lq, int Lk, int D, int causal, float scale, void *stream)
{
    fa2_status st = fa2::validate(q, k, v, o, lse, B, H, Lq, Lk, D, scale);
    if (st != FA2_OK || Lq == 0)
        return st;
    int dev = 0;
    if ((st = fa2::select_device_of(q, &dev)) != FA2_OK)
        return st;
    const int sms = fa2::sm_count(dev);
    if (sms <= 0)
        return FA2_ERR_CUDA;
    const size_t need = fa2::workspace_bytes(B, H, Lq, Lk, D, causal, sms);
    if (need > FA2_NOALLOC_SCRATCH_BYTES)
        return FA2_ERR_UNSUPPORTED;   // more workspace than the fixed scratch holds
    void *scratch = nullptr;
    if (need > 0) {
        scratch = fa2::noalloc_scratch_ptr(dev);
        if (!scratch)
            return FA2_ERR_CUDA;
        // the arrival counters (one int per CTA and Q tile, at most 2 Q tiles) start at zero
        const size_t zero_bytes = fa2::align256(static_cast<size_t>(sms) * 2 * sizeof(int));
        if (cudaMemsetAsync(scratch, 0, zero_bytes < need ? zero_bytes : need, static_cast<cudaStream_t>(stream)) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return FA2_ERR_CUDA;
        }
    }
    return fa2_fwd_ws(q, k, v, o, lse, B, H, Lq, Lk, D, causal, scale, scratch, FA2_NOALLOC_SCRATCH_BYTES,
                      stream);
}

FA2_EXPORT fa2_status fa2_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                              int Lq, int Lk, int D, int causal, float scale, void *stream)
{
    fa2_status st = fa2::validate(q, k, v, o, lse, B, H, Lq, Lk, D, scale);
    if (st != FA2_OK || Lq == 0)
        return st;
    return fa2::launch(q, k, v, o, lse, B, H, Lq, Lk, D, causal, scale, static_cast<cudaStream_t>(stream));
}

FA2_EXPORT fa2_status fa2_fwd_from_host(const void *q_host, const void *k_host, const void *v_host,
                                        void *o_host, float *lse_host, void *q_dev, void *k_dev, void *v_dev,
                                        void *o_dev, float *lse_dev, int B, int H, int Lq, int Lk, int D,
                                        int causal, float scale, void *stream)
{
    if (!q_host || !k_host || !v_host || !o_host || !lse_host)
        return FA2_ERR_INVALID_ARG;
    fa2_status st = fa2::validate(q_dev, k_dev, v_dev, o_dev, lse_dev, B, H, Lq, Lk, D, scale);
    if (st != FA2_OK || Lq == 0)
        return st;
    int dev = 0;
    st = fa2::select_device_of(q_dev, &dev);
    if (st != FA2_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bh = static_cast<size_t>(B) * static_cast<size_t>(H);
    const size_t q_bytes = bh * static_cast<size_t>(Lq) * D * 2;
    const size_t kv_bytes = bh * static_cast<size_t>(Lk) * D * 2;
    const size_t lse_bytes = bh * static_cast<size_t>(Lq) * sizeof(float);
    if (cudaMemcpyAsync(q_dev, q_host, q_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(k_dev, k_host, kv_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(v_dev, v_host, kv_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return FA2_ERR_CUDA;
    }
    st = fa2::launch(q_dev, k_dev, v_dev, o_dev, lse_dev, B, H, Lq, Lk, D, causal, scale, s);
    if (st != FA2_OK)
        return st;
    if (cudaMemcpyAsync(o_host, o_dev, q_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(lse_host, lse_dev, lse_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return FA2_ERR_CUDA;
    }
    return FA2_OK;
}

FA2_EXPORT fa2_status fa2_get_device_error(void *stream, int *detail)
{
    if (detail)
        *detail = 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        (void)cudaGetLastError();
        return FA2_ERR_CUDA;
    }
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, fa2::g_device_error, sizeof v) != cudaSuccess) {
        (void)cudaGetLastError();
        return FA2_ERR_CUDA;
    }
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(fa2::g_device_error, &zero, sizeof zero) != cudaSuccess) {
            (void)cudaGetLastError();
            return FA2_ERR_CUDA;
        }
    }
    if (detail)
        *detail = v;
    return v ? FA2_ERR_TIMEOUT : FA2_OK;
}

FA2_EXPORT const char *fa2_status_string(fa2_status status)
{
    switch (status) {
    case FA2_OK: return "FA2_OK";
    case FA2_ERR_INVALID_ARG: return "FA2_ERR_INVALID_ARG";
    case FA2_ERR_UNSUPPORTED: return "FA2_ERR_UNSUPPORTED";
    case FA2_ERR_CUDA: return "FA2_ERR_CUDA";
    case FA2_ERR_TIMEOUT: return "FA2_ERR_TIMEOUT";
    }
    return "FA2_ERR_UNKNOWN";
}

FA2_EXPORT int fa2_version(void) { return 100; }
