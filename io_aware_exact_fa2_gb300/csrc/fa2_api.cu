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

// Limit of the forward kernel's waits between its warps.  FA2_TEST_WAIT_LIMIT_NS
// (read on every call, nanoseconds) shortens it so that a test of the time-out path
// ends quickly; the waits with which a CTA drains its own copies and MMAs before
// exiting keep the full limit.
unsigned long long fwd_wait_limit_ns()
{
    const char *s = std::getenv("FA2_TEST_WAIT_LIMIT_NS");
    const long long ns = s ? std::atoll(s) : 0;
    return ns > 0 ? static_cast<unsigned long long>(ns) : wait_limit_ns();
}

// Tests of the time-out path: FA2_TEST_STALL=1 (read on every call) makes the forward
// kernel's softmax warps first wait on a barrier nothing completes, so that wait runs
// out, the waits of the other roles on those warps run out after it, and the call
// reports FA2_ERR_TIMEOUT.
int fwd_stall_test()
{
    const char *s = std::getenv("FA2_TEST_STALL");
    return s && std::strcmp(s, "1") == 0 ? 1 : 0;
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

// Streams and events with which fa2_fwd_from_host overlaps its host->device copies,
// kernels and device->host copies across chunks of heads: one stream per kind of
// work, so chunk c's kernel runs while chunk c+1's inputs arrive and chunk c-1's
// outputs leave.  One set per device, created on first use with the device current.
struct HostPipe {
    static constexpr int kChunks = 8;
    cudaStream_t h2d = nullptr, compute = nullptr, d2h = nullptr;
    cudaEvent_t entry = nullptr, exit = nullptr;
    cudaEvent_t inputs[kChunks] = {}, outputs[kChunks] = {};
    std::mutex mu;   // one call at a time enqueues (the events are shared)
    bool ok = false;
};

HostPipe *host_pipe(int dev)
{
    static std::mutex mu;
    static HostPipe *pipes[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!pipes[dev]) {
        HostPipe *hp = new HostPipe;
        bool ok = cudaStreamCreateWithFlags(&hp->h2d, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&hp->compute, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&hp->d2h, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&hp->entry, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&hp->exit, cudaEventDisableTiming) == cudaSuccess;
        for (int c = 0; ok && c < HostPipe::kChunks; ++c)
            ok = cudaEventCreateWithFlags(&hp->inputs[c], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&hp->outputs[c], cudaEventDisableTiming) == cudaSuccess;
        if (!ok)
            (void)cudaGetLastError();
        hp->ok = ok;
        pipes[dev] = hp;
    }
    return pipes[dev]->ok ? pipes[dev] : nullptr;
}

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
                  size_t workspace_bytes = 0, int window = -1, const BhlStrides *strides = nullptr,
                  const float *const *descales = nullptr)
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
    // Q, K, V, O: the caller's strides, or contiguous [B, H, L, D]
    a.sq = strides ? strides[0] : contiguous_bhl(H, Lq, D);
    a.sk = strides ? strides[1] : contiguous_bhl(H, Lk, D);
    a.sv = strides ? strides[2] : contiguous_bhl(H, Lk, D);
    a.so = strides ? strides[3] : contiguous_bhl(H, Lq, D);
    a.causal = causal;
    a.window = window;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
    a.err = device_error_ptr(dev);
    a.wait_limit_ns = fwd_wait_limit_ns();
    a.drain_limit_ns = wait_limit_ns();
    a.stall_test = fwd_stall_test();
    a.stream = stream;
    a.encode = encode_fn();
    a.device = dev;
    a.num_sms = sm_count(dev);
    a.split_policy = split_policy();
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    if (!a.err || !a.encode || a.num_sms <= 0)
        return FA2_ERR_CUDA;
    if (descales) {   // e4m3 inputs
        a.descale_q = descales[0];
        a.descale_k = descales[1];
        a.descale_v = descales[2];
        return D == 128 ? launch_fwd_fp8_d128(a) : FA2_ERR_UNSUPPORTED;
    }
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

FA2_EXPORT fa2_status fa2_fwd_fp8(const void *q, const void *k, const void *v, const float *descale_q,
                                  const float *descale_k, const float *descale_v, void *o, float *lse, int B, int H,
                                  int Lq, int Lk, int D, int causal, float scale, void *workspace,
                                  size_t workspace_bytes, void *stream)
{
    fa2_status st = fa2::validate(q, k, v, o, lse, B, H, Lq, Lk, D, scale);
    if (st != FA2_OK)
        return st;
    if (!descale_q || !descale_k || !descale_v || !fa2::aligned(descale_q, 4) || !fa2::aligned(descale_k, 4) ||
        !fa2::aligned(descale_v, 4))
        return FA2_ERR_INVALID_ARG;
    if (D != 128)
        return FA2_ERR_UNSUPPORTED;
    if (Lq == 0)
        return FA2_OK;
    if (workspace && !fa2::aligned(workspace, 256))
        return FA2_ERR_INVALID_ARG;
    const float *ds[3] = {descale_q, descale_k, descale_v};
    // the e4m3 configuration cuts and merges like the bf16 one at D = 128 (same query and
    // key tiles), so fa2_workspace_size(..., D = 128, ...) sizes its workspace
    return fa2::launch(q, k, v, o, lse, B, H, Lq, Lk, D, causal, scale, static_cast<cudaStream_t>(stream),
                       causal ? nullptr : workspace, causal ? 0 : workspace_bytes, -1, nullptr, ds);
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

FA2_EXPORT fa2_status fa2_bwd_workspace_size(int B, int H, int Lq, int Lk, int D, size_t *bytes)
{
    if (!bytes)
        return FA2_ERR_INVALID_ARG;
    *bytes = 0;
    if (B <= 0 || H <= 0 || Lq < 0 || Lk <= 0 || D <= 0 || static_cast<long long>(B) * H > INT_MAX)
        return FA2_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256)
        return FA2_ERR_UNSUPPORTED;
    *bytes = fa2::align256(fa2::bwd_stats_bytes(B, H, Lq));
    return FA2_OK;
}

namespace fa2 {
namespace {
// Zero the rows of a bf16 [B, H, L, D] view (rows of D contiguous) on `stream`.
bool zero_rows(void *ptr, int B, int H, int L, int D, const BhlStrides &st, cudaStream_t stream)
{
    const BhlStrides c = contiguous_bhl(H, L, D);
    if (st.b == c.b && st.h == c.h && st.l == c.l)
        return cudaMemsetAsync(ptr, 0, static_cast<size_t>(B) * H * L * D * 2, stream) == cudaSuccess;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            if (cudaMemset2DAsync(static_cast<uint16_t *>(ptr) + b * st.b + h * st.h, static_cast<size_t>(st.l) * 2,
                                  0, static_cast<size_t>(D) * 2, L, stream) != cudaSuccess)
                return false;
    return true;
}

// The backward pass; window >= 0 (causal only) restricts query i to keys i - window .. i.
// strides: NULL (everything contiguous) or 8 arrays of (batch, head, row) element strides,
// for q, k, v, o, dout, dq, dk, dv in that order, each NULL for a contiguous view.
fa2_status bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
               void *dq, void *dk, void *dv, int B, int H, int Lq, int Lk, int D, int causal, int window, float scale,
               void *workspace, size_t workspace_bytes, void *stream, const long long *const *strides = nullptr)
{
    // the forward's own checks cover q, k, v, o, lse, sizes and scale
    fa2_status st = fa2::validate(q, k, v, o, lse, B, H, Lq, Lk, D, scale);
    if (st != FA2_OK)
        return st;
    if (!dout || !dq || !dk || !dv || (!workspace && Lq > 0))
        return FA2_ERR_INVALID_ARG;
    if (!fa2::aligned(dout, 16) || !fa2::aligned(dq, 16) || !fa2::aligned(dk, 16) || !fa2::aligned(dv, 16) ||
        (workspace && !fa2::aligned(workspace, 16)))
        return FA2_ERR_INVALID_ARG;
    if (workspace_bytes < fa2::bwd_stats_bytes(B, H, Lq))
        return FA2_ERR_INVALID_ARG;
    // q, k, v, o, dout, dq, dk, dv
    BhlStrides sts[8] = {contiguous_bhl(H, Lq, D), contiguous_bhl(H, Lk, D), contiguous_bhl(H, Lk, D),
                         contiguous_bhl(H, Lq, D), contiguous_bhl(H, Lq, D), contiguous_bhl(H, Lq, D),
                         contiguous_bhl(H, Lk, D), contiguous_bhl(H, Lk, D)};
    for (int i = 0; strides && i < 8; ++i) {
        if (!strides[i])
            continue;
        // positive, and a multiple of 16 bytes (TMA strides; 16-byte row loads and stores)
        for (int d = 0; d < 3; ++d)
            if (strides[i][d] <= 0 || strides[i][d] % 8 != 0 || strides[i][d] > (1ll << 38))
                return FA2_ERR_INVALID_ARG;
        sts[i] = {strides[i][0], strides[i][1], strides[i][2]};
    }
    int dev = 0;
    if ((st = fa2::select_device_of(q, &dev)) != FA2_OK)
        return st;
    if (Lq == 0) {   // no queries: every key's gradients are zero
        if (!zero_rows(dk, B, H, Lk, D, sts[6], static_cast<cudaStream_t>(stream)) ||
            !zero_rows(dv, B, H, Lk, D, sts[7], static_cast<cudaStream_t>(stream))) {
            (void)cudaGetLastError();
            return FA2_ERR_CUDA;
        }
        return FA2_OK;
    }
    fa2::BwdArgs a;
    a.sq = sts[0];
    a.sk = sts[1];
    a.sv = sts[2];
    a.so = sts[3];
    a.sdo = sts[4];
    a.sdq = sts[5];
    a.sdk = sts[6];
    a.sdv = sts[7];
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.stats = static_cast<float *>(workspace);
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.B = B;
    a.H = H;
    a.Lq = Lq;
    a.Lk = Lk;
    a.D = D;
    a.causal = causal;
    a.window = window;
    a.scale = scale;
    a.err = fa2::device_error_ptr(dev);
    a.wait_limit_ns = fa2::wait_limit_ns();
    a.stream = static_cast<cudaStream_t>(stream);
    a.encode = fa2::encode_fn();
    a.device = dev;
    if (!a.err || !a.encode)
        return FA2_ERR_CUDA;
    return fa2::launch_bwd(a);
}
}  // namespace
}  // namespace fa2

FA2_EXPORT fa2_status fa2_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                              const void *dout, void *dq, void *dk, void *dv, int B, int H, int Lq, int Lk, int D,
                              int causal, float scale, void *workspace, size_t workspace_bytes, void *stream)
{
    return fa2::bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Lq, Lk, D, causal, -1, scale, workspace,
                    workspace_bytes, stream);
}

FA2_EXPORT fa2_status fa2_bwd_window(const void *q, const void *k, const void *v, const void *o, const float *lse,
                                     const void *dout, void *dq, void *dk, void *dv, int B, int H, int Lq, int Lk,
                                     int D, int window, float scale, void *workspace, size_t workspace_bytes,
                                     void *stream)
{
    if (window < 0 || Lq > Lk)
        return FA2_ERR_INVALID_ARG;
    return fa2::bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Lq, Lk, D, 1, window, scale, workspace,
                    workspace_bytes, stream);
}

FA2_EXPORT fa2_status fa2_bwd_ex(const void *q, const void *k, const void *v, const void *o, const float *lse,
                                 const void *dout, void *dq, void *dk, void *dv, int B, int H, int Lq, int Lk, int D,
                                 const long long *q_strides, const long long *k_strides, const long long *v_strides,
                                 const long long *o_strides, const long long *do_strides,
                                 const long long *dq_strides, const long long *dk_strides,
                                 const long long *dv_strides, int causal, int window, float scale, void *workspace,
                                 size_t workspace_bytes, void *stream)
{
    if (window < -1 || (window >= 0 && (!causal || Lq > Lk)))
        return FA2_ERR_INVALID_ARG;
    const long long *const strides[8] = {q_strides,  k_strides,  v_strides,  o_strides,
                                         do_strides, dq_strides, dk_strides, dv_strides};
    return fa2::bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Lq, Lk, D, causal, window, scale, workspace,
                    workspace_bytes, stream, strides);
}

FA2_EXPORT fa2_status fa2_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                                     int H, int Lq, int Lk, int D, int window, float scale, void *stream)
{
    fa2_status st = fa2::validate(q, k, v, o, lse, B, H, Lq, Lk, D, scale);
    if (st != FA2_OK || Lq == 0)
        return st;
    if (window < 0 || Lq > Lk)   // every row must keep its own key i
        return FA2_ERR_INVALID_ARG;
    return fa2::launch(q, k, v, o, lse, B, H, Lq, Lk, D, 1, scale, static_cast<cudaStream_t>(stream), nullptr, 0,
                       window);
}

FA2_EXPORT fa2_status fa2_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                                 int Lq, int Lk, int D, const long long *q_strides, const long long *k_strides,
                                 const long long *v_strides, const long long *o_strides, int causal, int window,
                                 float scale, void *workspace, size_t workspace_bytes, void *stream)
{
    fa2_status st = fa2::validate(q, k, v, o, lse, B, H, Lq, Lk, D, scale);
    if (st != FA2_OK)
        return st;
    if (window < -1 || (window >= 0 && (!causal || Lq > Lk)))
        return FA2_ERR_INVALID_ARG;
    if (workspace && !fa2::aligned(workspace, 256))
        return FA2_ERR_INVALID_ARG;
    fa2::BhlStrides sts[4] = {fa2::contiguous_bhl(H, Lq, D), fa2::contiguous_bhl(H, Lk, D),
                              fa2::contiguous_bhl(H, Lk, D), fa2::contiguous_bhl(H, Lq, D)};
    const long long *given[4] = {q_strides, k_strides, v_strides, o_strides};
    for (int i = 0; i < 4; ++i) {
        if (!given[i])
            continue;
        // positive, and a multiple of 16 bytes (TMA strides; 16-byte O row stores)
        for (int d = 0; d < 3; ++d)
            if (given[i][d] <= 0 || given[i][d] % 8 != 0 || given[i][d] > (1ll << 38))
                return FA2_ERR_INVALID_ARG;
        sts[i] = {given[i][0], given[i][1], given[i][2]};
    }
    if (Lq == 0)
        return FA2_OK;
    if (window >= 0 || causal)   // whole units; the workspace is not used
        return fa2::launch(q, k, v, o, lse, B, H, Lq, Lk, D, causal, scale, static_cast<cudaStream_t>(stream),
                           nullptr, 0, window, sts);
    return fa2::launch(q, k, v, o, lse, B, H, Lq, Lk, D, causal, scale, static_cast<cudaStream_t>(stream), workspace,
                       workspace_bytes, -1, sts);
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
    fa2::HostPipe *hp = fa2::host_pipe(dev);
    if (!hp)
        return FA2_ERR_CUDA;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int bh = B * H;   // validated: fits an int
    const size_t q_head = static_cast<size_t>(Lq) * D * 2, kv_head = static_cast<size_t>(Lk) * D * 2;
    const size_t lse_head = static_cast<size_t>(Lq) * sizeof(float);
    // chunks of whole heads, each moving at least ~4 MB in, so that copy set-up
    // costs stay small against the transfer
    const size_t in_bytes = static_cast<size_t>(bh) * (q_head + 2 * kv_head);
    int chunks = static_cast<int>(in_bytes / (size_t{4} << 20));
    chunks = chunks < 1 ? 1 : chunks > fa2::HostPipe::kChunks ? fa2::HostPipe::kChunks : chunks;
    chunks = chunks > bh ? bh : chunks;

    std::lock_guard<std::mutex> lock(hp->mu);
    auto fail = [] {
        (void)cudaGetLastError();
        return FA2_ERR_CUDA;
    };
    // everything below runs after the work already on `stream`
    if (cudaEventRecord(hp->entry, s) != cudaSuccess || cudaStreamWaitEvent(hp->h2d, hp->entry, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hp->compute, hp->entry, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hp->d2h, hp->entry, 0) != cudaSuccess)
        return fail();
    char *qd = static_cast<char *>(q_dev), *kd = static_cast<char *>(k_dev), *vd = static_cast<char *>(v_dev);
    char *od = static_cast<char *>(o_dev), *ld = reinterpret_cast<char *>(lse_dev);
    const char *qh = static_cast<const char *>(q_host), *kh = static_cast<const char *>(k_host);
    const char *vh = static_cast<const char *>(v_host);
    char *oh = static_cast<char *>(o_host), *lh = reinterpret_cast<char *>(lse_host);
    for (int c = 0; c < chunks; ++c) {
        const size_t h0 = static_cast<size_t>(bh) * c / chunks, h1 = static_cast<size_t>(bh) * (c + 1) / chunks;
        const size_t nh = h1 - h0;
        if (cudaMemcpyAsync(qd + h0 * q_head, qh + h0 * q_head, nh * q_head, cudaMemcpyHostToDevice, hp->h2d) !=
                cudaSuccess ||
            cudaMemcpyAsync(kd + h0 * kv_head, kh + h0 * kv_head, nh * kv_head, cudaMemcpyHostToDevice, hp->h2d) !=
                cudaSuccess ||
            cudaMemcpyAsync(vd + h0 * kv_head, vh + h0 * kv_head, nh * kv_head, cudaMemcpyHostToDevice, hp->h2d) !=
                cudaSuccess ||
            cudaEventRecord(hp->inputs[c], hp->h2d) != cudaSuccess ||
            cudaStreamWaitEvent(hp->compute, hp->inputs[c], 0) != cudaSuccess)
            return fail();
        st = fa2::launch(qd + h0 * q_head, kd + h0 * kv_head, vd + h0 * kv_head, od + h0 * q_head,
                         reinterpret_cast<float *>(ld + h0 * lse_head), 1, static_cast<int>(nh), Lq, Lk, D, causal,
                         scale, hp->compute);
        if (st != FA2_OK)
            return st;
        if (cudaEventRecord(hp->outputs[c], hp->compute) != cudaSuccess ||
            cudaStreamWaitEvent(hp->d2h, hp->outputs[c], 0) != cudaSuccess ||
            cudaMemcpyAsync(oh + h0 * q_head, od + h0 * q_head, nh * q_head, cudaMemcpyDeviceToHost, hp->d2h) !=
                cudaSuccess ||
            cudaMemcpyAsync(lh + h0 * lse_head, ld + h0 * lse_head, nh * lse_head, cudaMemcpyDeviceToHost,
                            hp->d2h) != cudaSuccess)
            return fail();
    }
    // `stream` continues once the last outputs are on the host (the d2h stream's
    // work follows every kernel, and every kernel follows its inputs)
    if (cudaEventRecord(hp->exit, hp->d2h) != cudaSuccess || cudaStreamWaitEvent(s, hp->exit, 0) != cudaSuccess)
        return fail();
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
