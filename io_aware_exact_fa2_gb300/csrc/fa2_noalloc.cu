// fa2_noalloc.cu -- the fixed scratch behind fa2_fwd_noalloc (include/fa2.h).
//
// Some callers may not allocate device memory: plug-ins hosted by a framework
// that owns all device memory through its own pool and budget, and
// latency-critical loops that rule out cudaMalloc / cudaFree because either can
// synchronise the device.  For them the split schedule's workspace comes from
// this file-scope buffer instead of the caller.  It is bounded by the schedule's
// grid (at most one CTA per SM), not by the problem: 40.5 MB at most (D = 128 or
// 256) on 152 SMs, against FA2_NOALLOC_SCRATCH_BYTES = 48 MiB.  The buffer sits in
// a translation unit of its own so that its CUDA module -- and the 48 MiB -- are
// only loaded on devices where fa2_fwd_noalloc is called (lazy module loading).
#include <mutex>

#include <cuda_runtime.h>

#include "fa2.h"

namespace fa2 {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA2_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch on `dev`, which must be the current device.
// Looked up once per device, the first call also loading the module that holds
// the buffer; returns nullptr if the lookup fails.
void *noalloc_scratch_ptr(int dev)
{
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static void *cache[kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < kMaxDevices && cache[dev])
        return cache[dev];
    unsigned char *ptr = nullptr;
    if (cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (dev >= 0 && dev < kMaxDevices)
        cache[dev] = ptr;
    return ptr;
}

}  // namespace fa2
