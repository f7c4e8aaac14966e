// fa2_launch.cuh -- host-side launch of the forward kernel for one tile
// configuration: TMA descriptor encoding and the kernel launch.  Included by
// the per-head-dimension translation units so they compile in parallel.
#pragma once

#include <atomic>
#include <climits>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fa2.h"
#include "fa2_fwd_kernel.cuh"

namespace fa2 {

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

struct LaunchArgs {
    const void *q, *k, *v;
    void *o;
    float *lse;
    int B, H, Lq, Lk;
    int causal;
    float scale_log2;
    int *err;
    unsigned long long wait_limit_ns;
    cudaStream_t stream;
    EncodeTiledFn encode;
    int device;
    int num_sms;    // streaming multiprocessors of `device`
};

// 3-D view of a contiguous bf16 [B*H, L, D] tensor: dims (D, L, B*H) innermost
// first, a box of 64 columns (128 bytes, one swizzle span) by box_rows rows by
// one head.  Rows outside [0, L) of a head read as zero.
inline bool encode_bhld(EncodeTiledFn encode, CUtensorMap *m, const void *ptr, int D, int L, int BH,
                        int box_rows)
{
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                             static_cast<cuuint64_t>(L) * static_cast<cuuint64_t>(D) * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <class C>
fa2_status launch_fwd(const LaunchArgs &a)
{
    const int BH = a.B * a.H;
    CUtensorMap tq, tk, tv;
    if (!encode_bhld(a.encode, &tq, a.q, C::D, a.Lq, BH, C::BM) ||
        !encode_bhld(a.encode, &tk, a.k, C::D, a.Lk, BH, C::BN) ||
        !encode_bhld(a.encode, &tv, a.v, C::D, a.Lk, BH, C::BN))
        return FA2_ERR_CUDA;

    FwdParams p;
    p.o = static_cast<uint16_t *>(a.o);
    p.lse = a.lse;
    p.err = a.err;
    p.wait_limit_ns = a.wait_limit_ns;
    p.Lq = a.Lq;
    p.Lk = a.Lk;
    p.BH = BH;
    p.n_qgroups = (a.Lq + C::NQ * C::BM - 1) / (C::NQ * C::BM);
    p.causal = a.causal ? 1 : 0;
    p.scale_log2 = a.scale_log2;
    const long long units = static_cast<long long>(p.n_qgroups) * BH;
    if (units > INT_MAX)
        return FA2_ERR_INVALID_ARG;
    p.n_units = static_cast<int>(units);
    // persistent grid: one CTA per SM (each holds all of TMEM), walking the units
    const long long grid = units < a.num_sms ? units : a.num_sms;

    // opt in to more than 48 KB of dynamic shared memory, once per device
    static std::atomic<unsigned long long> configured{0};
    const unsigned long long bit = (a.device >= 0 && a.device < 64) ? (1ull << a.device) : 0ull;
    if (!bit || !(configured.load() & bit)) {
        if (cudaFuncSetAttribute(fa2_fwd_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_BYTES) != cudaSuccess) {
            (void)cudaGetLastError();
            return FA2_ERR_CUDA;
        }
        configured.fetch_or(bit);
    }
    fa2_fwd_kernel<C><<<static_cast<unsigned>(grid), C::NUM_THREADS, C::SMEM_BYTES, a.stream>>>(tq, tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

// One entry per head dimension (defined in fa2_fwd_d{64,128,256}.cu).
fa2_status launch_fwd_d64(const LaunchArgs &a);
fa2_status launch_fwd_d128(const LaunchArgs &a);
fa2_status launch_fwd_d256(const LaunchArgs &a);

}  // namespace fa2
