// fa2_launch.cuh -- host-side launch of the forward kernel for one tile
// configuration: TMA descriptor encoding and the kernel launch.  Included by
// the per-head-dimension translation units so they compile in parallel.
#pragma once

#include <atomic>
#include <climits>
#include <mutex>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fa2.h"
#include "fa2_fwd_kernel.cuh"
#include "fa2_split_ranges.h"

namespace fa2 {

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

// Element strides of a bf16 [B, H, L, D] view whose rows of D are contiguous.
struct BhlStrides {
    long long b, h, l;
};

inline BhlStrides contiguous_bhl(int H, int L, int D)
{
    return {static_cast<long long>(H) * L * D, static_cast<long long>(L) * D, D};
}

struct LaunchArgs {
    const void *q, *k, *v;
    void *o;
    float *lse;
    // e4m3 inputs only (fa2_fwd_fp8): fp32 [B*H] descales, real input = stored value x descale
    const float *descale_q = nullptr, *descale_k = nullptr, *descale_v = nullptr;
    int B, H, Lq, Lk;
    BhlStrides sq, sk, sv, so;   // element strides of Q, K, V, O
    int causal;
    int window;               // causal sliding window, -1: none
    float scale_log2;
    int *err;
    unsigned long long wait_limit_ns;    // waits between warps
    unsigned long long drain_limit_ns;   // a CTA's waits for its own copies and MMAs before exit
    int stall_test = 0;       // tests only: make the softmax warps' first wait run out
    cudaStream_t stream;
    EncodeTiledFn encode;
    int device;
    int num_sms;    // streaming multiprocessors of `device`
    int split_policy;         // SPLIT_NEVER / SPLIT_AUTO / SPLIT_ALWAYS
    void *workspace;          // optional (split schedule for non-causal passes)
    size_t workspace_bytes;
};

// Workspace of the split schedule for a launch of G CTAs: arrival counters,
// then per CTA two part slots of NQ x 128 rows: an LSE pair per row, and O in
// fp32 (stored by 4-column groups of 128 rows).
struct WorkspaceLayout {
    size_t counters, part_lse, part_o, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

inline WorkspaceLayout workspace_layout(long long G, int NQ, int D)
{
    WorkspaceLayout w;
    w.counters = 0;
    w.part_lse = align256(static_cast<size_t>(G) * NQ * sizeof(int));
    w.part_o = w.part_lse + align256(static_cast<size_t>(G) * 2 * NQ * 128 * 2 * sizeof(float));
    w.total = w.part_o + align256(static_cast<size_t>(G) * 2 * NQ * 128 * D * sizeof(float));
    return w;
}

enum SplitPolicy { SPLIT_NEVER = 0, SPLIT_AUTO = 1, SPLIT_ALWAYS = 2 };

// A cut of the non-causal iterations into cost-balanced ranges (cut_ranges).  The
// cut is a pure function of (units, n_kv, G) but costs a binary search over greedy
// passes -- tens of microseconds of host time -- so the last few are kept and
// repeated launches of one shape reuse theirs.
struct SplitPlan {
    long long units = -1, n_kv = -1;
    int G = 0;
    int k = 0;        // ranges
    long long T = 0;  // largest range cost
    int begin[MAX_SPLIT_CTAS + 1];
};

inline SplitPlan split_plan(long long units, long long n_kv, int G)
{
    constexpr int SLOTS = 4;
    static std::mutex mu;
    static SplitPlan cache[SLOTS];
    static int next = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const SplitPlan &c : cache)
            if (c.units == units && c.n_kv == n_kv && c.G == G)
                return c;
    }
    SplitPlan plan;
    plan.units = units;
    plan.n_kv = n_kv;
    plan.G = G;
    plan.k = cut_ranges(units, n_kv, G, plan.begin, &plan.T);
    std::lock_guard<std::mutex> lock(mu);
    cache[next] = plan;
    next = (next + 1) % SLOTS;
    return plan;
}

inline bool use_split(int policy, long long units, long long n_kv, int num_sms)
{
    if (units * n_kv > INT_MAX)
        return false;
    if (policy == SPLIT_ALWAYS)
        return true;
    if (policy != SPLIT_AUTO)
        return false;
    const SplitPlan plan = split_plan(units, n_kv, static_cast<int>(split_grid(units, n_kv, num_sms)));
    return split_pays_given(units, n_kv, num_sms, plan.T);
}

// Bytes of workspace the pass needs for its split schedule (0: none is used).
template <class C>
size_t workspace_bytes_for(int B, int H, int Lq, int Lk, int causal, int num_sms, int policy)
{
    if (causal || Lq <= 0)
        return 0;
    const long long BH = static_cast<long long>(B) * H;
    const long long units = ((Lq + C::NQ * C::BM - 1) / (C::NQ * C::BM)) * BH;
    const long long n_kv = (Lk + C::BN - 1) / C::BN;
    if (!use_split(policy, units, n_kv, num_sms))
        return 0;
    return workspace_layout(split_grid(units, n_kv, num_sms), C::NQ, C::D).total;
}

// 4-D view of a bf16 [B, H, L, D] tensor with contiguous rows of D and the given
// element strides: dims (D, L, H, B) innermost first, a box of box_cols columns (64:
// 128 bytes under the 128B swizzle; 32: 64 bytes under the 64B swizzle -- one swizzle
// span either way) by box_rows rows of one head.  Loads read rows outside [0, L) as
// zero; stores leave them unwritten.
inline bool encode_bhld_strided(EncodeTiledFn encode, CUtensorMap *m, const void *ptr, int D, int L, int H, int B,
                                BhlStrides st, int box_rows, int box_cols = 64, int elem_bytes = 2)
{
    // elem_bytes 1: e4m3 bytes (moved as raw bytes), the box then 128 elements wide
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.l) * elem_bytes, static_cast<cuuint64_t>(st.h) * elem_bytes,
                             static_cast<cuuint64_t>(st.b) * elem_bytes};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle sw = box_cols * elem_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = encode(m, dt, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

#ifndef FA2_FWD_GROUP_MB
#define FA2_FWD_GROUP_MB 96
#endif

template <class C>
fa2_status launch_fwd(const LaunchArgs &a)
{
    const int BH = a.B * a.H;
    CUtensorMap tq, tk, tv, to;
    // O is written by TMA stores of 32 rows x OBW columns (one softmax warp's rows)
    if (!encode_bhld_strided(a.encode, &tq, a.q, C::D, a.Lq, a.H, a.B, a.sq, C::BM, C::ECOLS, C::EB) ||
        !encode_bhld_strided(a.encode, &tk, a.k, C::D, a.Lk, a.H, a.B, a.sk, C::BN, C::ECOLS, C::EB) ||
        !encode_bhld_strided(a.encode, &tv, a.v, C::D, a.Lk, a.H, a.B, a.sv, C::BN, C::ECOLS, C::EB) ||
        !encode_bhld_strided(a.encode, &to, a.o, C::D, a.Lq, a.H, a.B, a.so, 32, C::OBW))
        return FA2_ERR_CUDA;

    FwdParams p;
    p.H = a.H;
    p.descale_q = a.descale_q;
    p.descale_k = a.descale_k;
    p.descale_v = a.descale_v;
    p.lse = a.lse;
    p.err = a.err;
    p.wait_limit_ns = a.wait_limit_ns;
    p.drain_limit_ns = a.drain_limit_ns;
    p.stall_test = a.stall_test;
    p.Lq = a.Lq;
    p.Lk = a.Lk;
    p.BH = BH;
    p.n_qgroups = (a.Lq + C::NQ * C::BM - 1) / (C::NQ * C::BM);
    p.causal = a.causal ? 1 : 0;
    // Causal passes whose K and V exceed FA2_FWD_GROUP_MB take the heads in that many
    // evenly sized groups (each group's K and V fit in L2 beside the other traffic):
    // all heads at once would stream every head's K/V prefixes in from DRAM again for
    // each of its heaviest-first units.
    p.head_group = BH;
    if (a.causal) {
        // K and V rows a head's units read: all of them, or under a sliding window the
        // band (window + a unit's rows + one K/V tile), the same for every unit
        long long rows = a.Lk;
        if (a.window >= 0 && a.window + static_cast<long long>(C::NQ * C::BM + C::BN) < rows)
            rows = a.window + static_cast<long long>(C::NQ * C::BM + C::BN);
        const long long per_head = 2ll * rows * C::D * C::EB;   // K and V bytes of one head
        const long long budget = static_cast<long long>(FA2_FWD_GROUP_MB) << 20;
        if (budget > 0 && per_head * BH > budget) {
            const long long groups = (per_head * BH + budget - 1) / budget;
            p.head_group = static_cast<int>((BH + groups - 1) / groups);
        }
    }
    p.window = a.window;
    p.unit_rows = C::NQ * C::BM;
    p.kv_rows = C::BN;
    p.scale_log2 = a.scale_log2;
    const long long units = static_cast<long long>(p.n_qgroups) * BH;
    if (units > INT_MAX)
        return FA2_ERR_INVALID_ARG;
    p.n_units = static_cast<int>(units);
    p.n_kv = (a.Lk + C::BN - 1) / C::BN;
    // persistent grid: one CTA per SM (each holds all of TMEM), walking the units;
    // non-causal passes with a workspace cut the tile iterations into equal ranges
    p.split = (!a.causal && a.workspace != nullptr && use_split(a.split_policy, units, p.n_kv, a.num_sms)) ? 1 : 0;
    long long grid = units < a.num_sms ? units : a.num_sms;
    SplitRanges ranges{};
    p.counters = nullptr;
    p.part_lse = nullptr;
    p.part_o = nullptr;
    if (p.split) {
        const SplitPlan plan = split_plan(units, p.n_kv, static_cast<int>(split_grid(units, p.n_kv, a.num_sms)));
        grid = plan.k;
        for (int c = 0; c <= plan.k; ++c)
            ranges.begin[c] = plan.begin[c];
        const WorkspaceLayout w = workspace_layout(grid, C::NQ, C::D);
        if (a.workspace_bytes < w.total)
            return FA2_ERR_INVALID_ARG;
        char *base = static_cast<char *>(a.workspace);
        p.counters = reinterpret_cast<int *>(base + w.counters);
        p.part_lse = reinterpret_cast<float *>(base + w.part_lse);
        p.part_o = reinterpret_cast<float *>(base + w.part_o);
    }

    // opt in to more than 48 KB of dynamic shared memory, once per device (both
    // instantiations: whole units in one snake, and causal head groups)
    static std::atomic<unsigned long long> configured{0};
    const unsigned long long bit = (a.device >= 0 && a.device < 64) ? (1ull << a.device) : 0ull;
    if (!bit || !(configured.load() & bit)) {
        if (cudaFuncSetAttribute(fa2_fwd_kernel<C, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fa2_fwd_kernel<C, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_BYTES) != cudaSuccess) {
            (void)cudaGetLastError();
            return FA2_ERR_CUDA;
        }
        configured.fetch_or(bit);
    }
    if (p.causal && p.head_group < BH)
        fa2_fwd_kernel<C, true><<<static_cast<unsigned>(grid), C::NUM_THREADS, C::SMEM_BYTES, a.stream>>>(
            tq, tk, tv, to, p, ranges);
    else
        fa2_fwd_kernel<C, false><<<static_cast<unsigned>(grid), C::NUM_THREADS, C::SMEM_BYTES, a.stream>>>(
            tq, tk, tv, to, p, ranges);
    return cudaGetLastError() == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

// Arguments of the backward pass (fa2_bwd.cu).
struct BwdArgs {
    const void *q, *k, *v, *o, *dout;
    const float *lse;
    float *stats;             // workspace: per-row statistics tiles (bwd_stats_bytes)
    void *dq, *dk, *dv;
    int B, H, Lq, Lk, D;
    int causal;
    int window;               // >= 0 (causal): query i sees keys i - window .. i; -1: none
    // element strides (batch, head, row) of every [B, H, L, D] view; rows of D contiguous
    BhlStrides sq, sk, sv, so, sdo, sdq, sdk, sdv;
    float scale;
    int *err;
    unsigned long long wait_limit_ns;
    cudaStream_t stream;
    EncodeTiledFn encode;
    int device;
};
fa2_status launch_bwd(const BwdArgs &a);
// Bytes of the backward's statistics tiles: two fp32 per query row, rows padded
// to a multiple of BWD_STAT_TILE_ROWS per head.
constexpr int BWD_STAT_TILE_ROWS = 64;
constexpr size_t bwd_stats_bytes(int B, int H, int Lq)
{
    return static_cast<size_t>(B) * H * ((static_cast<size_t>(Lq) + BWD_STAT_TILE_ROWS - 1) / BWD_STAT_TILE_ROWS) *
           BWD_STAT_TILE_ROWS * 2 * sizeof(float);
}

// One entry per head dimension (defined in fa2_fwd_d{64,128,256}.cu).
fa2_status launch_fwd_d64(const LaunchArgs &a);
fa2_status launch_fwd_d128(const LaunchArgs &a);
fa2_status launch_fwd_d256(const LaunchArgs &a);
fa2_status launch_fwd_fp8_d128(const LaunchArgs &a);   // e4m3 Q, K, V (fa2_fwd_fp8_d128.cu)
size_t workspace_bytes_d64(int B, int H, int Lq, int Lk, int causal, int num_sms, int policy);
size_t workspace_bytes_d128(int B, int H, int Lq, int Lk, int causal, int num_sms, int policy);
size_t workspace_bytes_d256(int B, int H, int Lq, int Lk, int causal, int num_sms, int policy);

}  // namespace fa2
