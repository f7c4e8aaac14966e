// fa2_fwd_kernel.cuh -- exact FlashAttention-2 forward for sm_103a.
//
// The method (Olowookere, "FlashAttention-2 from scratch with a custom Triton
// kernel", sections "The core idea: making attention IO-aware" and "Running
// max m_i and running normaliser"; "Chapter 08: Flash Attention -- blocked
// attention", sections 1-5): a work unit is NQ query tiles of 128 rows of one
// (batch, head); the tiles stay on chip while K/V tiles of BN rows stream
// through shared memory; per row the kernel keeps a running max m, a running
// normaliser l and an unnormalised accumulator O, rescales O and l when m
// grows, and divides by l once at the end (deferred normalisation).  Scores
// are taken to base 2 (scale * log2 e folded into one FMA, then exp2), the
// log-sum-exp is written per row, causal key tiles above the diagonal are
// never visited and only tiles that straddle the diagonal (or the key tail)
// pay for element masking.
//
// GB300 mapping (the pages' kernels are Triton for A100/Ada; this is not a
// translation of them):
//   * Persistent CTAs (one per SM) walk a static list of work units; causal
//     units are ordered heaviest first and dealt out in a snake so heavy and
//     light units pair up.  All barrier phases run on across units, so the next
//     unit's Q and K/V tiles stream in while the current unit finishes.
//     Non-causal passes given a workspace may instead cut the K/V-tile
//     iterations of all units into one cost-balanced range per CTA (ranges
//     planned on the host); a unit cut between CTAs is computed in parts that
//     the last part to finish merges exactly (the online-softmax merge of two
//     key blocks).  A causal sliding window starts each unit at the first K/V
//     tile of its band.
//   * Optionally (QT, one Q tile per unit) the softmax warps copy each Q tile
//     from shared memory into TMEM, so S = Q K^T reads A from TMEM.
//   * TMA (cp.async.bulk.tensor, 128B swizzle) moves Q (per unit) and K/V (per
//     tile) into shared memory: a Q buffer per Q tile, refilled as soon as the
//     last S MMA that reads it completes, and a KS-stage K/V ring.
//   * One warp issues tcgen05.mma (a single elected lane, warp-uniform control
//     flow, descriptors precomputed): S = Q K^T into TMEM (fp32), then
//     O += P V with P read straight from TMEM (bf16, aliasing S) and V from
//     shared memory as an MN-major operand (no transpose pass).
//   * Softmax: CS warps share each row (TMEM lane == row; warp w may touch
//     lanes 32*(w%4)..+31), each owning BN/CS columns of S and D/CS columns
//     of O.  They write P back to TMEM and rescale O in TMEM only when a
//     row's max grows by more than 2^8 (the stale max is kept otherwise, which
//     is exact because l and LSE use the same max).
//   * Epilogue: the softmax warps read O out of TMEM, release it to the MMA
//     warp (the next unit's PV may then overwrite it), multiply by 1/l, stage
//     bf16 boxes of 32 rows x 32 columns in two alternating halves of a per-warp
//     shared-memory buffer and write each with one TMA store; the fp32 LSE goes
//     straight out.
//   * Every wait between warps is on an mbarrier with a time bound; a wait
//     that runs out records a code in a device error word and the CTA winds
//     down, so no input can hang the GPU.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda.h>

#include "fa2_split_ranges.h"
#include "sm103_ptx.cuh"

namespace fa2 {

struct FwdParams {
    float *lse;                 // fp32 [B*H, Lq] (O is written through its tensor map)
    // e4m3 inputs only: fp32 [B*H] descales of Q, K and V (real input = stored value x descale)
    const float *descale_q, *descale_k, *descale_v;
    int H;                      // heads (Q/K/V tensor maps are (D, L, H, B))
    int *err;                   // device error word
    unsigned long long wait_limit_ns;    // bound of every wait between warps
    int stall_test;             // tests only: the softmax warps first wait on a barrier nobody completes
    unsigned long long drain_limit_ns;   // bound of a CTA's waits for its own copies / MMAs before exit
    int Lq, Lk;
    int BH;                     // B * H
    int n_qgroups;              // ceil(Lq / (NQ * 128))
    int n_units;                // n_qgroups * BH
    // causal: heads per group (BH: one group).  The heads are taken in groups whose K
    // and V fit in L2 together, each group's units heaviest first and dealt out in a
    // snake of its own, so that the units in flight re-read K/V prefixes from L2.
    int head_group;
    int causal;
    // causal sliding window: query i sees keys i - window <= j <= i (-1: none)
    int window;
    int unit_rows;              // NQ * 128 query rows per work unit
    int kv_rows;                // BN rows per K/V tile
    float scale_log2;           // scale * log2(e), > 0
    // split schedule (non-causal, with a workspace): the n_units * n_kv K/V-tile
    // iterations are cut into gridDim.x contiguous ranges, one per CTA, of equal cost
    // (tiles plus a fixed cost per unit or part of a unit the range touches)
    int split;                  // 0: whole units (unit_at), 1: cost-balanced tile ranges
    int n_kv;                   // K/V tiles per unit (non-causal: ceil(Lk / BN))
    int *counters;              // [gridDim.x][NQ] arrivals per cut unit (zero at rest)
    float *part_lse;            // [gridDim.x][2][NQ][128][2] base-2 LSE of each part
    float *part_o;              // [gridDim.x][2][NQ][D/4][128] float4: each part's normalised O,
                                // column groups outermost so a warp's 32 rows are contiguous
};

// Ranges of the split schedule: CTA k works on iterations [begin[k], begin[k + 1]).
// A kernel parameter of its own (grid-constant, indexed in place), so the other
// parameters keep their register-resident layout.
struct SplitRanges {
    int begin[MAX_SPLIT_CTAS + 1];
};

// Device error codes: role in the high byte, barrier in the low byte.
enum : int {
    ERR_PRODUCER = 0x100,
    ERR_MMA = 0x200,
    ERR_SOFTMAX = 0x300,
    ERR_DRAIN = 0x400,
};

// Threshold (log2 units) above which a growing row max forces a rescale of O and l.
constexpr float RESCALE_THRESHOLD = 8.0f;
constexpr float LN2 = 0.69314718055994530942f;

template <int D_, int BN_, int NQ_, int KS_, int CS_, int NS_ = (NQ_ == 1 ? 2 : 1), int QT_ = 0, int P2_ = 0,
          int F8_ = 0>
struct FwdCfg {
    static constexpr int D = D_;     // head dimension
    static constexpr int BN = BN_;   // K/V rows per tile
    static constexpr int NQ = NQ_;   // 128-row Q tiles per work unit
    static constexpr int KS = KS_;   // K/V ring stages
    static constexpr int CS = CS_;   // softmax warps sharing one row (column split)
    static constexpr int BM = 128;   // Q rows per tile = TMEM lanes = MMA M
    static constexpr int NS = NS_;                // S/P TMEM buffers per Q tile
    // QT: Q lives in TMEM and S = Q K^T takes A from TMEM; the softmax warps copy each
    // Q tile there from shared memory.  Needs one Q tile per unit (TMEM budget).
    static constexpr bool QT = QT_ != 0;
    // P2: P goes to the PV MMA as two bf16 terms, p_hi = bf16(p) and the residual
    // p_lo = bf16(p - p_hi), over the two halves of the S buffer; O then weighs V
    // with p to about 2^-17 of itself (one bf16 term rounds each weight by up to
    // 2^-9), at the price of a second PV MMA per key tile.
    static constexpr bool P2 = P2_ != 0;
    // F8: Q, K, V and P are e4m3 bytes and both products run as kind::f8f6f4 MMAs (K
    // steps of 32 elements); the real inputs are the stored values times per-(batch,
    // head) descales, folded into the score scale (Q, K) and into O's 1/l (V)
    static constexpr bool F8 = F8_ != 0;
    static constexpr int EB = F8 ? 1 : 2;             // bytes per Q/K/V element
    static constexpr int ECOLS = 128 / EB;             // elements per 128-byte swizzle span
    static constexpr int KSTEP = 32 / EB;              // elements per MMA K step (32 bytes)
    // NP: P is handed to the MMA warp in NP key parts, so PV on the earlier parts
    // runs while the softmax computes the later ones (one warp per row only: with a
    // column split, a slice's parts are not contiguous key ranges)
#ifndef FA2_P_PARTS
#define FA2_P_PARTS 2
#endif
    static constexpr int NP = CS_ == 1 ? FA2_P_PARTS : 1;
    static_assert(NP == 1 || NP == 2 || NP == 4, "P goes over in 1, 2 or 4 parts");
    static constexpr int NCOL = BN / CS;          // S columns per softmax thread
    static constexpr int OCOL = D / CS;           // O columns per softmax thread
    static constexpr int DB = D / ECOLS;          // 128-byte swizzle blocks per row
    static constexpr int S_KSTEPS = D / KSTEP;    // K steps of S = Q K^T
    static constexpr int PV_KSTEPS = BN / KSTEP;  // K steps of O += P V
    static constexpr int PV_KSTEP_BYTES = KSTEP * 128;   // V rows of one K step (MN-major operand)
    static constexpr int PW = NCOL * EB / 4;      // 32-bit TMEM columns of one thread's slice of P
    static constexpr int Q_BLOCK = BM * 128;
    static constexpr int KV_BLOCK = BN * 128;
    static constexpr int Q_TILE = DB * Q_BLOCK;
    static constexpr int KV_TILE = DB * KV_BLOCK;

    // shared memory (offsets from a 1024-byte aligned base)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + NQ * Q_TILE;
    static constexpr int OFF_V = OFF_K + KS * KV_TILE;
    // O staging of the epilogue: each softmax warp has two halves, each the
    // shared-memory side of one TMA store box of its 32 rows x OBW = 32 columns of bf16
    // (64-byte rows, 64B-swizzled); consecutive boxes alternate halves, so a warp
    // fills one while the store of the other is still reading it
    static constexpr int OBW = 32;
    static constexpr int O_HALF = 32 * OBW * 2;
    static constexpr int O_STAGE = 2 * O_HALF;
    static constexpr int OFF_OST = OFF_V + KS * KV_TILE;                // [softmax warps] (1024-aligned)
    static constexpr int OFF_XMAX = OFF_OST + 4 * CS * NQ * O_STAGE;   // f32 [NQ][2][CS][128] (CS > 1)
    static constexpr int OFF_XL = OFF_XMAX + (CS > 1 ? NQ * 2 * CS * 128 * 4 : 0);  // f32x2 [NQ][CS][128] (CS > 1)
    static constexpr int OFF_FLAG = OFF_XL + (CS > 1 ? NQ * CS * 128 * 8 : 0);       // u32 [NQ] (+ pad)
    static constexpr int OFF_BAR = OFF_FLAG + 16;
    static constexpr int BAR_Q_FULL = 0;                     // [NQ]
    static constexpr int BAR_Q_EMPTY = BAR_Q_FULL + NQ;      // [NQ]
    static constexpr int BAR_K_FULL = BAR_Q_EMPTY + NQ;      // [KS]
    static constexpr int BAR_K_EMPTY = BAR_K_FULL + KS;
    static constexpr int BAR_V_FULL = BAR_K_EMPTY + KS;
    static constexpr int BAR_V_EMPTY = BAR_V_FULL + KS;
    static constexpr int BAR_S_FULL = BAR_V_EMPTY + KS;      // [NQ][NS]
    static constexpr int BAR_P_READY = BAR_S_FULL + NQ * NS; // [NQ][NS]
    static constexpr int BAR_O_DONE = BAR_P_READY + NQ * NS; // [NQ]
    static constexpr int BAR_O_FREE = BAR_O_DONE + NQ;       // [NQ]
    static constexpr int BAR_XMAX = BAR_O_FREE + NQ;         // [NQ][2]
    static constexpr int BAR_GROUP = BAR_XMAX + 2 * NQ;      // [NQ]
    static constexpr int BAR_DRAIN = BAR_GROUP + NQ;
    static constexpr int BAR_QT_FULL = BAR_DRAIN + 1;        // [2] Q copied into TMEM buffer
    static constexpr int BAR_QT_EMPTY = BAR_QT_FULL + 2;     // [2] last S MMA read the buffer
    static constexpr int BAR_PA_READY = BAR_QT_EMPTY + 2;    // [NQ][NS][NP-1] earlier key parts of P written
    static constexpr int BAR_NEVER = BAR_PA_READY + NQ * NS * (NP > 1 ? NP - 1 : 1);   // nothing arrives (tests)
    static constexpr int NUM_BARS = BAR_NEVER + 1;
    static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_TMEM_SLOT + 16 + 1024;  // + slack for base alignment

    // tensor memory columns
    static constexpr int TM_O = 0;        // O of tile t: columns [t*D, (t+1)*D)
    static constexpr int TM_S = NQ * D;   // S/P buffer (t, b): TM_S + (t*NS + b)*BN
    static constexpr int TM_Q = NQ * D + NQ * NS * BN;   // QT: Q buffer q at TM_Q + q*D/2
    // Q buffers in TMEM: two where they fit (segments alternate), else one, which the
    // next segment's copy reuses once the current segment's last S has read it
    static constexpr int QB = (TM_Q + D <= 512) ? 2 : 1;
    static constexpr int TMEM_USED = TM_Q + (QT ? QB * D / 2 : 0);
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64
                                   : TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;

    // warp roles: softmax warpgroups first, then a control warpgroup (TMA
    // producer warp, MMA warp and, when registers are re-split, two idle warps)
    static constexpr int GROUP_THREADS = 128 * CS;             // softmax threads per Q tile
    // Barriers the softmax warps signal take one arrival per warp (after a __syncwarp),
    // not one per thread: 32x fewer shared-memory atomics on every step's P_READY.
    static constexpr int GROUP_WARPS = GROUP_THREADS / 32;
    static constexpr int NUM_SOFTMAX_WARPS = 4 * CS * NQ;
    static constexpr int WARP_PRODUCER = NUM_SOFTMAX_WARPS;
    static constexpr int WARP_MMA = NUM_SOFTMAX_WARPS + 1;
    // With two softmax warpgroups the launch leaves 168 registers per thread; the
    // control warpgroup drops to REG_CTRL and the softmax warpgroups rise to
    // REG_SOFTMAX.  Budget: 2*128*200 + 128*104 = 64512 = 384 threads * 168.
    static constexpr bool REG_SPLIT = (NUM_SOFTMAX_WARPS == 8);
    static constexpr int REG_SOFTMAX = 200;
    static constexpr int REG_CTRL = 104;
    static constexpr int NUM_THREADS = 32 * (NUM_SOFTMAX_WARPS + (REG_SPLIT ? 4 : 2));
    static_assert(!REG_SPLIT || 2 * 128 * REG_SOFTMAX + 128 * REG_CTRL <= NUM_THREADS * 168,
                  "register split exceeds the launch allocation");

    static constexpr uint32_t IDESC_S =
        F8 ? ptx::idesc_e4m3_f32(BM, BN, false, false) : ptx::idesc_bf16_f32(BM, BN, false, false);
    static constexpr uint32_t IDESC_PV =
        F8 ? ptx::idesc_e4m3_f32(BM, D, false, true) : ptx::idesc_bf16_f32(BM, D, false, true);

    static_assert(D % 64 == 0 && D >= 64 && D <= 256, "D must be 64, 128 or 256");
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be a multiple of 64 in [64, 256]");
    static_assert(NQ == 1 || NQ == 2, "one or two Q tiles per work unit");
    static_assert(CS == 1 || CS == 2, "one or two warps per row");
    static_assert(NS == 1 || NS == 2, "one or two S buffers per Q tile");
    static_assert(NCOL % 32 == 0 && OCOL % 32 == 0, "per-thread column slices are whole 32-column loads");
    static_assert(TMEM_USED <= 512, "TMEM budget exceeded");
    static_assert(!QT || NQ == 1, "Q in TMEM needs one Q tile per unit");
    static_assert(!QT || (D / CS) % 64 == 0, "Q copy works on whole 64-column swizzle blocks");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
    static_assert(OFF_OST % 1024 == 0 && O_HALF % 512 == 0,
                  "a 64B-swizzled TMA box needs a 512-byte aligned shared-memory side");
    static_assert((D / CS) % OBW == 0, "a warp's O columns are whole store boxes");
    static_assert(!P2 || CS == 1, "two-term P keeps a row's residuals beside its own weights (one warp per row)");
    static_assert(!F8 || (!QT && !P2 && CS == 1 && D % 128 == 0), "e4m3 path: Q in shared memory, one-term P, "
                                                                   "one warp per row, whole 128-byte rows");
    static_assert(NCOL % (4 * NP) == 0, "P parts are whole 32-bit TMEM columns");
};

// Number of K/V tiles a 128-row Q tile starting at q0 visits (0 if the tile is empty).
// Causal: only keys j <= last row of the tile, so tiles above the diagonal are skipped.
__device__ __forceinline__ int kv_tiles_for(int q0, int Lq, int Lk, int causal, int BN)
{
    if (q0 >= Lq)
        return 0;
    if (!causal)
        return (Lk + BN - 1) / BN;
    const int last_row = min(q0 + 127, Lq - 1);
    const int last_key = min(last_row, Lk - 1);
    return last_key / BN + 1;
}

// The work unit a CTA handles at its i-th step, or -1 when it has no more.
// Units are numbered heaviest first for causal (query groups from the bottom
// of the score matrix up) and dealt to the CTAs in a snake, so a CTA that got
// a heavy unit in one round gets a light one in the next.  GRP (causal passes whose
// heads are taken in groups, head_group < BH): the units are numbered group of heads
// by group of heads, and each group starts its snake at the first CTA again (the
// direction alternating on from the previous group's last round), so every group is
// balanced on its own.  GRP is a separate instantiation: the grouped form's loop,
// inlined where it is never used, cost the other passes' step loops.
template <bool GRP>
__device__ __forceinline__ int unit_at(int i, const FwdParams &p)
{
    const int g = static_cast<int>(gridDim.x);
    const int k = static_cast<int>(blockIdx.x);
    if constexpr (GRP) {
        int base = 0, rounds = 0;
        for (int g0 = 0; g0 < p.BH; g0 += p.head_group) {
            const int n = min(p.head_group, p.BH - g0) * p.n_qgroups;   // this group's units
            const int full = n / g, rem = n % g;
            // the partial last round reaches this CTA only if its snake position is below rem
            const int pos_last = ((rounds + full) & 1) ? g - 1 - k : k;
            const int mine = full + (rem > 0 && pos_last < rem ? 1 : 0);
            if (i < mine)
                return base + i * g + (((rounds + i) & 1) ? g - 1 - k : k);
            i -= mine;
            base += n;
            rounds += full + (rem > 0 ? 1 : 0);
        }
        return -1;
    } else {
        const int idx = i * g + ((p.causal && (i & 1)) ? (g - 1 - k) : k);
        return idx < p.n_units ? idx : -1;
    }
}

// unit -> (query group, batch*head)
template <bool GRP>
__device__ __forceinline__ void decode_unit(int idx, const FwdParams &p, int &qg, int &bh)
{
    if constexpr (GRP) {
        const int per_group = p.head_group * p.n_qgroups;
        const int gi = idx / per_group, r = idx - gi * per_group;
        const int g0 = gi * p.head_group, gsize = min(p.head_group, p.BH - g0);
        qg = p.n_qgroups - 1 - r / gsize;
        bh = g0 + r % gsize;
    } else if (p.causal) {
        qg = p.n_qgroups - 1 - idx / p.BH;
        bh = idx % p.BH;
    } else {
        bh = idx / p.n_qgroups;
        qg = idx % p.n_qgroups;
    }
}

// A stretch of work of one CTA: the K/V tiles [kv_lo, kv_hi) of a work unit.
// Without the split schedule a segment is a whole unit (kv_hi is then taken
// per Q tile from kv_tiles_for).  With it, a unit whose tiles straddle a CTA
// boundary is cut: CTAs c_first..c_last each compute a part, and the last one
// to finish combines them.
struct Segment {
    int unit;
    int kv_lo, kv_hi;
    int slot;              // this CTA's partial-result slot for the segment (0: first, 1: last)
    int c_first, c_last;   // CTAs sharing the unit (equal for a whole unit)
};

// CTA whose tile range holds iteration x: the largest k with range_begin[k] <= x.
__device__ __forceinline__ int cta_of(int x, const SplitRanges &r)
{
    int lo = 0, hi = static_cast<int>(gridDim.x) - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (r.begin[mid] <= x)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

template <bool GRP>
__device__ __forceinline__ bool segment_at(int i, const FwdParams &p, const SplitRanges &r, Segment &sg)
{
    if (!p.split) {
        const int u = unit_at<GRP>(i, p);
        if (u < 0)
            return false;
        sg.unit = u;
        sg.kv_lo = 0;
        if (p.window >= 0) {   // the unit's first K/V tile holding a key its first row may see
            int qg, bh;
            decode_unit<GRP>(u, p, qg, bh);
            sg.kv_lo = max(0, qg * p.unit_rows - p.window) / p.kv_rows;
        }
        sg.kv_hi = 0x7fffffff;
        sg.slot = 0;
        sg.c_first = sg.c_last = static_cast<int>(blockIdx.x);
        return true;
    }
    const int b = r.begin[blockIdx.x], e = r.begin[blockIdx.x + 1];
    const int u = b / p.n_kv + i;
    if (u * p.n_kv >= e)
        return false;
    sg.unit = u;
    sg.kv_lo = b > u * p.n_kv ? b - u * p.n_kv : 0;
    sg.kv_hi = e < (u + 1) * p.n_kv ? e - u * p.n_kv : p.n_kv;
    sg.slot = i == 0 ? 0 : 1;
    sg.c_first = cta_of(u * p.n_kv, r);
    sg.c_last = cta_of((u + 1) * p.n_kv - 1, r);
    return true;
}

// K/V tiles the Q tile starting at q0_t visits in segment sg (0 if the tile is empty).
__device__ __forceinline__ int segment_tiles(const Segment &sg, int q0_t, const FwdParams &p, int BN)
{
    if (!p.split)
        return max(0, kv_tiles_for(q0_t, p.Lq, p.Lk, p.causal, BN) - sg.kv_lo);
    return q0_t < p.Lq ? sg.kv_hi - sg.kv_lo : 0;
}

// All lanes wait (bounded); the warp agrees on the outcome so warp-collective
// tcgen05 instructions are executed by all lanes or by none.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int *err, int code,
                                          unsigned long long limit)
{
    const bool ok = ptx::mbar_wait(bar, parity, err, code, limit);
    return __all_sync(0xffffffffu, ok);
}

template <class C, bool GRP = false>
__global__ void __launch_bounds__(C::NUM_THREADS, 1)
    fa2_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const FwdParams p, const __grid_constant__ SplitRanges ranges)
{
    using namespace ptx;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };

    // ---- setup: barriers, TMEM
    if (threadIdx.x == 0) {
        for (int t = 0; t < C::NQ; ++t) {
            mbar_init(bar(C::BAR_Q_FULL + t), 1);
            // with Q in TMEM the softmax threads free the shared-memory copy once copied
            mbar_init(bar(C::BAR_Q_EMPTY + t), C::QT ? C::GROUP_WARPS : 1);
            mbar_init(bar(C::BAR_O_DONE + t), 1);
            mbar_init(bar(C::BAR_O_FREE + t), C::GROUP_WARPS);
            mbar_init(bar(C::BAR_XMAX + 2 * t), C::GROUP_WARPS);
            mbar_init(bar(C::BAR_XMAX + 2 * t + 1), C::GROUP_WARPS);
            mbar_init(bar(C::BAR_GROUP + t), C::GROUP_WARPS);
        }
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(bar(C::BAR_K_FULL + s), 1);
            mbar_init(bar(C::BAR_K_EMPTY + s), 1);
            mbar_init(bar(C::BAR_V_FULL + s), 1);
            mbar_init(bar(C::BAR_V_EMPTY + s), 1);
        }
        for (int i = 0; i < C::NQ * C::NS; ++i) {
            mbar_init(bar(C::BAR_S_FULL + i), 1);
            mbar_init(bar(C::BAR_P_READY + i), C::GROUP_WARPS);
            for (int q = 0; q < C::NP - 1; ++q)
                mbar_init(bar(C::BAR_PA_READY + i * (C::NP - 1) + q), C::GROUP_WARPS);
        }
        mbar_init(bar(C::BAR_DRAIN), 1);
        mbar_init(bar(C::BAR_NEVER), 1);
        for (int q = 0; q < 2; ++q) {
            mbar_init(bar(C::BAR_QT_FULL + q), C::GROUP_WARPS);
            mbar_init(bar(C::BAR_QT_EMPTY + q), 1);
        }
        fence_mbar_init();
    }
    if (warp == C::WARP_MMA) {
        tmem_alloc(sbase + C::OFF_TMEM_SLOT, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem =
        *reinterpret_cast<volatile uint32_t *>(smem_raw + (sbase - raw) + C::OFF_TMEM_SLOT);

    if (warp >= C::NUM_SOFTMAX_WARPS) {
      // control warpgroup: every warp of it gives up registers at the same point
      if constexpr (C::REG_SPLIT)
          setmaxnreg_dec<C::REG_CTRL>();
      if (warp == C::WARP_PRODUCER) {
        // ================================================== TMA producer (one lane)
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            uint32_t kv_iter = 0;            // K/V tiles issued so far (ring position)
            uint32_t q_loads[C::NQ] = {};    // Q loads issued per Q buffer
            bool k_pending = false;          // a K load of ring slot kv_iter is in flight without its V
            bool ok = true;
            for (int i = 0; ok; ++i) {
                Segment sg;
                if (!segment_at<GRP>(i, p, ranges, sg))
                    break;
                int qg, bh;
                decode_unit<GRP>(sg.unit, p, qg, bh);
                const int q0 = qg * (C::NQ * C::BM);
                int n_max = 0;
#pragma unroll
                for (int t = 0; t < C::NQ; ++t) {
                    const int n = segment_tiles(sg, q0 + t * C::BM, p, C::BN);
                    n_max = max(n_max, n);
                    if (n > 0 && ok) {
                        // the buffer is free once the last S MMA of the previous unit read it
                        if (q_loads[t] > 0 &&
                            !mbar_wait(bar(C::BAR_Q_EMPTY + t), (q_loads[t] - 1) & 1, p.err, ERR_PRODUCER | 3,
                                       p.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar(C::BAR_Q_FULL + t), C::Q_TILE);
#pragma unroll
                        for (int c = 0; c < C::DB; ++c)
                            tma_load_4d_hint(sbase + C::OFF_Q + t * C::Q_TILE + c * C::Q_BLOCK, &tm_q, C::ECOLS * c,
                                             q0 + t * C::BM, bh % p.H, bh / p.H, bar(C::BAR_Q_FULL + t), pol_q);
                        ++q_loads[t];
                    }
                }
                for (int j = 0; j < n_max && ok; ++j, ++kv_iter) {
                    const int s = kv_iter % C::KS;
                    const uint32_t ph = (kv_iter / C::KS) & 1;
                    if (!mbar_wait(bar(C::BAR_K_EMPTY + s), ph ^ 1u, p.err, ERR_PRODUCER | 1, p.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(C::BAR_K_FULL + s), C::KV_TILE);
#pragma unroll
                    for (int c = 0; c < C::DB; ++c)
                        tma_load_4d_hint(sbase + C::OFF_K + s * C::KV_TILE + c * C::KV_BLOCK, &tm_k, C::ECOLS * c,
                                         (sg.kv_lo + j) * C::BN, bh % p.H, bh / p.H, bar(C::BAR_K_FULL + s), pol_kv);
                    k_pending = true;
                    if (!mbar_wait(bar(C::BAR_V_EMPTY + s), ph ^ 1u, p.err, ERR_PRODUCER | 2, p.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(C::BAR_V_FULL + s), C::KV_TILE);
#pragma unroll
                    for (int c = 0; c < C::DB; ++c)
                        tma_load_4d_hint(sbase + C::OFF_V + s * C::KV_TILE + c * C::KV_BLOCK, &tm_v, C::ECOLS * c,
                                         (sg.kv_lo + j) * C::BN, bh % p.H, bh / p.H, bar(C::BAR_V_FULL + s), pol_kv);
                    k_pending = false;
                }
            }
            // Before the CTA may exit, every load this thread started must have landed
            // (immediate on the normal path: all of them were consumed).  After an
            // abort between a K and its V load, that K load is awaited too.
#pragma unroll
            for (int t = 0; t < C::NQ; ++t)
                if (q_loads[t] > 0)
                    mbar_wait(bar(C::BAR_Q_FULL + t), (q_loads[t] - 1) & 1, p.err, ERR_DRAIN | 1, p.drain_limit_ns);
            const uint32_t k_done = kv_iter + (k_pending ? 1u : 0u);
            for (uint32_t it = (k_done > C::KS ? k_done - C::KS : 0); it < k_done; ++it)
                mbar_wait(bar(C::BAR_K_FULL + it % C::KS), (it / C::KS) & 1, p.err, ERR_DRAIN | 2,
                          p.drain_limit_ns);
            for (uint32_t it = (kv_iter > C::KS ? kv_iter - C::KS : 0); it < kv_iter; ++it)
                mbar_wait(bar(C::BAR_V_FULL + it % C::KS), (it / C::KS) & 1, p.err, ERR_DRAIN | 3,
                          p.drain_limit_ns);
        }
        __syncwarp();
      } else if (warp == C::WARP_MMA) {
        // ================================================== MMA issuer
        // One elected lane runs the whole issue loop -- its waits, MMAs and
        // commits -- and the other lanes wait at the final __syncwarp.  (MMAs
        // issued from a branch that the rest of the warp skips, once per group,
        // cost 20-40 clk more each than back-to-back issue from one thread.)
        if (elect_one()) {
            // Descriptor bases; a K step moves the start address, which is the low
            // field of the descriptor in 16-byte units, so it is a plain add.
            const uint64_t desc_q = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
            const uint64_t desc_k = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
            const uint64_t desc_v = sdesc_sw128(sbase + C::OFF_V, C::KV_BLOCK, 1024);
            uint32_t kv_iter = 0;              // ring position of the current unit's K/V tile 0
            uint32_t tbase[C::NQ] = {};        // S/PV tiles of each Q buffer in earlier units
            uint32_t q_loads[C::NQ] = {};      // Q loads consumed per Q buffer
            uint32_t units[C::NQ] = {};        // earlier units that used each Q buffer
            bool ok = true;

            for (int i = 0; ok; ++i) {
                Segment sg;
                if (!segment_at<GRP>(i, p, ranges, sg))
                    break;
                int qg, bh;
                decode_unit<GRP>(sg.unit, p, qg, bh);
                const int q0 = qg * (C::NQ * C::BM);
                int n_t[C::NQ];
                int n_max = 0;
#pragma unroll
                for (int t = 0; t < C::NQ; ++t) {
                    n_t[t] = segment_tiles(sg, q0 + t * C::BM, p, C::BN);
                    n_max = max(n_max, n_t[t]);
                }
                // QT: the TMEM buffer holding this segment's Q (segments alternate)
                const uint32_t qt_buf = q_loads[0] % C::QB;
                // the last Q tile (highest t) that reads K/V tile j
                auto last_user = [&](int j) {
                    int lu = 0;
#pragma unroll
                    for (int t = 0; t < C::NQ; ++t)
                        if (j < n_t[t])
                            lu = t;
                    return lu;
                };

                // S(t, j) = Q_t K_j^T  into S/P buffer (t, (tbase + j) % NS)
                auto issue_s = [&](int t, int j) -> bool {
                    const uint32_t it = kv_iter + j;
                    const int s = it % C::KS;
                    if (!lone_wait(bar(C::BAR_K_FULL + s), (it / C::KS) & 1, p.err, ERR_MMA | 2, p.wait_limit_ns))
                        return false;
                    tc_fence_after();
                    const uint32_t g = tbase[t] + j;
                    const int b = g % C::NS;
                    {
                        const uint32_t d = tmem + C::TM_S + (t * C::NS + b) * C::BN;
                        const uint64_t dk = desc_k + static_cast<uint64_t>((s * C::KV_TILE) >> 4);
                        if constexpr (C::QT) {
                            // A = Q from TMEM buffer qt_buf: 16 bf16 (8 columns) per K step
                            const uint32_t a = tmem + C::TM_Q + qt_buf * (C::D / 2);
#pragma unroll
                            for (int kk = 0; kk < C::D / 16; ++kk)
                                mma_ts(d, a + kk * 8,
                                       dk + static_cast<uint64_t>(((kk >> 2) * C::KV_BLOCK + (kk & 3) * 32) >> 4),
                                       C::IDESC_S, kk > 0 ? 1u : 0u);
                        } else {
                            const uint64_t dq = desc_q + static_cast<uint64_t>((t * C::Q_TILE) >> 4);
#pragma unroll
                            for (int kk = 0; kk < C::S_KSTEPS; ++kk)
                                mma_ss<C::F8>(d, dq + static_cast<uint64_t>(((kk >> 2) * C::Q_BLOCK + (kk & 3) * 32) >> 4),
                                       dk + static_cast<uint64_t>(((kk >> 2) * C::KV_BLOCK + (kk & 3) * 32) >> 4),
                                       C::IDESC_S, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(bar(C::BAR_S_FULL + t * C::NS + b));
                        if (last_user(j) == t)
                            mma_commit(bar(C::BAR_K_EMPTY + s));
                        if (j == n_t[t] - 1)   // last read of this unit's Q tile
                            mma_commit(bar(C::QT ? C::BAR_QT_EMPTY + qt_buf : C::BAR_Q_EMPTY + t));
                    }
                    return true;
                };
                // O_t (+)= P(t, j) V_j, P read from TMEM
                auto issue_pv = [&](int t, int j) -> bool {
                    const uint32_t it = kv_iter + j;
                    const int s = it % C::KS;
                    const uint32_t g = tbase[t] + j;
                    const int b = g % C::NS;
                    // P arrives in NP key parts: each part's barrier before its K steps
                    auto part_bar = [&](int q) {
                        return q < C::NP - 1 ? bar(C::BAR_PA_READY + (t * C::NS + b) * (C::NP - 1) + q)
                                             : bar(C::BAR_P_READY + t * C::NS + b);
                    };
                    if (!lone_wait(part_bar(0), (g / C::NS) & 1, p.err, ERR_MMA | 3, p.wait_limit_ns))
                        return false;
                    if (!lone_wait(bar(C::BAR_V_FULL + s), (it / C::KS) & 1, p.err, ERR_MMA | 4, p.wait_limit_ns))
                        return false;
                    // the first PV of a unit overwrites O_t: the previous unit's epilogue
                    // must have read it out of TMEM
                    if (j == 0 && units[t] > 0 &&
                        !lone_wait(bar(C::BAR_O_FREE + t), (units[t] - 1) & 1, p.err, ERR_MMA | 5, p.wait_limit_ns))
                        return false;
                    tc_fence_after();
                    {
                        const uint32_t d = tmem + C::TM_O + t * C::D;
                        const uint32_t a = tmem + C::TM_S + (t * C::NS + b) * C::BN;
                        const uint64_t dv = desc_v + static_cast<uint64_t>((s * C::KV_TILE) >> 4);
                        constexpr int KP = C::PV_KSTEPS / C::NP;   // K steps per part of P
#pragma unroll
                        for (int q = 0; q < C::NP; ++q) {
                            if (q > 0) {
                                if (!lone_wait(part_bar(q), (g / C::NS) & 1, p.err, ERR_MMA | 7, p.wait_limit_ns))
                                    return false;
                                tc_fence_after();
                            }
#pragma unroll
                            for (int kk = q * KP; kk < (q + 1) * KP; ++kk)
                                mma_ts<C::F8>(d, a + kk * 8, dv + static_cast<uint64_t>((kk * C::PV_KSTEP_BYTES) >> 4),
                                              C::IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                            if constexpr (C::P2) {   // the residual weights, from the buffer's upper half
#pragma unroll
                                for (int kk = q * KP; kk < (q + 1) * KP; ++kk)
                                    mma_ts(d, a + C::BN / 2 + kk * 8,
                                           dv + static_cast<uint64_t>((kk * C::PV_KSTEP_BYTES) >> 4), C::IDESC_PV, 1u);
                            }
                        }
                        mma_commit(bar(C::BAR_O_DONE + t));
                        if (last_user(j) == t)
                            mma_commit(bar(C::BAR_V_EMPTY + s));
                    }
                    return true;
                };

                // this unit's Q tiles: in shared memory (TMA), or copied into TMEM buffer
                // qt_buf by the softmax warps
#pragma unroll
                for (int t = 0; t < C::NQ; ++t) {
                    if (ok && n_t[t] > 0) {
                        if constexpr (C::QT)
                            ok = lone_wait(bar(C::BAR_QT_FULL + qt_buf), (q_loads[0] / C::QB) & 1, p.err,
                                           ERR_MMA | 6, p.wait_limit_ns);
                        else
                            ok = lone_wait(bar(C::BAR_Q_FULL + t), q_loads[t] & 1, p.err, ERR_MMA | 1,
                                           p.wait_limit_ns);
                        ++q_loads[t];
                    }
                }
                // Issue order: S for the first NS tiles of every Q tile, then per K/V
                // tile j and Q tile t: PV(t, j) followed by S(t, j + NS), which reuses
                // the TMEM buffer PV(t, j) just read (tcgen05 ops execute in order).
#pragma unroll
                for (int b = 0; b < C::NS; ++b)
#pragma unroll
                    for (int t = 0; t < C::NQ; ++t)
                        if (ok && b < n_t[t])
                            ok = issue_s(t, b);
                for (int j = 0; j < n_max && ok; ++j) {
#pragma unroll
                    for (int t = 0; t < C::NQ; ++t) {
                        if (ok && j < n_t[t]) {
                            ok = issue_pv(t, j);
                            if (ok && j + C::NS < n_t[t])
                                ok = issue_s(t, j + C::NS);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < C::NQ; ++t) {
                    if (n_t[t] > 0) {
                        tbase[t] += n_t[t];
                        ++units[t];
                    }
                }
                kv_iter += n_max;
            }
            // drain: every MMA issued above has completed before TMEM can be released
            mma_commit(bar(C::BAR_DRAIN));
            lone_wait(bar(C::BAR_DRAIN), 0, p.err, ERR_DRAIN | 4, p.drain_limit_ns);
        }
        __syncwarp();
      }
    } else {
        // ================================================== softmax warps
        if constexpr (C::REG_SPLIT)
            setmaxnreg_inc<C::REG_SOFTMAX>();
        const int t = warp / (4 * C::CS);        // Q tile slot
        const int h = (warp >> 2) % C::CS;       // column slice
        const int quarter = warp & 3;            // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t o_addr = tmem + lane_base + C::TM_O + t * C::D + h * C::OCOL;
        const uint32_t o_stage = sbase + C::OFF_OST + warp * C::O_STAGE;   // this warp's O staging
        uint32_t o_boxes = 0;   // O boxes this warp has staged (their half alternates)
        const uint32_t xmax = sbase + C::OFF_XMAX + t * (2 * C::CS * 128 * 4);
        const uint32_t xl = sbase + C::OFF_XL + t * (C::CS * 128 * 8);
        // one arrival per warp: every lane's prior writes (shared memory, and TMEM
        // after its own wait + fence) are ordered before lane 0's arrive by the
        // __syncwarp, and the arrive releases them to the waiting side
        auto warp_arrive = [&](uint32_t b) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(b);
        };
        uint32_t tbase = 0;    // S tiles of this slot in earlier segments (running phase base)
        uint32_t group_uses = 0;   // completed phases of this slot's group barrier
        // tests of the time-out path: a wait that must run out (the other roles' waits on
        // these warps then run out too, and every CTA drains its own work and exits)
        bool ok = !p.stall_test ||
                  warp_wait(bar(C::BAR_NEVER), 0, p.err, ERR_SOFTMAX | 0xF, p.wait_limit_ns);
        // QT: copy the next Q tile from shared memory into TMEM buffer (q_copies % QB).
        // Each thread moves its own row's slice of D/CS columns: 16-byte pieces of the
        // 128B-swizzled rows (piece c of row r sits at c ^ (r % 8)) become packed bf16
        // pairs, two per TMEM column, as the MMA's A operand expects.
        uint32_t q_copies = 0;
        auto copy_q = [&]() -> bool {
            const uint32_t qb = q_copies % C::QB;
            if (!warp_wait(bar(C::BAR_Q_FULL), q_copies & 1, p.err, ERR_SOFTMAX | 8, p.wait_limit_ns))
                return false;
            // the segment that used this buffer before (QB copies ago) has issued its last S
            if (q_copies >= C::QB && !warp_wait(bar(C::BAR_QT_EMPTY + qb), (q_copies / C::QB - 1) & 1, p.err,
                                                ERR_SOFTMAX | 9, p.wait_limit_ns))
                return false;
            tc_fence_after();
#pragma unroll
            for (int bq = h * (C::OCOL / 64); bq < (h + 1) * (C::OCOL / 64); ++bq) {
                const uint32_t src = sbase + C::OFF_Q + bq * C::Q_BLOCK + row * 128;
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    ld_shared_v4(src + ((c ^ (row & 7)) * 16), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                tmem_st32(tmem + lane_base + C::TM_Q + qb * (C::D / 2) + bq * 32, w);
            }
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(bar(C::BAR_QT_FULL + qb));
            warp_arrive(bar(C::BAR_Q_EMPTY));
            ++q_copies;
            return true;
        };

        for (int i = 0; ok; ++i) {
            Segment sg;
            if (!segment_at<GRP>(i, p, ranges, sg))
                break;
            int qg, bh;
            decode_unit<GRP>(sg.unit, p, qg, bh);
            const int q0_t = qg * (C::NQ * C::BM) + t * C::BM;
            const int grow = q0_t + row;             // query index
            // score multiplier in log2 units (e4m3: the head's Q and K descales folded in)
            const float c2 = C::F8 ? p.scale_log2 * __ldg(p.descale_q + bh) * __ldg(p.descale_k + bh) : p.scale_log2;
            const int n = segment_tiles(sg, q0_t, p, C::BN);
            if (n == 0)
                continue;
            const int kv0 = sg.kv_lo;                // absolute index of the segment's first K/V tile
            if constexpr (C::QT) {
                if (i == 0 && !(ok = copy_q()))
                    break;
            }
            float m_use = -INFINITY;   // running max (log2 domain, possibly stale by < 2^THRESHOLD)
            float l = 0.f;             // running normaliser of the fp32 weights (for LSE)
            float l_o = 0.f;           // running normaliser of the bf16 weights the PV MMA sees (for O)

            for (int j = 0; j < n && ok; ++j) {
                const uint32_t g = tbase + j;
                const int b = g % C::NS;
                ok = warp_wait(bar(C::BAR_S_FULL + t * C::NS + b), (g / C::NS) & 1, p.err, ERR_SOFTMAX | 1,
                               p.wait_limit_ns);
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t s_addr = tmem + lane_base + C::TM_S + (t * C::NS + b) * C::BN;

                float s[C::NCOL];
                {
                    uint32_t r[C::NCOL / 32][32];
#pragma unroll
                    for (int q = 0; q < C::NCOL / 32; ++q)
                        tmem_ld32(s_addr + h * C::NCOL + 32 * q, r[q]);
#pragma unroll
                    for (int q = 0; q < C::NCOL / 32; ++q)
                        tmem_ld_wait(r[q]);
#pragma unroll
                    for (int q = 0; q < C::NCOL / 32; ++q)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            s[32 * q + e] = __uint_as_float(r[q][e]);
                }

                // mask: key tail (j >= Lk), on tiles crossing the diagonal causal j > i, and
                // on tiles crossing a sliding window's left edge j < i - window
                const int jj = kv0 + j;                  // absolute K/V tile
                const int k0 = jj * C::BN + h * C::NCOL;
                const bool band_left = p.window >= 0 && jj * C::BN < q0_t + C::BM - 1 - p.window;
                if ((p.causal && jj * C::BN + C::BN - 1 > q0_t) || (jj * C::BN + C::BN > p.Lk) || band_left) {
                    const int lim = p.causal ? min(grow + 1, p.Lk) : p.Lk;  // keys < lim are visible
                    // as column bounds of this slice: columns c >= hi are masked, and under a
                    // window also columns c < lo (c is a constant once the loop is unrolled,
                    // so each test is one compare against a register)
                    const int hi = lim - k0;
                    if (p.window >= 0) {
                        const int lo = grow - p.window - k0;
#pragma unroll
                        for (int c = 0; c < C::NCOL; ++c)
                            s[c] = (c >= hi || c < lo) ? -INFINITY : s[c];
                    } else {
#pragma unroll
                        for (int c = 0; c < C::NCOL; ++c)
                            s[c] = c >= hi ? -INFINITY : s[c];
                    }
                }

                // row max of this tile (own slice, then the other slices through shared
                // memory): four independent chains of 3-input maxima
                float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
                for (int c = 4; c < C::NCOL; c += 8) {
                    mx0 = max3(mx0, s[c], s[c + 1]);
                    mx1 = max3(mx1, s[c + 2], s[c + 3]);
                    if (c + 4 < C::NCOL) {
                        mx2 = max3(mx2, s[c + 4], s[c + 5]);
                        mx3 = max3(mx3, s[c + 6], s[c + 7]);
                    }
                }
                float mx = fmaxf(max3(mx0, mx1, mx2), mx3);
                if constexpr (C::CS > 1) {
                    const uint32_t xb = xmax + (g & 1) * (C::CS * 128 * 4);
                    st_shared_f32(xb + (h * 128 + row) * 4, mx);
                    warp_arrive(bar(C::BAR_XMAX + 2 * t + (g & 1)));
                    ok = warp_wait(bar(C::BAR_XMAX + 2 * t + (g & 1)), (g >> 1) & 1, p.err, ERR_SOFTMAX | 4,
                                   p.wait_limit_ns);
                    if (!ok)
                        break;
#pragma unroll
                    for (int hh = 0; hh < C::CS; ++hh)
                        if (hh != h)
                            mx = fmaxf(mx, ld_shared_f32(xb + (hh * 128 + row) * 4));
                }
                const float m_tile = mx * c2;

                // The first tile of a segment holds a key every row may see (key 0 for whole
                // units; any tile for the non-causal split schedule) except under a sliding
                // window, where a row's first visible key may come later: its max is then
                // -inf until it does, and the first finite max replaces it through a
                // rescale by 2^-inf = 0.  Later tiles keep the stale max unless it grows a
                // lot.  All slices of a row see the same m_tile and so take the same decision.
                float alpha = 1.f;
                bool rescale = false;
                if (j == 0) {
                    m_use = m_tile;
                } else if (m_tile > m_use + RESCALE_THRESHOLD) {
                    alpha = ex2_approx(m_use - m_tile);
                    m_use = m_tile;
                    rescale = true;
                }

                // Rescale this slice of O (only warps in which some row's max grew) once
                // the previous PV has landed, before any of this tile's P is handed over,
                // so that PV(j) accumulates onto the rescaled O.  Without a rescale there
                // is nothing to wait for: the MMA warp orders PV(j) after PV(j-1) by
                // itself.  A parity wait on O_DONE is only unambiguous while that barrier
                // is at most one phase behind the awaited one: here S(j) completing
                // implies PV(j - NS) completed (and every earlier unit's PVs completed
                // before its epilogue), so waiting for PV(j-1) is safe; the wait at the
                // last tile (taken even without a rescale) keeps the epilogue's wait for
                // PV(n-1) safe too.
                const bool grow_any = __any_sync(0xffffffffu, rescale);
                if (j > 0 && grow_any) {
                    ok = warp_wait(bar(C::BAR_O_DONE + t), (g - 1) & 1, p.err, ERR_SOFTMAX | 2, p.wait_limit_ns);
                    if (!ok)
                        break;
                    tc_fence_after();
#pragma unroll 1
                    for (int cc = 0; cc < C::OCOL / 32; ++cc) {
                        uint32_t r[32];
                        tmem_ld32(o_addr + 32 * cc, r);
                        tmem_ld_wait(r);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                        tmem_st32(o_addr + 32 * cc, r);
                    }
                }

                // p = 2^(s * scale * log2e - m); masked entries give 2^-inf = 0.  P goes to
                // TMEM as bf16 (two per 32-bit column, over the first BN/2 columns of the S
                // buffer; this slice's keys land in columns h*NCOL/2 ..).  Two normalisers
                // are kept: l sums the fp32 p (LSE needs the exact sum) and l_o sums the
                // bf16-rounded p that the PV MMA multiplies, so O's numerator and
                // denominator use the same weights -- with one dominant key the rounding
                // of its weight then cancels instead of showing up in O.
                // (scale and subtract, and the exact sum, run as packed fp32 pairs)
                const uint64_t c2x2 = f32x2(c2, c2);
                // a row may see no key of a window's first tile: its max is then -inf and
                // its weights are 2^-inf = 0 with any finite base
                const float m_sub = m_use == -INFINITY ? 0.f : m_use;
                const uint64_t negm2 = f32x2(-m_sub, -m_sub);
                uint64_t ls01 = 0, ls23 = 0;   // packed (0.f, 0.f)
                float lr0 = 0.f, lr1 = 0.f;
                uint32_t pk[C::PW];
                uint32_t pl[C::P2 ? C::PW : 1];   // P2: the residual terms
                const uint32_t p_addr = s_addr + h * C::PW;
                // weights of columns [CB, CE) into pk (bf16 pairs) and the two sums
                auto exp_cols = [&](auto cb, auto ce) {
                    constexpr int CB = decltype(cb)::value, CE = decltype(ce)::value;
#pragma unroll
                    for (int c = CB; c < CE; c += 4) {
                        float x0, x1, x2, x3;
                        unpack_f32x2(fma_f32x2(f32x2(s[c], s[c + 1]), c2x2, negm2), x0, x1);
                        unpack_f32x2(fma_f32x2(f32x2(s[c + 2], s[c + 3]), c2x2, negm2), x2, x3);
                        const float p0 = ex2_approx(x0);
                        const float p1 = ex2_approx(x1);
                        const float p2 = ex2_approx(x2);
                        const float p3 = ex2_approx(x3);
                        ls01 = add_f32x2(ls01, f32x2(p0, p1));
                        ls23 = add_f32x2(ls23, f32x2(p2, p3));
                        if constexpr (C::F8) {
                            // four keys per TMEM column; l_o sums the e4m3 values the MMA sees
                            const uint32_t w = pack_e4m3x4(p0, p1, p2, p3);
                            pk[c / 4] = w;
                            lr0 = add_e4m3x4_to_f32(lr0, w);
                        } else {
                            const uint32_t w0 = pack_bf16x2(p0, p1);
                            const uint32_t w1 = pack_bf16x2(p2, p3);
                            pk[c / 2] = w0;
                            pk[c / 2 + 1] = w1;
                            if constexpr (C::P2) {
                                // p - bf16(p) is exact in fp32; rounding it to bf16 leaves p_hi + p_lo
                                // within about 2^-17 of p, so O is divided by the exact sum l
                                pl[c / 2] = pack_bf16x2_of_f32x2(sub_f32x2(f32x2(p0, p1), widen_bf16x2(w0)));
                                pl[c / 2 + 1] = pack_bf16x2_of_f32x2(sub_f32x2(f32x2(p2, p3), widen_bf16x2(w1)));
                            } else {
                                lr0 = add_bf16x2_to_f32(lr0, w0);
                                lr1 = add_bf16x2_to_f32(lr1, w1);
                            }
                        }
                    }
                };
                // words [W0, W0 + NW) of pk to their TMEM columns
                auto store_words = [&](auto w0, auto nw) {
                    constexpr int W0 = decltype(w0)::value, NW = decltype(nw)::value;
                    static_assert(NW % 32 == 0 || NW == 16 || NW == 8, "P stores move 8, 16 or 32 columns at a time");
                    auto put = [&](uint32_t addr, const uint32_t *src) {
                        if constexpr (NW % 32 == 0) {
#pragma unroll
                            for (int q = 0; q < NW / 32; ++q)
                                tmem_st32(addr + 32 * q, *reinterpret_cast<const uint32_t(*)[32]>(src + 32 * q));
                        } else if constexpr (NW == 16) {
                            tmem_st16(addr, src);
                        } else {
                            tmem_st8(addr, src);
                        }
                    };
                    put(p_addr + W0, pk + W0);
                    if constexpr (C::P2)   // residual terms over the buffer's upper half
                        put(p_addr + C::BN / 2 + W0, pl + W0);
                };
                // part q of NP: its weights, stored, and (all but the last) handed to the
                // MMA warp before the next part is computed
                auto part = [&](auto qc) {
                    constexpr int Q = decltype(qc)::value, PC = C::NCOL / C::NP;
                    exp_cols(std::integral_constant<int, Q * PC>{}, std::integral_constant<int, (Q + 1) * PC>{});
                    store_words(std::integral_constant<int, Q * PC * C::EB / 4>{},
                                std::integral_constant<int, PC * C::EB / 4>{});
                    if constexpr (Q < C::NP - 1) {
                        tmem_st_wait();
                        tc_fence_before();
                        warp_arrive(bar(C::BAR_PA_READY + (t * C::NS + b) * (C::NP - 1) + Q));
                    }
                };
                part(std::integral_constant<int, 0>{});
                if constexpr (C::NP > 1)
                    part(std::integral_constant<int, 1>{});
                if constexpr (C::NP > 2) {
                    part(std::integral_constant<int, 2>{});
                    part(std::integral_constant<int, 3>{});
                }
                {
                    float a0, a1, a2, a3;
                    unpack_f32x2(ls01, a0, a1);
                    unpack_f32x2(ls23, a2, a3);
                    l = l * alpha + ((a0 + a1) + (a2 + a3));
                }
                if constexpr (C::P2)
                    l_o = l;   // the two terms together carry p itself
                else
                    l_o = l_o * alpha + (lr0 + lr1);
                if (j > 0 && !grow_any && j == n - 1) {
                    ok = warp_wait(bar(C::BAR_O_DONE + t), (g - 1) & 1, p.err, ERR_SOFTMAX | 2, p.wait_limit_ns);
                    if (!ok)
                        break;
                }
                tmem_st_wait();
                tc_fence_before();
                // P_READY is per S buffer: the softmax may finish tile j+1 before the MMA
                // warp has seen tile j, but it can only reuse a buffer after the MMA warp
                // issued the S that refills it, i.e. after it consumed that buffer's P.
                warp_arrive(bar(C::BAR_P_READY + t * C::NS + b));
            }
            if (!ok)
                break;
            if constexpr (C::QT) {
                // the next segment's Q goes into TMEM now, so its first S MMAs run during
                // this epilogue
                Segment next;
                if (segment_at<GRP>(i + 1, p, ranges, next) && !(ok = copy_q()))
                    break;
            }

            // ---- epilogue: O out of TMEM (then released to the MMA warp), O / l -> bf16
            // rows and LSE straight to global memory; a cut unit's part goes to the
            // workspace first and the last part to finish combines all of them
            const uint32_t g_last = tbase + n - 1;
            ok = warp_wait(bar(C::BAR_O_DONE + t), g_last & 1, p.err, ERR_SOFTMAX | 3, p.wait_limit_ns);
            if (!ok)
                break;
            // all threads of this slot's group arrive, then wait for the phase to complete
            auto group_sync = [&](int code) -> bool {
                warp_arrive(bar(C::BAR_GROUP + t));
                const bool r = warp_wait(bar(C::BAR_GROUP + t), group_uses & 1, p.err, ERR_SOFTMAX | code,
                                         p.wait_limit_ns);
                ++group_uses;
                return r;
            };
            float l_tot = l, lo_tot = l_o;
            if constexpr (C::CS > 1) {
                st_shared_f32(xl + (h * 128 + row) * 8, l);
                st_shared_f32(xl + (h * 128 + row) * 8 + 4, l_o);
                if (!(ok = group_sync(5)))
                    break;
                l_tot = 0.f;
                lo_tot = 0.f;
#pragma unroll
                for (int hh = 0; hh < C::CS; ++hh) {
                    l_tot += ld_shared_f32(xl + (hh * 128 + row) * 8);
                    lo_tot += ld_shared_f32(xl + (hh * 128 + row) * 8 + 4);
                }
            }
            tc_fence_after();
            // 1/l_o, times the head's V descale for e4m3 inputs
            const float inv_l = (C::F8 ? __ldg(p.descale_v + bh) : 1.f) / lo_tot;
            const bool live = grow < p.Lq;
            const size_t out_row = static_cast<size_t>(bh) * p.Lq + (live ? grow : 0);
            const bool whole = sg.c_first == sg.c_last;
            // O leaves through the warp's staging halves, one 32-column box at a time:
            // o_block_begin waits until the store that last read the next half is done
            // with it (at most one store, the other half's, may still be reading) and
            // returns that half, o_block_put writes 16 bf16 words (32 columns) of this
            // thread's row into it, and o_block_store writes the warp's 32 rows x 32
            // columns with one TMA store (whole 64-byte pieces of its rows; rows past Lq
            // lie outside the tensor map and are not written).
            auto o_block_begin = [&]() -> uint32_t {
                if (lane == 0)
                    bulk_wait_group_read1();
                __syncwarp();
                return o_stage + (o_boxes & 1) * C::O_HALF;
            };
            // (16-byte chunk k of row r sits at k ^ ((r / 2) % 4) in 64-byte rows under the
            // 64B swizzle)
            auto o_block_put = [&](uint32_t buf, const uint32_t (&w)[16]) {
                const uint32_t rowp = buf + lane * (C::OBW * 2);
                const int sw = (lane >> 1) & 3;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    st_shared_v4(rowp + ((c ^ sw) * 16), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
            };
            auto o_block_store = [&](uint32_t buf, int bq) {
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    if (q0_t + quarter * 32 < p.Lq) {
                        tma_store_4d(&tm_o, buf, h * C::OCOL + C::OBW * bq, q0_t + quarter * 32, bh % p.H, bh / p.H);
                        bulk_commit_group();
                    } else {
                        // no store for rows past Lq: with no group committed for this box,
                        // the next begin's one-pending allowance must not cover its half
                        bulk_wait_group_read0();
                    }
                }
                ++o_boxes;
            };
            // this part's workspace rows (cut units only): LSE pairs by row, O as float4
            // column groups of 128 rows each
            const size_t part_tile = (static_cast<size_t>(blockIdx.x) * 2 + sg.slot) * C::NQ + t;
            const size_t part_row = part_tile * 128 + row;
            const int n_parts = sg.c_last - sg.c_first + 1;
            int *counter = p.counters + sg.c_first * C::NQ + t;
            const uint32_t flag = sbase + C::OFF_FLAG + 4 * t;
            // Part statistics (base 2): lse_o weighs this part's O (its bf16 mass, the
            // normaliser O was divided by), lse_x is its exact log-sum-exp.
            const float own_lse_o = m_use + lg2_approx(lo_tot);
            const float own_lse_x = m_use + lg2_approx(l_tot);

            // Merge of all parts of a cut unit into bf16 O and LSE.  Each part's O is
            // taken as its fp32 values divided by its own normaliser, and the parts are
            // summed in CTA order two at a time, so the result does not depend on which
            // CTA merges or on whether its own part comes from TMEM or the workspace.
            auto combine = [&](bool own_from_tmem) {
                // The slot of part c: every CTA after the unit's first one starts its
                // range inside the unit, so the unit is its first segment (slot 0); the
                // first CTA used slot 0 only if its range starts exactly at the unit's
                // first tile.
                const int first_slot = ranges.begin[sg.c_first] == sg.unit * p.n_kv ? 0 : 1;
                auto tile_of = [&](int c) -> size_t {
                    return (static_cast<size_t>(c) * 2 + (c == sg.c_first ? first_slot : 0)) * C::NQ + t;
                };
                const int self = own_from_tmem ? static_cast<int>(blockIdx.x) : -1;
                auto lse_o_of = [&](int c) {
                    return c == self ? own_lse_o : __ldcg(p.part_lse + (tile_of(c) * 128 + row) * 2);
                };
                // combine weights: O parts by their bf16 masses (lse_o), LSE exactly
                float mo = -INFINITY, mx = -INFINITY;
                for (int c = sg.c_first; c <= sg.c_last; ++c) {
                    mo = fmaxf(mo, lse_o_of(c));
                    mx = fmaxf(mx, c == self ? own_lse_x : __ldcg(p.part_lse + (tile_of(c) * 128 + row) * 2 + 1));
                }
                float wsum = 0.f, xsum = 0.f;
                for (int c = sg.c_first; c <= sg.c_last; ++c) {
                    wsum += ex2_approx(lse_o_of(c) - mo);
                    xsum += ex2_approx((c == self ? own_lse_x : __ldcg(p.part_lse + (tile_of(c) * 128 + row) * 2 + 1)) - mx);
                }
                const float inv_w = 1.f / wsum;
                const float4 *part4 = reinterpret_cast<const float4 *>(p.part_o);
#pragma unroll 1
                for (int bq = 0; bq < C::OCOL / C::OBW; ++bq) {
                  const int cc = bq;   // one 32-column TMEM chunk per box
                  {
                    const size_t col4 = static_cast<size_t>((h * C::OCOL + 32 * cc) / 4) * 128 + row;
                    // this CTA's own part, read out of TMEM when its turn in the sum comes
                    auto load_own = [&](float4 *dst) {
                        uint32_t r[32];
                        tmem_ld32(o_addr + 32 * cc, r);
                        tmem_ld_wait(r);
                        if (cc == C::OCOL / 32 - 1) {
                            tc_fence_before();
                            warp_arrive(bar(C::BAR_O_FREE + t));
                        }
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[q] = make_float4(__uint_as_float(r[4 * q]) * inv_l, __uint_as_float(r[4 * q + 1]) * inv_l,
                                                 __uint_as_float(r[4 * q + 2]) * inv_l,
                                                 __uint_as_float(r[4 * q + 3]) * inv_l);
                    };
                    float acc[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        acc[e] = 0.f;
                    // two parts per step, so 16 loads are in flight per round trip
                    for (int c = sg.c_first; c <= sg.c_last; c += 2) {
                        const bool two = c + 1 <= sg.c_last;
                        const size_t ta = tile_of(c), tb = two ? tile_of(c + 1) : ta;
                        const float wa = ex2_approx(lse_o_of(c) - mo) * inv_w;
                        const float wb = two ? ex2_approx(lse_o_of(c + 1) - mo) * inv_w : 0.f;
                        const float4 *sa = part4 + ta * (C::D / 4) * 128 + col4;
                        const float4 *sb = part4 + tb * (C::D / 4) * 128 + col4;
                        const bool a_own = c == self, b_own = two && c + 1 == self;
                        float4 va[8], vb[8];
                        if (a_own) {
                            load_own(va);
                        } else {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                va[q] = __ldcg(sa + q * 128);
                        }
                        if (b_own) {
                            load_own(vb);
                        } else {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                vb[q] = __ldcg(sb + q * 128);
                        }
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            acc[4 * q] += wa * va[q].x + wb * vb[q].x;
                            acc[4 * q + 1] += wa * va[q].y + wb * vb[q].y;
                            acc[4 * q + 2] += wa * va[q].z + wb * vb[q].z;
                            acc[4 * q + 3] += wa * va[q].w + wb * vb[q].w;
                        }
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
                    const uint32_t buf = o_block_begin();
                    o_block_put(buf, w);
                    o_block_store(buf, bq);
                  }
                }
                if (h == 0 && live)
                    p.lse[out_row] = (mx + lg2_approx(xsum)) * LN2;
            };

            // A cut unit's part that finds every other part already published merges
            // straight from TMEM; otherwise it publishes itself first.
            bool direct = false;
            if (!whole) {
                if (h == 0 && row == 0) {
                    const int arrived = ld_acquire_gpu(counter);
                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(flag), "r"(arrived == n_parts - 1 ? 1 : 0)
                                 : "memory");
                }
                if (!(ok = group_sync(6)))
                    break;
                uint32_t d;
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(d) : "r"(flag) : "memory");
                direct = d != 0;
            }
            if (direct) {
                fence_acq_rel_gpu();
                combine(true);
                if (h == 0 && row == 0)
                    atomicExch(counter, 0);   // leave the workspace ready for the next call
            } else {
                if (whole) {
                    // one 32-column chunk at a time (loading more of them at once measured
                    // slower: the registers they hold cost the step loop), each staged in
                    // the half that the store before last has finished reading
#pragma unroll 1
                    for (int cc = 0; cc < C::OCOL / 32; ++cc) {
                        uint32_t r[32];
                        tmem_ld32(o_addr + 32 * cc, r);
                        tmem_ld_wait(r);
                        if (cc == C::OCOL / 32 - 1) {
                            // every read of O_t is done: the next segment's first PV may overwrite it
                            tc_fence_before();
                            warp_arrive(bar(C::BAR_O_FREE + t));
                        }
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
                        const uint32_t buf = o_block_begin();
                        o_block_put(buf, w);
                        o_block_store(buf, cc);
                    }
                } else {
                    float4 *ptile = reinterpret_cast<float4 *>(p.part_o) + part_tile * (C::D / 4) * 128;
#pragma unroll 1
                    for (int cc = 0; cc < C::OCOL / 32; ++cc) {
                        uint32_t r[32];
                        tmem_ld32(o_addr + 32 * cc, r);
                        tmem_ld_wait(r);
                        if (cc == C::OCOL / 32 - 1) {
                            tc_fence_before();
                            warp_arrive(bar(C::BAR_O_FREE + t));
                        }
                        const int g0 = (h * C::OCOL + 32 * cc) / 4;   // first float4 column group
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            ptile[(g0 + q) * 128 + row] = make_float4(
                                __uint_as_float(r[4 * q]) * inv_l, __uint_as_float(r[4 * q + 1]) * inv_l,
                                __uint_as_float(r[4 * q + 2]) * inv_l, __uint_as_float(r[4 * q + 3]) * inv_l);
                    }
                }
                if (whole) {
                    if (h == 0 && live)
                        p.lse[out_row] = (m_use + lg2_approx(l_tot)) * LN2;
                } else {
                    if (h == 0) {
                        p.part_lse[part_row * 2] = own_lse_o;
                        p.part_lse[part_row * 2 + 1] = own_lse_x;
                    }
                    // publish the part, count it, and let the last part in do the merge
                    fence_acq_rel_gpu();
                    if (!(ok = group_sync(7)))
                        break;
                    if (h == 0 && row == 0) {
                        const int before = atomicAdd(counter, 1);
                        const int last = before == n_parts - 1;
                        if (last)
                            atomicExch(counter, 0);   // leave the workspace ready for the next call
                        asm volatile("st.shared.u32 [%0], %1;" ::"r"(flag), "r"(last) : "memory");
                    }
                    if (!(ok = group_sync(8)))
                        break;
                    uint32_t last;
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(last) : "r"(flag) : "memory");
                    if (last) {
                        fence_acq_rel_gpu();
                        combine(false);
                    }
                }
            }
            tbase += n;
        }
        // a loop left early (a wait that ran out) may leave P stores in flight
        tmem_st_wait();
        if (lane == 0)   // O stores complete before the CTA (and its staging buffer) goes
            bulk_wait_group0();
        __syncwarp();
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == C::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace fa2
