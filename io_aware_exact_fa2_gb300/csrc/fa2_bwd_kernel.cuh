// fa2_bwd_kernel.cuh -- exact FlashAttention-2 backward pass for sm_103a.
//
// The method ("Chapter 08: Flash Attention -- blocked attention", section 6):
// given dO, the forward's O and per-row LSE, recompute the probabilities P
// instead of storing them, and
//   6.2  Delta_i = sum_d dO_id O_id                      (one scalar per query row)
//   6.3  dS = P * (dP - Delta),  dP = dO V^T             (softmax backward)
//   6.4  dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K
// with the two loop structures the section gives: K/V tiles stay on chip while
// query tiles stream past (dK and dV of those keys need every query's P and
// dS column), and Q tiles stay on chip while key tiles stream past (dQ of those
// queries needs every key).  Scores are taken to base 2 (scale * log2 e folded
// into one FMA, LSE * log2 e per row), so P = 2^(s * c - lse2) exactly as in
// the forward; in natural-log terms the section's ln 2 factors cancel.
//
// GB300 mapping, per kernel:
//   * TMA (128B swizzle) moves the resident tiles once and the streamed tiles
//     through a ring; one warp issues tcgen05.mma (elected lane); the
//     elementwise warps own 32-lane TMEM quarters (one TMEM lane = one row), two
//     per quarter with half of a step's 64 columns each, or (D = 256, 32-row
//     steps) one per quarter.
//   * The two score-like products of a step (S and dP, or their transposes)
//     go into one of two TMEM buffer pairs, so the next step's pair is computed
//     while the elementwise warps work on this one.  P and dS are written back
//     over them as bf16 and read by the gradient MMAs straight from TMEM; the
//     streamed tiles serve as the MMA's B operand both K-major (for S, dP) and
//     MN-major (for dV, dK, dQ) without a transpose pass.
//   * The Delta kernel also writes each query row's -lse * log2 e beside -Delta,
//     in 64-row tiles, so a streamed query tile's statistics ride bulk copies
//     on the same ring barrier as its Q and dO tiles (no global loads in the
//     producer's loop).
//   * Every wait is bounded (a device error word records which one ran out).
#pragma once

#include <cstdint>
#include <cuda.h>

#include "sm103_ptx.cuh"

namespace fa2 {

// Per-row statistics the gradient kernels read, written by the Delta kernel in
// tiles of BWD_STAT_ROWS query rows: fp32 [B*H][tiles][2][BWD_STAT_ROWS] holding
// (-lse * log2 e, -Delta) per row, so that one bulk copy brings a streamed query
// tile's statistics into shared memory.  Rows past Lq hold (-inf, 0): P = 0 there.
constexpr int BWD_STAT_ROWS = 64;

struct BwdParams {
    const float *stats;     // the statistics tiles above
    int n_stat_tiles;       // tiles per head = ceil(Lq / BWD_STAT_ROWS)
    uint16_t *dq;           // bf16 [B, H, Lq, D] view: row (b, h, i) at b*dq_sb + h*dq_sh + i*dq_sl
    uint16_t *dk, *dv;      // bf16 [B, H, Lk, D] views, likewise
    long long dq_sb, dq_sh, dq_sl, dk_sb, dk_sh, dk_sl, dv_sb, dv_sh, dv_sl;   // element strides
    int H;                  // heads: flat head bh = b * H + h
    int head_group;         // causal grids: heads per group (heaviest tiles first within a group)
    // bit m set: tensor map m (BWD_MAP_*) is 3-D (D, L, B*H), else 4-D (D, L, H, B)
    int maps3;
    int *err;
    unsigned long long wait_limit_ns;
    int Lq, Lk, BH;
    int causal;
    int window;             // >= 0 (with causal): query i sees keys i - window .. i; -1: no window
    float scale;            // softmax scale (dK, dQ carry it)
    float scale_log2;       // scale * log2(e)
};

enum : int {
    ERR_BWD_PRODUCER = 0x500,
    ERR_BWD_MMA = 0x600,
    ERR_BWD_ELEM = 0x700,
};

constexpr float BWD_LOG2E = 1.4426950408889634074f;

// All lanes wait (bounded) and agree on the outcome, so warp-collective tcgen05
// instructions that follow run on all lanes or none.
__device__ __forceinline__ bool warp_wait_all(uint32_t bar, uint32_t parity, int *err, int code,
                                              unsigned long long limit)
{
    const bool ok = ptx::mbar_wait(bar, parity, err, code, limit);
    return __all_sync(0xffffffffu, ok);
}

// The tensor maps of the gradient kernels.  A view whose batch stride is H times its head
// stride (a contiguous tensor, for one) is mapped as 3-D (D, L, B*H); others as 4-D
// (D, L, H, B).  Streamed 64-row boxes through 4-D maps measured 7 % slower in dK/dV.
enum : int { BWD_MAP_Q = 0, BWD_MAP_K = 1, BWD_MAP_V = 2, BWD_MAP_DO = 3 };

// One box of a [B, H, L, D] view: columns c0.., rows row.. of flat head bh (= hb * H + hh).
__device__ __forceinline__ void bwd_tma_load(uint32_t dst, const void *tmap, bool map3, int c0, int row, int bh,
                                             int hh, int hb, uint32_t bar)
{
    if (map3)
        ptx::tma_load_3d(dst, tmap, c0, row, bh, bar);
    else
        ptx::tma_load_4d(dst, tmap, c0, row, hh, hb, bar);
}

// Element strides (batch, head, row) of a [B, H, L, D] view whose rows of D are contiguous.
struct BwdRowStrides {
    long long b, h, l;
};

// ---------------------------------------------------------------- Delta (6.2)
// Delta = sum_d dO * O in fp32 from the bf16 tensors, for every query row (padded
// rows included), stored negated beside -lse * log2 e in the statistics tiles.  A
// row is D/8 lanes, each with one 16-byte piece of O and of dO, so a warp covers
// 32 / (D/8) rows with two vector loads per lane.
constexpr int BWD_DELTA_THREADS = 256;

template <int D>
__host__ __device__ constexpr int bwd_delta_rows_per_block()
{
    return (BWD_DELTA_THREADS / 32) * (32 / (D / 8));
}

template <int D>
__global__ void __launch_bounds__(BWD_DELTA_THREADS) fa2_bwd_delta_kernel(const uint16_t *__restrict__ o,
                                                                          const uint16_t *__restrict__ dout,
                                                                          const float *__restrict__ lse,
                                                                          float *__restrict__ stats, int Lq,
                                                                          int n_tiles, long long rows, int H,
                                                                          BwdRowStrides o_st, BwdRowStrides do_st)
{
    constexpr int LPR = D / 8;            // lanes per row
    const int lane = threadIdx.x & 31;
    const int piece = lane % LPR;
    const long long r = static_cast<long long>(blockIdx.x) * bwd_delta_rows_per_block<D>() +
                        (threadIdx.x >> 5) * (32 / LPR) + lane / LPR;
    const long long per_head = static_cast<long long>(n_tiles) * BWD_STAT_ROWS;
    const long long bh = r / per_head;
    const int i = static_cast<int>(r - bh * per_head);
    const bool live = r < rows && i < Lq;
    float acc = 0.f;
    if (live) {
        const long long b_ = bh / H, h_ = bh % H;
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(o + b_ * o_st.b + h_ * o_st.h + i * o_st.l + piece * 8));
        const uint4 b = __ldg(
            reinterpret_cast<const uint4 *>(dout + b_ * do_st.b + h_ * do_st.h + i * do_st.l + piece * 8));
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = fmaf(__uint_as_float(wa[e] << 16), __uint_as_float(wb[e] << 16), acc);
            acc = fmaf(__uint_as_float(wa[e] & 0xffff0000u), __uint_as_float(wb[e] & 0xffff0000u), acc);
        }
    }
    // sum over the row's lanes (xor offsets below LPR stay within the row's group)
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (piece == 0 && r < rows) {
        float *t = stats + (bh * n_tiles + i / BWD_STAT_ROWS) * 2 * BWD_STAT_ROWS + i % BWD_STAT_ROWS;
        t[0] = i < Lq ? -(lse[bh * Lq + i] * BWD_LOG2E) : -INFINITY;
        t[BWD_STAT_ROWS] = i < Lq ? -acc : 0.f;
    }
}

// Shared configuration of the two gradient kernels: RES rows of the resident
// tiles (TMEM lanes), STR rows per streamed tile, head dimension D, EW
// elementwise warps (4: one per 32-lane TMEM quarter; 8: two per quarter, each
// with half of a step's columns), DH gradient columns per CTA.  With DH = D / 2
// (D = 256) two CTAs share each resident tile: both compute the step's full-D
// score products, each accumulates and stores one half of the gradient columns,
// so that the gradient accumulators and the score buffers fit the 512 TMEM columns.
template <int D_, int RES_, int STR_, int RING_, int EW_, int DH_ = D_>
struct BwdCfg {
    static constexpr int D = D_;
    static constexpr int RES = RES_;     // resident rows per CTA (= 128 TMEM lanes)
    static constexpr int STR = STR_;     // rows of a streamed tile per step
    static constexpr int RING = RING_;   // streamed-tile ring stages
    static constexpr int EW = EW_;       // elementwise warps
    static constexpr int DH = DH_;       // gradient columns this CTA accumulates
    static constexpr int NH = D / DH;    // CTAs per resident tile (one per column half)
    // score pairs issued ahead of the gradient MMAs: two buffer pairs, but never more
    // than the ring holds (a pair waits for its stage's tiles)
    static constexpr int LA = RING >= 2 ? 2 : 1;
    // the dQ kernel keeps Q and dO as TMEM A operands where TMEM has room beside dQ and
    // the two score-buffer pairs; otherwise its score products read them from shared
    // memory
    static constexpr bool RES_IN_TMEM = DH + 4 * STR + D <= 512;
    // likewise the dK/dV kernel keeps K as the TMEM A operand of S^T = K Q^T where it fits
    // beside dV, dK and the score buffers (D = 64 and 256; V stays in shared memory).  A
    // score MMA with its A operand in shared memory re-reads all of A for each
    // instruction, which bounds the narrow (N = STR) score products.
#ifndef FA2_BWD_K_IN_TMEM
#define FA2_BWD_K_IN_TMEM 1
#endif
    static constexpr bool K_IN_TMEM = FA2_BWD_K_IN_TMEM && 2 * DH + 4 * STR + D / 2 <= 512;
    // and V as the A operand of dP^T = V dO^T, where both fit (D = 64)
    static constexpr bool V_IN_TMEM = K_IN_TMEM && 2 * DH + 4 * STR + D <= 512;
    static constexpr int DB = D / 64;    // 64-column (128-byte) swizzle blocks
    static constexpr int RES_BLOCK = RES * 128;
    static constexpr int RES_TILE = DB * RES_BLOCK;
    static constexpr int STR_BLOCK = STR * 128;
    static constexpr int STR_TILE = DB * STR_BLOCK;
    // shared memory: two resident tiles, the ring (two streamed tiles per stage),
    // per-stage row statistics (two floats per streamed row), barriers
    static constexpr int OFF_RES0 = 0;
    static constexpr int OFF_RES1 = RES_TILE;
    static constexpr int OFF_STR0 = 2 * RES_TILE;                 // [RING]
    static constexpr int OFF_STR1 = OFF_STR0 + RING * STR_TILE;    // [RING]
    static constexpr int STAT_BYTES = 2 * STR * 4;                  // -lse2 and -Delta of STR rows
    static constexpr int OFF_STAT = OFF_STR1 + RING * STR_TILE;    // [RING][2][STR] f32
    static constexpr int OFF_BAR = OFF_STAT + RING * STAT_BYTES;
    static constexpr int BAR_RES_FULL = 0;
    static constexpr int BAR_STR_FULL = 1;                  // [RING]
    static constexpr int BAR_STR_EMPTY = BAR_STR_FULL + RING;   // [RING]
    static constexpr int BAR_SCORE_FULL = BAR_STR_EMPTY + RING; // [2] a step's S^T and dP^T (dK/dV) or S (dQ)
    static constexpr int BAR_DP_FULL = BAR_SCORE_FULL + 2;      // [2] a step's dP (dQ kernel)
    static constexpr int BAR_GRAD_READY = BAR_DP_FULL + 2;      // [2] bf16 operands of the gradient MMAs written
    static constexpr int BAR_DONE = BAR_GRAD_READY + 2;         // every MMA completed
    static constexpr int BAR_RES_TMEM = BAR_DONE + 1;           // resident tiles copied into TMEM
    static constexpr int NUM_BARS = BAR_RES_TMEM + 1;
    static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_TMEM_SLOT + 16 + 1024;
    static constexpr int NUM_THREADS = 32 * EW + 64;   // elementwise warps, producer, MMA
    static constexpr int WARP_PRODUCER = EW;
    static constexpr int WARP_MMA = EW + 1;
    static constexpr uint32_t IDESC_PAIR = ptx::idesc_bf16_f32(RES, STR, false, false);
    static constexpr uint32_t IDESC_GRAD = ptx::idesc_bf16_f32(RES, DH, false, true);
    static_assert(D == 64 || D == 128 || D == 256, "gradient kernels support D = 64, 128 and 256");
    static_assert(DH == D || (D == 256 && DH == 128), "the gradient columns are split in two at D = 256 only");
    static_assert(RES == 128 && STR % 16 == 0 && STR >= 32 && STR <= 128, "tile shape");
    static_assert(EW == 4 || EW == 8, "one or two elementwise warps per TMEM lane quarter");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
};

// This thread's row of a resident tile (RES rows, 128B-swizzled 64-column blocks:
// 16-byte piece c of row r sits at c ^ (r % 8)) into TMEM as packed bf16 pairs,
// two per column -- the layout of an MMA A operand read from TMEM.
template <int DB, int BLOCK>
__device__ __forceinline__ void copy_row_to_tmem(uint32_t smem_tile, int row, uint32_t tmem_dst)
{
    using namespace ptx;
#pragma unroll
    for (int bq = 0; bq < DB; ++bq) {
        const uint32_t src = smem_tile + bq * BLOCK + row * 128;
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c)
            ld_shared_v4(src + ((c ^ (row & 7)) * 16), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        tmem_st32(tmem_dst + bq * 32, w);
    }
}

// bf16 pair from two fp32 values (round to nearest even)
__device__ __forceinline__ uint32_t bwd_pack(float lo, float hi) { return ptx::pack_bf16x2(lo, hi); }

// Write this thread's row of a D-column fp32 TMEM accumulator, times `mul`, as bf16
// to global memory (row `valid` == false: nothing is stored).
template <int D>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, float mul, uint16_t *row_ptr, bool valid)
{
    using namespace ptx;
#pragma unroll 1
    for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t r[32];
        tmem_ld32(taddr + 32 * cc, r);
        tmem_ld_wait(r);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
            w[e] = bwd_pack(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
        if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(row_ptr + 32 * cc);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
    }
}

// CTA idx of a gradient grid (n_tiles resident tiles per head, all heads) -> (tile, head).
// Causal grids go group by group (head_group heads each) and, within a group, tile by
// tile across its heads; other grids go head by head.
__device__ __forceinline__ void bwd_cta_tile(int idx, int n_tiles, const BwdParams &p, int &tile, int &bh)
{
    if (!p.causal) {
        tile = idx % n_tiles;
        bh = idx / n_tiles;
        return;
    }
    const int grp = idx / (p.head_group * n_tiles), rem = idx % (p.head_group * n_tiles);
    const int g0 = grp * p.head_group, gn = min(p.head_group, p.BH - g0);
    tile = rem / gn;
    bh = g0 + rem % gn;
}

// ============================================================== dK, dV kernel
// CTA = one tile of RES = 128 keys of one (b, h); steps = query tiles of STR rows.
// TMEM: dV (DH cols), dK (DH cols), two S^T buffers and two dP^T buffers (STR cols
// each; P^T and dS^T overwrite half of each elementwise warp's columns as bf16
// pairs), and where they fit K (K_IN_TMEM) and V (V_IN_TMEM) as packed bf16 pairs.
// The score MMAs read K and V from TMEM when they are there, else from the resident
// shared-memory tiles.
template <class C>
__global__ void __launch_bounds__(C::NUM_THREADS, 1)
    fa2_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                      const BwdParams p)
{
    using namespace ptx;
    static_assert(BWD_STAT_ROWS % C::STR == 0, "a streamed query tile lies in one statistics tile");
    static_assert((C::EW == 8 && C::STR == 64) || (C::EW == 4 && C::STR == 32),
                  "32 query columns per elementwise warp: two warps per lane quarter at 64, one at 32");
    constexpr int TM_DV = 0, TM_DK = C::DH, TM_ST = 2 * C::DH, TM_DPT = 2 * C::DH + 2 * C::STR;
    constexpr int TM_KA = TM_DPT + 2 * C::STR;   // K as packed bf16 pairs (K_IN_TMEM only)
    constexpr int TM_VA = TM_KA + C::D / 2;      // V likewise (V_IN_TMEM only)
    constexpr int TMEM_COLS = 512;
    static_assert(TM_KA + (C::K_IN_TMEM ? C::D / 2 : 0) + (C::V_IN_TMEM ? C::D / 2 : 0) <= TMEM_COLS,
                  "TMEM budget exceeded");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *sgen = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };

    // Causal: groups of head_group heads whose streamed Q and dO fit in L2 together; within
    // a group, key tiles in order across its heads, heaviest first (low keys are seen by
    // the most queries).  Otherwise head by head, so the CTAs running at one time stream
    // the same few heads' Q and dO through L2.
    const int n_kt = (p.Lk + C::RES - 1) / C::RES;
    const int dh = static_cast<int>(blockIdx.x) % C::NH;   // this CTA's half of the gradient columns
    int kt, bh;
    bwd_cta_tile(static_cast<int>(blockIdx.x) / C::NH, n_kt, p, kt, bh);
    if (kt >= n_kt)
        return;
    const int hh = bh % p.H, hb = bh / p.H;   // head and batch of this CTA's tiles
    const bool q3 = (p.maps3 >> BWD_MAP_Q) & 1, k3 = (p.maps3 >> BWD_MAP_K) & 1;   // 3-D tensor maps
    const bool v3 = (p.maps3 >> BWD_MAP_V) & 1, do3 = (p.maps3 >> BWD_MAP_DO) & 1;
    const int k0 = kt * C::RES;
    const int n_qt = (p.Lq + C::STR - 1) / C::STR;
    // causal (top-left): query i sees key j iff j <= i, so query tiles before the
    // one holding row k0 see none of these keys
    const int qt0 = p.causal ? min(k0 / C::STR, n_qt) : 0;
    // under a sliding window only queries up to the last key + window see these keys
    const int qt_end = p.window >= 0 ? min(n_qt, (k0 + C::RES - 1 + p.window) / C::STR + 1) : n_qt;
    const int n_steps = max(0, qt_end - qt0);

    if (threadIdx.x == 0) {
        mbar_init(bar(C::BAR_RES_FULL), 1);
        for (int s = 0; s < C::RING; ++s) {
            mbar_init(bar(C::BAR_STR_FULL + s), 1);
            mbar_init(bar(C::BAR_STR_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::BAR_SCORE_FULL + b), 1);
            mbar_init(bar(C::BAR_DP_FULL + b), 1);
            mbar_init(bar(C::BAR_GRAD_READY + b), C::EW);   // one arrival per elementwise warp
        }
        mbar_init(bar(C::BAR_DONE), 1);
        mbar_init(bar(C::BAR_RES_TMEM), C::EW);
        fence_mbar_init();
    }
    if (warp == C::WARP_MMA) {
        tmem_alloc(sbase + C::OFF_TMEM_SLOT, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sgen + C::OFF_TMEM_SLOT);

    if (warp == C::WARP_PRODUCER) {
        // ------------------------------------------------ TMA producer (whole warp)
        bool ok = true;
        if (n_steps > 0) {
            if (lane == 0) {
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_do);
                mbar_arrive_expect_tx(bar(C::BAR_RES_FULL), 2 * C::RES_TILE);
#pragma unroll
                for (int c = 0; c < C::DB; ++c) {
                    bwd_tma_load(sbase + C::OFF_RES0 + c * C::RES_BLOCK, &tm_k, k3, 64 * c, k0, bh, hh, hb,
                                 bar(C::BAR_RES_FULL));
                    bwd_tma_load(sbase + C::OFF_RES1 + c * C::RES_BLOCK, &tm_v, v3, 64 * c, k0, bh, hh, hb,
                                 bar(C::BAR_RES_FULL));
                }
            }
            // this head's statistics tiles (-lse2 and -Delta of BWD_STAT_ROWS rows each): a
            // step's STR rows of both, one bulk copy each (one copy when STR fills a tile)
            const float *stat_head = p.stats + static_cast<size_t>(bh) * p.n_stat_tiles * 2 * BWD_STAT_ROWS;
            for (int s = 0; s < n_steps && ok; ++s) {
                const int st = s % C::RING;
                if (s >= C::RING)
                    ok = mbar_wait(bar(C::BAR_STR_EMPTY + st), ((s / C::RING) - 1) & 1, p.err,
                                   ERR_BWD_PRODUCER | 1, p.wait_limit_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
                const int q0 = (qt0 + s) * C::STR;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(C::BAR_STR_FULL + st), 2 * C::STR_TILE + C::STAT_BYTES);
                    const float *stat_src = stat_head + (q0 / BWD_STAT_ROWS) * 2 * BWD_STAT_ROWS + q0 % BWD_STAT_ROWS;
                    if constexpr (C::STR < BWD_STAT_ROWS) {
                        bulk_load(sbase + C::OFF_STAT + st * C::STAT_BYTES, stat_src, C::STR * 4,
                                  bar(C::BAR_STR_FULL + st));
                        bulk_load(sbase + C::OFF_STAT + st * C::STAT_BYTES + C::STR * 4, stat_src + BWD_STAT_ROWS,
                                  C::STR * 4, bar(C::BAR_STR_FULL + st));
                    } else {
                        bulk_load(sbase + C::OFF_STAT + st * C::STAT_BYTES, stat_src, C::STAT_BYTES,
                                  bar(C::BAR_STR_FULL + st));
                    }
#pragma unroll
                    for (int c = 0; c < C::DB; ++c) {
                        bwd_tma_load(sbase + C::OFF_STR0 + st * C::STR_TILE + c * C::STR_BLOCK, &tm_q, q3,
                                     64 * c, q0, bh, hh, hb, bar(C::BAR_STR_FULL + st));
                        bwd_tma_load(sbase + C::OFF_STR1 + st * C::STR_TILE + c * C::STR_BLOCK, &tm_do, do3,
                                     64 * c, q0, bh, hh, hb, bar(C::BAR_STR_FULL + st));
                    }
                }
                __syncwarp();
            }
            // every load this warp started has landed before the CTA may exit
            if (lane == 0) {
                mbar_wait(bar(C::BAR_RES_FULL), 0, p.err, ERR_BWD_PRODUCER | 2, p.wait_limit_ns);
                const int issued = ok ? n_steps : 0;
                for (int s = issued > C::RING ? issued - C::RING : 0; s < issued; ++s)
                    mbar_wait(bar(C::BAR_STR_FULL + s % C::RING), (s / C::RING) & 1, p.err, ERR_BWD_PRODUCER | 3,
                              p.wait_limit_ns);
            }
        }
        __syncwarp();
    } else if (warp == C::WARP_MMA) {
        // ------------------------------------------------ MMA issuer
        // One elected lane runs the whole issue loop (waits, MMAs, commits); the
        // rest of the warp waits at the final __syncwarp.
        if (elect_one()) {
            bool ok = true;
            if (n_steps > 0) {
                const uint64_t desc_q = sdesc_sw128(sbase + C::OFF_STR0, 16, 1024);
                const uint64_t desc_do = sdesc_sw128(sbase + C::OFF_STR1, 16, 1024);
                // the same streamed tiles as MN-major B operands (N = this CTA's DH columns
                // along the rows' 128-byte lines, K = query rows)
                const uint32_t half_off = dh * (C::DH / 64) * C::STR_BLOCK;
                const uint64_t desc_q_mn = sdesc_sw128(sbase + C::OFF_STR0 + half_off, C::STR_BLOCK, 1024);
                const uint64_t desc_do_mn = sdesc_sw128(sbase + C::OFF_STR1 + half_off, C::STR_BLOCK, 1024);
                // the resident K and V tiles as K-major A operands
                const uint64_t desc_k = sdesc_sw128(sbase + C::OFF_RES0, 16, 1024);
                const uint64_t desc_v = sdesc_sw128(sbase + C::OFF_RES1, 16, 1024);
                ok = lone_wait(bar(C::BAR_RES_FULL), 0, p.err, ERR_BWD_MMA | 1, p.wait_limit_ns);
                if (C::K_IN_TMEM && ok)   // K copied into TMEM by the elementwise warps
                    ok = lone_wait(bar(C::BAR_RES_TMEM), 0, p.err, ERR_BWD_MMA | 9, p.wait_limit_ns);
                tc_fence_after();
                const auto stage_off = [](int st) { return static_cast<uint64_t>((st * C::STR_TILE) >> 4); };
                // S^T(b) = K Q^T and dP^T(b) = V dO^T for step s
                auto issue_pair = [&](int s) -> bool {
                    const int st = s % C::RING, b = s & 1;
                    if (!lone_wait(bar(C::BAR_STR_FULL + st), (s / C::RING) & 1, p.err, ERR_BWD_MMA | 2,
                                   p.wait_limit_ns))
                        return false;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < C::D / 16; ++kk) {
                        const uint64_t ko = static_cast<uint64_t>(((kk >> 2) * C::RES_BLOCK + (kk & 3) * 32) >> 4);
                        const uint64_t to = static_cast<uint64_t>(((kk >> 2) * C::STR_BLOCK + (kk & 3) * 32) >> 4);
                        if constexpr (C::K_IN_TMEM)
                            mma_ts(tmem + TM_ST + b * C::STR, tmem + TM_KA + kk * 8, desc_q + stage_off(st) + to,
                                   C::IDESC_PAIR, kk > 0 ? 1u : 0u);
                        else
                            mma_ss(tmem + TM_ST + b * C::STR, desc_k + ko, desc_q + stage_off(st) + to,
                                   C::IDESC_PAIR, kk > 0 ? 1u : 0u);
                        if constexpr (C::V_IN_TMEM)
                            mma_ts(tmem + TM_DPT + b * C::STR, tmem + TM_VA + kk * 8, desc_do + stage_off(st) + to,
                                   C::IDESC_PAIR, kk > 0 ? 1u : 0u);
                        else
                            mma_ss(tmem + TM_DPT + b * C::STR, desc_v + ko, desc_do + stage_off(st) + to,
                                   C::IDESC_PAIR, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(C::BAR_SCORE_FULL + b));
                    return true;
                };
                // dV += P^T dO and dK += dS^T Q for step s.  The bf16 pairs of query columns
                // 16 kk .. 16 kk + 15 sit 8 columns each from the start of the 32 columns of
                // the elementwise warp that owns those queries, where it wrote them.
                auto issue_grad = [&](int s) -> bool {
                    const int st = s % C::RING, b = s & 1;
                    if (!lone_wait(bar(C::BAR_GRAD_READY + b), (s >> 1) & 1, p.err, ERR_BWD_MMA | 3,
                                   p.wait_limit_ns))
                        return false;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < C::STR / 16; ++kk) {
                        const uint64_t ko = static_cast<uint64_t>((kk * 16 * 128) >> 4);   // 16 rows
                        const uint32_t acc = (s > 0 || kk > 0) ? 1u : 0u;
                        const int pc = 32 * (kk >> 1) + 8 * (kk & 1);   // pair column of these queries
                        mma_ts(tmem + TM_DV, tmem + TM_ST + b * C::STR + pc, desc_do_mn + stage_off(st) + ko,
                               C::IDESC_GRAD, acc);
                        mma_ts(tmem + TM_DK, tmem + TM_DPT + b * C::STR + pc, desc_q_mn + stage_off(st) + ko,
                               C::IDESC_GRAD, acc);
                    }
                    mma_commit(bar(C::BAR_STR_EMPTY + st));   // this step's Q, dO and stats are free
                    return true;
                };
                for (int s = 0; s < C::LA && s < n_steps && ok; ++s)
                    ok = issue_pair(s);
                for (int s = 0; s < n_steps && ok; ++s) {
                    ok = issue_grad(s);
                    if (ok && s + C::LA < n_steps)
                        ok = issue_pair(s + C::LA);   // into the buffers issue_grad(s + LA - 2) read
                }
                mma_commit(bar(C::BAR_DONE));
                lone_wait(bar(C::BAR_DONE), 0, p.err, ERR_BWD_MMA | 4, p.wait_limit_ns);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ elementwise warps
        // Two warps per 32-lane TMEM quarter: `half` 0 takes query columns 0..31 of
        // every step (and stores dV), `half` 1 columns 32..63 (and stores dK).  With
        // one warp per quarter (32-column steps) that warp does both.
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;         // key row within the tile (TMEM lane)
        const int kj = k0 + row;                     // key index
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int c0 = 32 * half;                    // this warp's first query column of a step
        const float c2 = p.scale_log2;
        bool ok = true;
        if (C::K_IN_TMEM && n_steps > 0) {
            // this row of K into TMEM (the first warp of each quarter), as the A operand of
            // S^T = K Q^T, and (V_IN_TMEM) of V (the second warp), for dP^T = V dO^T
            ok = warp_wait_all(bar(C::BAR_RES_FULL), 0, p.err, ERR_BWD_ELEM | 7, p.wait_limit_ns);
            if (ok) {
                if (half == 0)
                    copy_row_to_tmem<C::DB, C::RES_BLOCK>(sbase + C::OFF_RES0, row, tmem + lane_base + TM_KA);
                if (C::V_IN_TMEM && (half == 1 || C::EW == 4))
                    copy_row_to_tmem<C::DB, C::RES_BLOCK>(sbase + C::OFF_RES1, row, tmem + lane_base + TM_VA);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(C::BAR_RES_TMEM));
            }
        }
        for (int s = 0; s < n_steps && ok; ++s) {
            const int st = s % C::RING, b = s & 1;
            ok = warp_wait_all(bar(C::BAR_SCORE_FULL + b), (s >> 1) & 1, p.err, ERR_BWD_ELEM | 1, p.wait_limit_ns);
            if (!ok)
                break;
            tc_fence_after();
            // the row statistics arrive with the stage's tiles: wait on that barrier
            // directly (it cannot have moved on, since the stage is only refilled
            // after this step's MMAs)
            ok = warp_wait_all(bar(C::BAR_STR_FULL + st), (s / C::RING) & 1, p.err, ERR_BWD_ELEM | 5,
                               p.wait_limit_ns);
            if (!ok)
                break;
            const uint32_t a_st = tmem + lane_base + TM_ST + b * C::STR + c0;
            const uint32_t a_dp = tmem + lane_base + TM_DPT + b * C::STR + c0;
            const uint32_t stat = sbase + C::OFF_STAT + st * C::STAT_BYTES;
            const int q0 = (qt0 + s) * C::STR;
            // query columns c < kj - q0 are masked (causal, key after query); only tiles
            // whose first query of this half lies before this warp's last key need it
            const int first_visible = kj - q0;
            // under a window, query columns c > kj + window - q0 are masked too
            const int last_visible = p.window >= 0 ? kj + p.window - q0 : C::STR;
            const bool need_mask = (p.causal && q0 + c0 < k0 + quarter * 32 + 31) ||
                                   (p.window >= 0 && q0 + c0 + 31 > k0 + quarter * 32 + p.window);
            const uint64_t c2x2 = f32x2(c2, c2);
            const uint64_t zero2 = 0;
            uint32_t rs[32], rd[32], nl[32], nd[32];
            tmem_ld32(a_st, rs);
            tmem_ld32(a_dp, rd);
            // -lse2 and -Delta of this warp's 32 queries (the same for every lane)
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                ld_shared_v4(stat + (c0 + 4 * q) * 4, nl[4 * q], nl[4 * q + 1], nl[4 * q + 2], nl[4 * q + 3]);
                ld_shared_v4(stat + (C::STR + c0 + 4 * q) * 4, nd[4 * q], nd[4 * q + 1], nd[4 * q + 2],
                             nd[4 * q + 3]);
            }
            tmem_ld_wait(rs);
            tmem_ld_wait(rd);
            float pv[32], dv[32];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                float x0, x1;
                unpack_f32x2(fma_f32x2(f32x2(__uint_as_float(rs[e]), __uint_as_float(rs[e + 1])), c2x2,
                                       f32x2(__uint_as_float(nl[e]), __uint_as_float(nl[e + 1]))),
                             x0, x1);
                pv[e] = ex2_approx(x0);
                pv[e + 1] = ex2_approx(x1);
                const uint64_t diff = add_f32x2(f32x2(__uint_as_float(rd[e]), __uint_as_float(rd[e + 1])),
                                                f32x2(__uint_as_float(nd[e]), __uint_as_float(nd[e + 1])));
                unpack_f32x2(fma_f32x2(f32x2(pv[e], pv[e + 1]), diff, zero2), dv[e], dv[e + 1]);
            }
            if (need_mask) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (c0 + e < first_visible || c0 + e > last_visible) {
                        pv[e] = 0.f;
                        dv[e] = 0.f;
                    }
            }
            // P^T and dS^T as bf16 pairs over the first 16 of this warp's 32 columns
            uint32_t pw[16], dw[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                pw[e / 2] = bwd_pack(pv[e], pv[e + 1]);
                dw[e / 2] = bwd_pack(dv[e], dv[e + 1]);
            }
            tmem_st16(a_st, pw);
            tmem_st16(a_dp, dw);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(C::BAR_GRAD_READY + b));
        }
        // epilogue: dV (half 0) or scale * dK (half 1) rows, both with one warp per
        // quarter; zeros when no query sees these keys
        const bool valid = kj < p.Lk;
        const long long ob = hb, oh = hh, orow = valid ? kj : 0;
        uint16_t *dv_row = p.dv + ob * p.dv_sb + oh * p.dv_sh + orow * p.dv_sl + dh * C::DH;
        uint16_t *dk_row = p.dk + ob * p.dk_sb + oh * p.dk_sh + orow * p.dk_sl + dh * C::DH;
        const bool do_v = C::EW == 4 || half == 0, do_k = C::EW == 4 || half == 1;
        if (n_steps == 0) {
            if (valid) {
                for (int d = 0; d < C::DH; d += 8) {
                    if (do_v)
                        *reinterpret_cast<uint4 *>(dv_row + d) = make_uint4(0, 0, 0, 0);
                    if (do_k)
                        *reinterpret_cast<uint4 *>(dk_row + d) = make_uint4(0, 0, 0, 0);
                }
            }
        } else if (ok && warp_wait_all(bar(C::BAR_DONE), 0, p.err, ERR_BWD_ELEM | 2, p.wait_limit_ns)) {
            tc_fence_after();
            if (do_v)
                store_acc_row<C::DH>(tmem + lane_base + TM_DV, 1.f, dv_row, valid);
            if (do_k)
                store_acc_row<C::DH>(tmem + lane_base + TM_DK, p.scale, dk_row, valid);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == C::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ================================================================= dQ kernel
// CTA = one tile of RES = 128 queries of one (b, h); steps = key tiles of STR rows.
// TMEM: dQ (D cols), two S buffers and two dP buffers (STR cols each; each
// elementwise warp writes the dS pairs of its 32 key columns over the first 16 of
// them in the S buffer).
template <class C>
__global__ void __launch_bounds__(C::NUM_THREADS, 1)
    fa2_bwd_q_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const BwdParams p)
{
    using namespace ptx;
    static_assert((C::EW == 8 && C::STR == 64) || (C::EW == 4 && C::STR == 32),
                  "32 key columns per elementwise warp: two warps per lane quarter at 64, one at 32");
    // Q and dO are also copied into TMEM (TM_QA, TM_DOA) so that S = Q K^T and
    // dP = dO V^T read their A operand from TMEM instead of loading it from shared
    // memory for every instruction
    constexpr int TM_DQ = 0, TM_S = C::DH, TM_DP = C::DH + 2 * C::STR;
    constexpr int TM_QA = C::DH + 4 * C::STR, TM_DOA = TM_QA + C::D / 2;   // RES_IN_TMEM only
    constexpr int TMEM_COLS = 512;
    static_assert((C::RES_IN_TMEM ? TM_DOA + C::D / 2 : TM_QA) <= TMEM_COLS, "TMEM budget exceeded");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *sgen = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };

    // Causal: groups of head_group heads, within a group query tiles across its heads,
    // last (heaviest) first.  Otherwise head by head, so the CTAs running at one time
    // stream the same few heads' K and V through L2.
    const int n_qt = (p.Lq + C::RES - 1) / C::RES;
    const int dh = static_cast<int>(blockIdx.x) % C::NH;   // this CTA's half of dQ's columns
    int qt, bh;
    bwd_cta_tile(static_cast<int>(blockIdx.x) / C::NH, n_qt, p, qt, bh);
    if (p.causal)
        qt = n_qt - 1 - qt;
    if (qt < 0)
        return;
    const int hh = bh % p.H, hb = bh / p.H;   // head and batch of this CTA's tiles
    const bool q3 = (p.maps3 >> BWD_MAP_Q) & 1, k3 = (p.maps3 >> BWD_MAP_K) & 1;   // 3-D tensor maps
    const bool v3 = (p.maps3 >> BWD_MAP_V) & 1, do3 = (p.maps3 >> BWD_MAP_DO) & 1;
    const int q0 = qt * C::RES;
    // key tiles this query tile visits (causal: up to its last row's key)
    const int n_kt_all = (p.Lk + C::STR - 1) / C::STR;
    const int last_row = min(q0 + C::RES - 1, p.Lq - 1);
    const int kt_end = p.causal ? min(min(last_row, p.Lk - 1) / C::STR + 1, n_kt_all) : n_kt_all;
    // under a sliding window the tile's first row sees nothing left of key q0 - window
    const int kt0 = p.window >= 0 ? min(max(0, q0 - p.window) / C::STR, kt_end) : 0;
    const int n_steps = kt_end - kt0;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::BAR_RES_FULL), 1);
        for (int s = 0; s < C::RING; ++s) {
            mbar_init(bar(C::BAR_STR_FULL + s), 1);
            mbar_init(bar(C::BAR_STR_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::BAR_SCORE_FULL + b), 1);
            mbar_init(bar(C::BAR_DP_FULL + b), 1);
            mbar_init(bar(C::BAR_GRAD_READY + b), C::EW);   // one arrival per elementwise warp
        }
        mbar_init(bar(C::BAR_DONE), 1);
        mbar_init(bar(C::BAR_RES_TMEM), C::EW);
        fence_mbar_init();
    }
    if (warp == C::WARP_MMA) {
        tmem_alloc(sbase + C::OFF_TMEM_SLOT, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sgen + C::OFF_TMEM_SLOT);

    if (warp == C::WARP_PRODUCER) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_do);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(bar(C::BAR_RES_FULL), 2 * C::RES_TILE);
#pragma unroll
            for (int c = 0; c < C::DB; ++c) {
                bwd_tma_load(sbase + C::OFF_RES0 + c * C::RES_BLOCK, &tm_q, q3, 64 * c, q0, bh, hh, hb,
                                 bar(C::BAR_RES_FULL));
                bwd_tma_load(sbase + C::OFF_RES1 + c * C::RES_BLOCK, &tm_do, do3, 64 * c, q0, bh, hh, hb,
                                 bar(C::BAR_RES_FULL));
            }
            bool ok = true;
            int issued = 0;
            for (int s = 0; s < n_steps && ok; ++s) {
                const int st = s % C::RING;
                if (s >= C::RING &&
                    !mbar_wait(bar(C::BAR_STR_EMPTY + st), ((s / C::RING) - 1) & 1, p.err, ERR_BWD_PRODUCER | 4,
                               p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                const int j0 = (kt0 + s) * C::STR;
                mbar_arrive_expect_tx(bar(C::BAR_STR_FULL + st), 2 * C::STR_TILE);
#pragma unroll
                for (int c = 0; c < C::DB; ++c) {
                    bwd_tma_load(sbase + C::OFF_STR0 + st * C::STR_TILE + c * C::STR_BLOCK, &tm_k, k3,
                                 64 * c, j0, bh, hh, hb, bar(C::BAR_STR_FULL + st));
                    bwd_tma_load(sbase + C::OFF_STR1 + st * C::STR_TILE + c * C::STR_BLOCK, &tm_v, v3,
                                 64 * c, j0, bh, hh, hb, bar(C::BAR_STR_FULL + st));
                }
                ++issued;
            }
            mbar_wait(bar(C::BAR_RES_FULL), 0, p.err, ERR_BWD_PRODUCER | 5, p.wait_limit_ns);
            for (int s = issued > C::RING ? issued - C::RING : 0; s < issued; ++s)
                mbar_wait(bar(C::BAR_STR_FULL + s % C::RING), (s / C::RING) & 1, p.err, ERR_BWD_PRODUCER | 6,
                          p.wait_limit_ns);
        }
        __syncwarp();
    } else if (warp == C::WARP_MMA) {
        // one elected lane runs the whole issue loop (waits, MMAs, commits)
        if (elect_one()) {
            const uint64_t desc_k = sdesc_sw128(sbase + C::OFF_STR0, 16, 1024);
            const uint64_t desc_v = sdesc_sw128(sbase + C::OFF_STR1, 16, 1024);
            const uint64_t desc_k_mn =
                sdesc_sw128(sbase + C::OFF_STR0 + dh * (C::DH / 64) * C::STR_BLOCK, C::STR_BLOCK, 1024);
            // the resident Q and dO tiles as K-major A operands (when they stay in shared memory)
            const uint64_t desc_q = sdesc_sw128(sbase + C::OFF_RES0, 16, 1024);
            const uint64_t desc_do = sdesc_sw128(sbase + C::OFF_RES1, 16, 1024);
            // Q and dO copied into TMEM by the elementwise warps, or landed in shared memory
            bool ok = C::RES_IN_TMEM ? lone_wait(bar(C::BAR_RES_TMEM), 0, p.err, ERR_BWD_MMA | 5, p.wait_limit_ns)
                                     : lone_wait(bar(C::BAR_RES_FULL), 0, p.err, ERR_BWD_MMA | 5, p.wait_limit_ns);
            tc_fence_after();
            const auto stage_off = [](int st) { return static_cast<uint64_t>((st * C::STR_TILE) >> 4); };
            // S(b) = Q K^T for step s, once the step's tiles have landed
            auto issue_s = [&](int s) -> bool {
                const int st = s % C::RING, b = s & 1;
                if (!lone_wait(bar(C::BAR_STR_FULL + st), (s / C::RING) & 1, p.err, ERR_BWD_MMA | 6,
                               p.wait_limit_ns))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < C::D / 16; ++kk) {
                    const uint64_t to = static_cast<uint64_t>(((kk >> 2) * C::STR_BLOCK + (kk & 3) * 32) >> 4);
                    if constexpr (C::RES_IN_TMEM)
                        mma_ts(tmem + TM_S + b * C::STR, tmem + TM_QA + kk * 8, desc_k + stage_off(st) + to,
                               C::IDESC_PAIR, kk > 0 ? 1u : 0u);
                    else
                        mma_ss(tmem + TM_S + b * C::STR,
                               desc_q + static_cast<uint64_t>(((kk >> 2) * C::RES_BLOCK + (kk & 3) * 32) >> 4),
                               desc_k + stage_off(st) + to, C::IDESC_PAIR, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::BAR_SCORE_FULL + b));
                return true;
            };
            // dP(b) = dO V^T for step s (issued after issue_s(s), which waited for the tiles)
            auto issue_dp = [&](int s) {
                const int st = s % C::RING, b = s & 1;
#pragma unroll
                for (int kk = 0; kk < C::D / 16; ++kk) {
                    const uint64_t to = static_cast<uint64_t>(((kk >> 2) * C::STR_BLOCK + (kk & 3) * 32) >> 4);
                    if constexpr (C::RES_IN_TMEM)
                        mma_ts(tmem + TM_DP + b * C::STR, tmem + TM_DOA + kk * 8, desc_v + stage_off(st) + to,
                               C::IDESC_PAIR, kk > 0 ? 1u : 0u);
                    else
                        mma_ss(tmem + TM_DP + b * C::STR,
                               desc_do + static_cast<uint64_t>(((kk >> 2) * C::RES_BLOCK + (kk & 3) * 32) >> 4),
                               desc_v + stage_off(st) + to, C::IDESC_PAIR, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::BAR_DP_FULL + b));
            };
            // dQ += dS K for step s.  The bf16 pairs of key columns 16 kk .. 16 kk + 15
            // sit 8 columns each from the start of the 32 columns of the elementwise
            // warp that owns those keys, where it wrote them.
            auto issue_grad = [&](int s) -> bool {
                const int st = s % C::RING, b = s & 1;
                if (!lone_wait(bar(C::BAR_GRAD_READY + b), (s >> 1) & 1, p.err, ERR_BWD_MMA | 7, p.wait_limit_ns))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < C::STR / 16; ++kk) {
                    const int pc = 32 * (kk >> 1) + 8 * (kk & 1);   // pair column of these keys
                    mma_ts(tmem + TM_DQ, tmem + TM_S + b * C::STR + pc,
                           desc_k_mn + stage_off(st) + static_cast<uint64_t>((kk * 16 * 128) >> 4), C::IDESC_GRAD,
                           (s > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(C::BAR_STR_EMPTY + st));
                return true;
            };
            // S and dP are committed separately so that the elementwise warps start on
            // the exponentials while dP is still being computed
            for (int s = 0; s < C::LA && s < n_steps && ok; ++s) {
                ok = issue_s(s);
                if (ok)
                    issue_dp(s);
            }
            for (int s = 0; s < n_steps && ok; ++s) {
                ok = issue_grad(s);
                if (ok && s + C::LA < n_steps)
                    ok = issue_s(s + C::LA);
                if (ok && s + C::LA < n_steps)
                    issue_dp(s + C::LA);
            }
            mma_commit(bar(C::BAR_DONE));
            lone_wait(bar(C::BAR_DONE), 0, p.err, ERR_BWD_MMA | 8, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ elementwise warps
        // Two warps per 32-lane TMEM quarter: `half` 0 takes key columns 0..31 of
        // every step, `half` 1 columns 32..63; each stores half of dQ's columns.  With
        // one warp per quarter (32-column steps) it takes them all.
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;         // query row within the tile (TMEM lane)
        const int qi = q0 + row;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int c0 = 32 * half;                    // this warp's first key column of a step
        const float c2 = p.scale_log2;
        const bool live = qi < p.Lq;
        const float *stat = p.stats +
                            (static_cast<size_t>(bh) * p.n_stat_tiles + (live ? qi : 0) / BWD_STAT_ROWS) * 2 * BWD_STAT_ROWS +
                            (live ? qi : 0) % BWD_STAT_ROWS;
        const float lse2 = live ? -stat[0] : INFINITY;
        const float dl = live ? -stat[BWD_STAT_ROWS] : 0.f;
        // keys lo <= j < lim are visible to this row
        const int lim = p.causal ? min(qi + 1, p.Lk) : p.Lk;
        const int lo = p.window >= 0 ? qi - p.window : 0;
        // this row of Q (half 0) or of dO (half 1) into TMEM, as a score MMA's A operand
        bool ok = !C::RES_IN_TMEM || warp_wait_all(bar(C::BAR_RES_FULL), 0, p.err, ERR_BWD_ELEM | 6, p.wait_limit_ns);
        if (ok && C::RES_IN_TMEM) {
            // two warps per quarter: one copies Q, the other dO; one warp per quarter: both
            if (half == 0)
                copy_row_to_tmem<C::DB, C::RES_BLOCK>(sbase + C::OFF_RES0, row, tmem + lane_base + TM_QA);
            if (half == 1 || C::EW == 4)
                copy_row_to_tmem<C::DB, C::RES_BLOCK>(sbase + C::OFF_RES1, row, tmem + lane_base + TM_DOA);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(C::BAR_RES_TMEM));
        }
        const uint64_t c2x2 = f32x2(c2, c2);
        const uint64_t nl2 = f32x2(-lse2, -lse2);
        const uint64_t nd2 = f32x2(-dl, -dl);
        const uint64_t zero2 = 0;
        for (int s = 0; s < n_steps && ok; ++s) {
            const int b = s & 1;
            ok = warp_wait_all(bar(C::BAR_SCORE_FULL + b), (s >> 1) & 1, p.err, ERR_BWD_ELEM | 3, p.wait_limit_ns);
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t a_s = tmem + lane_base + TM_S + b * C::STR + c0;
            const uint32_t a_dp = tmem + lane_base + TM_DP + b * C::STR + c0;
            const int j0 = (kt0 + s) * C::STR + c0;  // this warp's first key
            // key columns at or past lim (and, under a window, before lo) are masked; only
            // a tile reaching past those bounds for some row of this warp needs the test
            const bool need_mask = __any_sync(0xffffffffu, j0 + 32 > lim || j0 < lo);
            // P = 2^(S c - lse2) for this warp's 32 keys, before dP is needed
            float pv[32];
            {
                uint32_t rs[32];
                tmem_ld32(a_s, rs);
                tmem_ld_wait(rs);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float x0, x1;
                    unpack_f32x2(fma_f32x2(f32x2(__uint_as_float(rs[e]), __uint_as_float(rs[e + 1])), c2x2, nl2), x0,
                                 x1);
                    pv[e] = ex2_approx(x0);
                    pv[e + 1] = ex2_approx(x1);
                }
            }
            // dS = P (dP - Delta), once dP is in
            ok = warp_wait_all(bar(C::BAR_DP_FULL + b), (s >> 1) & 1, p.err, ERR_BWD_ELEM | 9, p.wait_limit_ns);
            if (!ok)
                break;
            tc_fence_after();
            uint32_t rd[32];
            tmem_ld32(a_dp, rd);
            tmem_ld_wait(rd);
            float dv[32];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const uint64_t diff = add_f32x2(f32x2(__uint_as_float(rd[e]), __uint_as_float(rd[e + 1])), nd2);
                unpack_f32x2(fma_f32x2(f32x2(pv[e], pv[e + 1]), diff, zero2), dv[e], dv[e + 1]);
            }
            if (need_mask) {
                const int hi = lim - j0;             // columns c >= hi are masked
                const int lo_c = lo - j0;            // and columns c < lo_c
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    dv[e] = (e >= hi || e < lo_c) ? 0.f : dv[e];
            }
            // dS as bf16 pairs over the first 16 of this warp's 32 columns of the S buffer
            uint32_t dw[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2)
                dw[e / 2] = bwd_pack(dv[e], dv[e + 1]);
            tmem_st16(a_s, dw);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(C::BAR_GRAD_READY + b));
        }
        // epilogue: scale * dQ, columns dh * DH + [half * W, (half + 1) * W) of this row, W the
        // columns per warp of a lane quarter (DH / 2 with two warps, DH with one)
        constexpr int W = C::DH / (C::EW / 4);
        if (ok && warp_wait_all(bar(C::BAR_DONE), 0, p.err, ERR_BWD_ELEM | 4, p.wait_limit_ns)) {
            tc_fence_after();
            store_acc_row<W>(tmem + lane_base + TM_DQ + half * W, p.scale,
                             p.dq + static_cast<long long>(hb) * p.dq_sb + static_cast<long long>(hh) * p.dq_sh +
                                 static_cast<long long>(live ? qi : 0) * p.dq_sl + dh * C::DH + half * W,
                             live);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == C::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace fa2
