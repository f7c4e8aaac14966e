// fa2_fwd_kernel.cuh -- exact FlashAttention-2 forward for sm_103a.
//
// The method (Olowookere, "FlashAttention-2 from scratch with a custom Triton
// kernel", sections "The core idea: making attention IO-aware" and "Running
// max m_i and running normaliser"; "Chapter 08: Flash Attention -- blocked
// attention", sections 1-5): one CTA owns NQ query tiles of 128 rows of one
// (batch, head); the tiles stay on chip while K/V tiles of BN rows stream
// through shared memory; per row the kernel keeps a running max m, a running
// normaliser l and an unnormalised accumulator O, rescales O and l when m
// grows, and divides by l once at the end (deferred normalisation).  Scores
// are taken to base 2 (scale * log2 e folded into one FMA, then exp2), the
// log-sum-exp is written per row, causal key tiles above the diagonal are
// never visited and only tiles that straddle the diagonal (or the key tail)
// pay for element masking.
//
// GB300 mapping (prior art on the pages is Triton on A100/Ada; this is not a
// translation of it):
//   * TMA (cp.async.bulk.tensor, 128B swizzle) moves Q once and K/V per tile
//     into a KS-stage shared-memory ring guarded by mbarriers.
//   * One thread issues tcgen05.mma: S = Q K^T into TMEM (fp32), then
//     O += P V with P read straight from TMEM (bf16, aliasing S) and V from
//     shared memory (MN-major operand: no transpose pass).
//   * One warpgroup per Q tile (thread <-> row, TMEM lane == row) runs the
//     online softmax out of TMEM, writes P back to TMEM, and rescales O in
//     TMEM only when a row's max grows by more than 2^8 (the stale max is
//     kept otherwise, which is exact because l and LSE use the same max).
//   * The epilogue multiplies by 1/l, packs bf16 into the (now free) Q tile
//     in the swizzled layout and stores it with TMA (one 32-row box per warp;
//     rows >= Lq are clipped by the tensor bounds); LSE goes out as
//     coalesced fp32 stores.
//   * Every inter-warp wait is bounded in time; a wait that runs out records
//     a code in a device error word and the CTA winds down.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "sm103_ptx.cuh"

namespace fa2 {

struct FwdParams {
    float *lse;                 // fp32 [B*H, Lq]
    int *err;                   // device error word
    unsigned long long wait_limit_ns;
    int Lq, Lk;
    int BH;                     // B * H
    int n_qgroups;              // ceil(Lq / (NQ * 128))
    int causal;
    float scale_log2;           // scale * log2(e), > 0
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

template <int D_, int BN_, int NQ_, int KS_>
struct FwdCfg {
    static constexpr int D = D_;     // head dimension
    static constexpr int BN = BN_;   // K/V rows per tile
    static constexpr int NQ = NQ_;   // 128-row Q tiles per CTA (one softmax warpgroup each)
    static constexpr int KS = KS_;   // K/V ring stages
    static constexpr int BM = 128;   // Q rows per tile = TMEM lanes = MMA M
    static constexpr int NS = (NQ == 1) ? 2 : 1;  // S/P TMEM buffers per Q tile
    static constexpr int DB = D / 64;             // 64-column (128-byte) swizzle blocks
    static constexpr int Q_BLOCK = BM * 128;
    static constexpr int KV_BLOCK = BN * 128;
    static constexpr int Q_TILE = DB * Q_BLOCK;
    static constexpr int KV_TILE = DB * KV_BLOCK;

    // shared memory (offsets from a 1024-byte aligned base)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + NQ * Q_TILE;
    static constexpr int OFF_V = OFF_K + KS * KV_TILE;
    static constexpr int OFF_BAR = OFF_V + KS * KV_TILE;
    static constexpr int BAR_Q = 0;
    static constexpr int BAR_K_FULL = 1;
    static constexpr int BAR_K_EMPTY = BAR_K_FULL + KS;
    static constexpr int BAR_V_FULL = BAR_K_EMPTY + KS;
    static constexpr int BAR_V_EMPTY = BAR_V_FULL + KS;
    static constexpr int BAR_S_FULL = BAR_V_EMPTY + KS;   // [NQ][NS]
    static constexpr int BAR_O_DONE = BAR_S_FULL + NQ * NS;  // [NQ]
    static constexpr int BAR_P_READY = BAR_O_DONE + NQ;      // [NQ]
    static constexpr int BAR_DRAIN = BAR_P_READY + NQ;
    static constexpr int NUM_BARS = BAR_DRAIN + 1;
    static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_TMEM_SLOT + 16 + 1024;  // + slack for base alignment

    // tensor memory columns
    static constexpr int TM_O = 0;        // O of tile t: columns [t*D, (t+1)*D)
    static constexpr int TM_S = NQ * D;   // S/P buffer (t, b): TM_S + (t*NS + b)*BN
    static constexpr int TMEM_USED = NQ * D + NQ * NS * BN;
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64
                                   : TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;

    // warp roles
    static constexpr int NUM_SOFTMAX_WARPS = 4 * NQ;
    static constexpr int WARP_PRODUCER = NUM_SOFTMAX_WARPS;
    static constexpr int WARP_MMA = NUM_SOFTMAX_WARPS + 1;
    static constexpr int NUM_THREADS = 32 * (NUM_SOFTMAX_WARPS + 2);

    static constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(BM, BN, false, false);
    static constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(BM, D, false, true);

    static_assert(D % 64 == 0 && D >= 64 && D <= 256, "D must be 64, 128 or 256");
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be a multiple of 64 in [64, 256]");
    static_assert(TMEM_USED <= 512, "TMEM budget exceeded");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
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

// All lanes wait (bounded); the warp agrees on the outcome so warp-collective
// tcgen05 instructions are executed by all lanes or by none.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int *err, int code,
                                          unsigned long long limit)
{
    const bool ok = ptx::mbar_wait(bar, parity, err, code, limit);
    return __all_sync(0xffffffffu, ok);
}

template <class C>
__global__ void __launch_bounds__(C::NUM_THREADS, 1)
    fa2_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const FwdParams p)
{
    using namespace ptx;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work unit: (query group, batch*head).  Causal: heaviest groups first.
    int qg, bh;
    if (p.causal) {
        qg = p.n_qgroups - 1 - static_cast<int>(blockIdx.x) / p.BH;
        bh = static_cast<int>(blockIdx.x) % p.BH;
    } else {
        bh = static_cast<int>(blockIdx.x) / p.n_qgroups;
        qg = static_cast<int>(blockIdx.x) % p.n_qgroups;
    }
    const int q0 = qg * (C::NQ * C::BM);
    // K/V tiles visited by Q tile t (computed, not indexed, to keep it in registers)
    auto n_of = [&](int t) { return kv_tiles_for(q0 + t * C::BM, p.Lq, p.Lk, p.causal, C::BN); };
    int n_max = 0;
#pragma unroll
    for (int t = 0; t < C::NQ; ++t)
        n_max = max(n_max, n_of(t));
    // the last Q tile (highest t) that reads K/V tile j
    auto last_user = [&](int j) {
        int u = 0;
#pragma unroll
        for (int t = 0; t < C::NQ; ++t)
            if (j < n_of(t))
                u = t;
        return u;
    };
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };

    // ---- setup: barriers, TMEM
    if (threadIdx.x == 0) {
        mbar_init(bar(C::BAR_Q), 1);
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(bar(C::BAR_K_FULL + s), 1);
            mbar_init(bar(C::BAR_K_EMPTY + s), 1);
            mbar_init(bar(C::BAR_V_FULL + s), 1);
            mbar_init(bar(C::BAR_V_EMPTY + s), 1);
        }
        for (int i = 0; i < C::NQ * C::NS; ++i)
            mbar_init(bar(C::BAR_S_FULL + i), 1);
        for (int t = 0; t < C::NQ; ++t) {
            mbar_init(bar(C::BAR_O_DONE + t), 1);
            mbar_init(bar(C::BAR_P_READY + t), 128);
        }
        mbar_init(bar(C::BAR_DRAIN), 1);
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

    if (warp == C::WARP_PRODUCER) {
        // ================================================== TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_o);
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            uint32_t q_bytes = 0;
#pragma unroll
            for (int t = 0; t < C::NQ; ++t)
                if (n_of(t) > 0)
                    q_bytes += C::Q_TILE;
            mbar_arrive_expect_tx(bar(C::BAR_Q), q_bytes);
#pragma unroll
            for (int t = 0; t < C::NQ; ++t)
                if (n_of(t) > 0)
#pragma unroll
                    for (int c = 0; c < C::DB; ++c)
                        tma_load_3d_hint(sbase + C::OFF_Q + t * C::Q_TILE + c * C::Q_BLOCK, &tm_q, 64 * c,
                                         q0 + t * C::BM, bh, bar(C::BAR_Q), pol_q);
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < n_max; ++j) {
                const int s = j % C::KS;
                const uint32_t ph = (j / C::KS) & 1;
                if (!mbar_wait(bar(C::BAR_K_EMPTY + s), ph ^ 1u, p.err, ERR_PRODUCER | 1, p.wait_limit_ns))
                    break;
                mbar_arrive_expect_tx(bar(C::BAR_K_FULL + s), C::KV_TILE);
#pragma unroll
                for (int c = 0; c < C::DB; ++c)
                    tma_load_3d_hint(sbase + C::OFF_K + s * C::KV_TILE + c * C::KV_BLOCK, &tm_k, 64 * c,
                                     j * C::BN, bh, bar(C::BAR_K_FULL + s), pol_kv);
                k_issued = j + 1;
                if (!mbar_wait(bar(C::BAR_V_EMPTY + s), ph ^ 1u, p.err, ERR_PRODUCER | 2, p.wait_limit_ns))
                    break;
                mbar_arrive_expect_tx(bar(C::BAR_V_FULL + s), C::KV_TILE);
#pragma unroll
                for (int c = 0; c < C::DB; ++c)
                    tma_load_3d_hint(sbase + C::OFF_V + s * C::KV_TILE + c * C::KV_BLOCK, &tm_v, 64 * c,
                                     j * C::BN, bh, bar(C::BAR_V_FULL + s), pol_kv);
                v_issued = j + 1;
            }
            // Before the CTA may exit, every load this thread started must have landed
            // (immediate on the normal path: all of them were consumed).
            mbar_wait(bar(C::BAR_Q), 0, p.err, ERR_DRAIN | 1, p.wait_limit_ns);
            for (int j = max(0, k_issued - C::KS); j < k_issued; ++j)
                mbar_wait(bar(C::BAR_K_FULL + j % C::KS), (j / C::KS) & 1, p.err, ERR_DRAIN | 2,
                          p.wait_limit_ns);
            for (int j = max(0, v_issued - C::KS); j < v_issued; ++j)
                mbar_wait(bar(C::BAR_V_FULL + j % C::KS), (j / C::KS) & 1, p.err, ERR_DRAIN | 3,
                          p.wait_limit_ns);
        }
        __syncwarp();
    } else if (warp == C::WARP_MMA) {
        // ================================================== MMA issuer (one thread)
        if (lane == 0) {
            bool ok = mbar_wait(bar(C::BAR_Q), 0, p.err, ERR_MMA | 1, p.wait_limit_ns);
            tc_fence_after();

            // S(t, j) = Q_t K_j^T  into S/P buffer (t, j % NS)
            auto issue_s = [&](int t, int j) -> bool {
                const int s = j % C::KS;
                if (!mbar_wait(bar(C::BAR_K_FULL + s), (j / C::KS) & 1, p.err, ERR_MMA | 2, p.wait_limit_ns))
                    return false;
                tc_fence_after();
                const uint32_t d = tmem + C::TM_S + (t * C::NS + j % C::NS) * C::BN;
                const uint32_t qa = sbase + C::OFF_Q + t * C::Q_TILE;
                const uint32_t kb = sbase + C::OFF_K + s * C::KV_TILE;
#pragma unroll
                for (int kk = 0; kk < C::D / 16; ++kk) {
                    const uint32_t oq = (kk >> 2) * C::Q_BLOCK + (kk & 3) * 32;
                    const uint32_t ok_ = (kk >> 2) * C::KV_BLOCK + (kk & 3) * 32;
                    mma_ss(d, sdesc_sw128(qa + oq, 16, 1024), sdesc_sw128(kb + ok_, 16, 1024), C::IDESC_S,
                           kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::BAR_S_FULL + t * C::NS + j % C::NS));
                if (last_user(j) == t)
                    mma_commit(bar(C::BAR_K_EMPTY + s));
                return true;
            };
            // O_t (+)= P(t, j) V_j, P read from TMEM
            auto issue_pv = [&](int t, int j) -> bool {
                const int s = j % C::KS;
                if (!mbar_wait(bar(C::BAR_P_READY + t), j & 1, p.err, ERR_MMA | 3, p.wait_limit_ns))
                    return false;
                if (!mbar_wait(bar(C::BAR_V_FULL + s), (j / C::KS) & 1, p.err, ERR_MMA | 4, p.wait_limit_ns))
                    return false;
                tc_fence_after();
                const uint32_t d = tmem + C::TM_O + t * C::D;
                const uint32_t a = tmem + C::TM_S + (t * C::NS + j % C::NS) * C::BN;
                const uint32_t vb = sbase + C::OFF_V + s * C::KV_TILE;
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)
                    mma_ts(d, a + kk * 8, sdesc_sw128(vb + kk * 2048, C::KV_BLOCK, 1024), C::IDESC_PV,
                           (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(C::BAR_O_DONE + t));
                if (last_user(j) == t)
                    mma_commit(bar(C::BAR_V_EMPTY + s));
                return true;
            };

            // Issue order: S for the first NS tiles of every Q tile, then per K/V
            // tile j and Q tile t: PV(t, j) followed by S(t, j + NS), which reuses
            // the TMEM buffer PV(t, j) just read (tcgen05 ops execute in order).
            for (int b = 0; b < C::NS && ok; ++b)
                for (int t = 0; t < C::NQ && ok; ++t)
                    if (b < n_of(t))
                        ok = issue_s(t, b);
            for (int j = 0; j < n_max && ok; ++j)
                for (int t = 0; t < C::NQ && ok; ++t)
                    if (j < n_of(t)) {
                        ok = issue_pv(t, j);
                        if (ok && j + C::NS < n_of(t))
                            ok = issue_s(t, j + C::NS);
                    }
            // drain: every MMA issued above has completed before TMEM can be released
            mma_commit(bar(C::BAR_DRAIN));
            mbar_wait(bar(C::BAR_DRAIN), 0, p.err, ERR_DRAIN | 4, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ================================================== softmax warpgroups
        const int t = warp >> 2;        // Q tile
        const int quarter = warp & 3;   // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const int q0_t = q0 + t * C::BM;
        const int grow = q0_t + row;    // query index
        const int n = n_of(t);
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t o_addr = tmem + lane_base + C::TM_O + t * C::D;
        const float c2 = p.scale_log2;
        float m_use = -INFINITY;   // running max (log2 domain, possibly stale by < 2^THRESHOLD)
        float l = 0.f;             // running normaliser of the fp32 weights (for LSE)
        float l_o = 0.f;           // running normaliser of the bf16 weights the PV MMA sees (for O)
        bool ok = true;

        for (int j = 0; j < n && ok; ++j) {
            const int b = j % C::NS;
            ok = warp_wait(bar(C::BAR_S_FULL + t * C::NS + b), (j / C::NS) & 1, p.err, ERR_SOFTMAX | 1,
                           p.wait_limit_ns);
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t s_addr = tmem + lane_base + C::TM_S + (t * C::NS + b) * C::BN;

            float s[C::BN];
            {
                uint32_t r[C::BN / 32][32];
#pragma unroll
                for (int q = 0; q < C::BN / 32; ++q)
                    tmem_ld32(s_addr + 32 * q, r[q]);
#pragma unroll
                for (int q = 0; q < C::BN / 32; ++q)
                    tmem_ld_wait(r[q]);
#pragma unroll
                for (int q = 0; q < C::BN / 32; ++q)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        s[32 * q + i] = __uint_as_float(r[q][i]);
            }

            // mask: key tail (j >= Lk) and, on tiles crossing the diagonal, causal j > i
            const int k0 = j * C::BN;
            if ((p.causal && k0 + C::BN - 1 > q0_t) || (k0 + C::BN > p.Lk)) {
                const int lim = p.causal ? min(grow + 1, p.Lk) : p.Lk;  // keys < lim are visible
#pragma unroll
                for (int c = 0; c < C::BN; ++c)
                    if (k0 + c >= lim)
                        s[c] = -INFINITY;
            }

            // row max of this tile, in the scaled log2 domain
            float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
            for (int c = 4; c < C::BN; c += 4) {
                mx0 = fmaxf(mx0, s[c]);
                mx1 = fmaxf(mx1, s[c + 1]);
                mx2 = fmaxf(mx2, s[c + 2]);
                mx3 = fmaxf(mx3, s[c + 3]);
            }
            const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c2;

            // The first tile always holds key 0, which every row may see, so m_tile is
            // finite there; later tiles keep the stale max unless it grows a lot.
            float alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_use = m_tile;
            } else if (m_tile > m_use + RESCALE_THRESHOLD) {
                alpha = ex2_approx(m_use - m_tile);
                m_use = m_tile;
                rescale = true;
            }

            // p = 2^(s * scale * log2e - m); masked entries give 2^-inf = 0.  P goes to
            // TMEM as bf16 (two per 32-bit column, over the first BN/2 columns of the S
            // buffer).  Two normalisers are kept: l sums the fp32 p (LSE needs the exact
            // sum) and l_o sums the bf16-rounded p that the PV MMA multiplies, so O's
            // numerator and denominator use the same weights -- with one dominant key
            // the rounding of its weight then cancels instead of showing up in O.
            const float neg_m = -m_use;
            float ls0 = 0.f, ls1 = 0.f, lr0 = 0.f, lr1 = 0.f;
            {
                uint32_t pk[C::BN / 64][32];
#pragma unroll
                for (int c = 0; c < C::BN; c += 2) {
                    const float p0 = ex2_approx(fmaf(s[c], c2, neg_m));
                    const float p1 = ex2_approx(fmaf(s[c + 1], c2, neg_m));
                    const uint32_t w = pack_bf16x2(p0, p1);
                    pk[(c / 2) / 32][(c / 2) % 32] = w;
                    ls0 += p0;
                    ls1 += p1;
                    lr0 += __uint_as_float(w << 16);
                    lr1 += __uint_as_float(w & 0xFFFF0000u);
                }
#pragma unroll
                for (int q = 0; q < C::BN / 64; ++q)
                    tmem_st32(s_addr + 32 * q, pk[q]);
            }
            l = l * alpha + (ls0 + ls1);
            l_o = l_o * alpha + (lr0 + lr1);

            // rescale O once the previous PV has landed (only warps with a grown max)
            if (j > 0) {
                ok = warp_wait(bar(C::BAR_O_DONE + t), (j - 1) & 1, p.err, ERR_SOFTMAX | 2, p.wait_limit_ns);
                if (!ok)
                    break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                    for (int cc = 0; cc < C::D / 32; ++cc) {
                        uint32_t r[32];
                        tmem_ld32(o_addr + 32 * cc, r);
                        tmem_ld_wait(r);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(o_addr + 32 * cc, r);
                    }
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(C::BAR_P_READY + t));
        }

        // ---- epilogue: O / l -> bf16 -> swizzled smem (the Q tile) -> TMA store; LSE
        if (ok && n > 0) {
            ok = warp_wait(bar(C::BAR_O_DONE + t), (n - 1) & 1, p.err, ERR_SOFTMAX | 3, p.wait_limit_ns);
            if (ok) {
                tc_fence_after();
                const float inv_l = 1.f / l_o;
                const float lse = (m_use + lg2_approx(l)) * LN2;
                const uint32_t stage = sbase + C::OFF_Q + t * C::Q_TILE;
#pragma unroll 1
                for (int cc = 0; cc < C::D / 32; ++cc) {
                    uint32_t r[32];
                    tmem_ld32(o_addr + 32 * cc, r);
                    tmem_ld_wait(r);
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
                    const uint32_t row_addr = stage + (cc >> 1) * C::Q_BLOCK + row * 128;
                    const int chunk0 = (cc & 1) * 4;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st_shared_v4(row_addr + (((chunk0 + q) ^ (row & 7)) << 4), w[4 * q], w[4 * q + 1],
                                     w[4 * q + 2], w[4 * q + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                const int r0 = q0_t + quarter * 32;
                if (lane == 0 && r0 < p.Lq) {
#pragma unroll
                    for (int c = 0; c < C::DB; ++c)
                        tma_store_3d(&tm_o, 64 * c, r0, bh, stage + c * C::Q_BLOCK + quarter * 32 * 128);
                    tma_store_commit();
                    tma_store_wait_read_all();
                }
                __syncwarp();
                if (grow < p.Lq)
                    p.lse[static_cast<size_t>(bh) * p.Lq + grow] = lse;
            }
        }
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
