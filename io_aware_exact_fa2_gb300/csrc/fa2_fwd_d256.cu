// Forward kernel instantiation for head dimension 256: one 128-row Q tile per
// CTA with two S buffers, K/V tiles of 64 rows, a 2-stage ring, one softmax
// warp per row, and Q copied into TMEM so that S = Q K^T reads A from TMEM
// (an N = 64 MMA with both operands in shared memory spends most of its time
// loading A).
// Q tile + ring fit the 227 KB shared-memory budget; O (256 columns), the two
// S buffers (128) and Q (128) fill the 512 TMEM columns.  Defaults picked by
// measured c5 throughput on GB300.
#include "fa2_launch.cuh"

namespace fa2 {

// Tile configuration (K/V rows, Q tiles per CTA, ring stages, warps per row,
// S buffers per Q tile, Q kept in TMEM, P in two terms);
// overridable at compile time for tuning sweeps.
#ifndef FA2_D256_BN
#define FA2_D256_BN 64
#endif
#ifndef FA2_D256_NQ
#define FA2_D256_NQ 1
#endif
#ifndef FA2_D256_KS
#define FA2_D256_KS 2
#endif
#ifndef FA2_D256_NS
#define FA2_D256_NS (FA2_D256_NQ == 1 ? 2 : 1)
#endif
#ifndef FA2_D256_QT
#define FA2_D256_QT 1
#endif
#ifndef FA2_D256_CS
#define FA2_D256_CS 1
#endif
// P as two bf16 terms (weight and residual): keeps O within the bf16 output's own
// rounding where two or three keys dominate a row, at the price of a second PV MMA
#ifndef FA2_D256_P2
#define FA2_D256_P2 (FA2_D256_CS == 1)
#endif

using CfgD256 = FwdCfg<256, FA2_D256_BN, FA2_D256_NQ, FA2_D256_KS, FA2_D256_CS, FA2_D256_NS,
                      FA2_D256_QT, FA2_D256_P2>;

fa2_status launch_fwd_d256(const LaunchArgs &a) { return launch_fwd<CfgD256>(a); }

size_t workspace_bytes_d256(int B, int H, int Lq, int Lk, int causal, int num_sms, int policy)
{
    return workspace_bytes_for<CfgD256>(B, H, Lq, Lk, causal, num_sms, policy);
}

}  // namespace fa2
