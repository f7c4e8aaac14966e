// Forward kernel instantiation for head dimension 128: two 128-row Q tiles per
// CTA (one S buffer each), K/V tiles of 128 rows, a 2-stage ring, one softmax
// warp per row.
// Q tiles + ring fit the 227 KB shared-memory budget and the O accumulators +
// S buffers fit the 512 TMEM columns.  Defaults picked by measured c2/c3/c5
// throughput on GB300.
#include "fa2_launch.cuh"

namespace fa2 {

// Tile configuration (K/V rows, Q tiles per CTA, ring stages, warps per row,
// S buffers per Q tile, Q kept in TMEM);
// overridable at compile time for tuning sweeps.
#ifndef FA2_D128_BN
#define FA2_D128_BN 128
#endif
#ifndef FA2_D128_NQ
#define FA2_D128_NQ 2
#endif
#ifndef FA2_D128_KS
#define FA2_D128_KS 2
#endif
#ifndef FA2_D128_NS
#define FA2_D128_NS (FA2_D128_NQ == 1 ? 2 : 1)
#endif
#ifndef FA2_D128_QT
#define FA2_D128_QT 0
#endif
#ifndef FA2_D128_CS
#define FA2_D128_CS 1
#endif

using CfgD128 = FwdCfg<128, FA2_D128_BN, FA2_D128_NQ, FA2_D128_KS, FA2_D128_CS, FA2_D128_NS,
                      FA2_D128_QT>;

fa2_status launch_fwd_d128(const LaunchArgs &a) { return launch_fwd<CfgD128>(a); }

size_t workspace_bytes_d128(int B, int H, int Lq, int Lk, int causal, int num_sms, int policy)
{
    return workspace_bytes_for<CfgD128>(B, H, Lq, Lk, causal, num_sms, policy);
}

}  // namespace fa2
