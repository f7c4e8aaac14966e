// Forward kernel instantiation for e4m3 Q, K, V at head dimension 128: two 128-row
// Q tiles per CTA (one S buffer each), K/V tiles of 128 rows, a 4-stage ring, one
// softmax warp per row; S = Q K^T and O += P V run as kind::f8f6f4 MMAs with P
// rounded to e4m3 in TMEM.  Byte-wide tiles leave room for the deeper ring (Q 32 KB,
// ring 128 KB, O staging 32 KB); TMEM is laid out as for bf16 (O 2 x 128 columns,
// S 2 x 128, P over the first 32 columns of its S buffer).
#include "fa2_launch.cuh"

namespace fa2 {

#ifndef FA2_FP8_KS
#define FA2_FP8_KS 4
#endif

using CfgFp8D128 = FwdCfg<128, 128, 2, FA2_FP8_KS, 1, 1, 0, 0, 1>;

fa2_status launch_fwd_fp8_d128(const LaunchArgs &a) { return launch_fwd<CfgFp8D128>(a); }

}  // namespace fa2
