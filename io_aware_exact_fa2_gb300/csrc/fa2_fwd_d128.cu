// Forward kernel instantiation for head dimension 128: 2 Q tile(s) of 128 rows
// per CTA, K/V tiles of 128 rows, a 2-stage K/V ring (sized so Q tiles + ring
// fit the 227 KB shared-memory budget and S/P + O fit the 512 TMEM columns).
#include "fa2_launch.cuh"

namespace fa2 {

fa2_status launch_fwd_d128(const LaunchArgs &a) { return launch_fwd<FwdCfg<128, 128, 2, 2>>(a); }

}  // namespace fa2
