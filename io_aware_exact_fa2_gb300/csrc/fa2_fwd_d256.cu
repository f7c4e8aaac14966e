// Forward kernel instantiation for head dimension 256: 1 Q tile(s) of 128 rows
// per CTA, K/V tiles of 64 rows, a 2-stage K/V ring (sized so Q tiles + ring
// fit the 227 KB shared-memory budget and S/P + O fit the 512 TMEM columns).
#include "fa2_launch.cuh"

namespace fa2 {

fa2_status launch_fwd_d256(const LaunchArgs &a) { return launch_fwd<FwdCfg<256, 64, 1, 2>>(a); }

}  // namespace fa2
