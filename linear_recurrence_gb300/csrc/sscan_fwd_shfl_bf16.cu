// bfloat16-I/O instantiations of the TMA-fed selective-scan kernel with
// outputs summed by warp shuffles (plain scan, single and local passes).
#define SSCAN_TMA_IMPL
#include "sscan_fwd_tma.cuh"

namespace sscan {

using UnitT = bf16;
SSCAN_DEFINE_SHFL_UNIT(bf16)

}  // namespace sscan
