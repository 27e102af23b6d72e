// float32-I/O instantiations of the TMA-fed selective-scan kernel.
#define SSCAN_TMA_IMPL
#include "sscan_fwd_tma.cuh"

namespace sscan {

using UnitT = float;
SSCAN_DEFINE_TMA_UNIT(f32)

}  // namespace sscan
