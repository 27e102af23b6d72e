// float32-I/O instantiations of the TMA-fed selective-scan kernel: the delta bias / softplus / gate options.
#define SSCAN_TMA_IMPL
#include "sscan_fwd_tma.cuh"

namespace sscan {

using UnitT = float;
constexpr int UnitOPT = 1;
SSCAN_DEFINE_TMA_UNIT(f32_o)

}  // namespace sscan
