// float32-I/O instantiations of the TMA-fed selective-scan kernel: the options and the zero-order hold.
#define SSCAN_TMA_IMPL
#include "sscan_fwd_tma.cuh"

namespace sscan {

using UnitT = float;
constexpr int UnitOPT = 2;
SSCAN_DEFINE_TMA_UNIT(f32_z)

}  // namespace sscan
