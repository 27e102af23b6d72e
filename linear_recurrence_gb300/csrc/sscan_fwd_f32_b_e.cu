// float32-I/O variants of the selective-scan kernel (lanes per channel >= 8), the plain scan.
#define SSCAN_DISPATCH_IMPL
#include "sscan_dispatch.cuh"

namespace sscan {

using UnitT = float;
constexpr int UnitOPT = 0;
SSCAN_DEFINE_UNIT(f32_b_e, SSCAN_SHAPES_B)

}  // namespace sscan
