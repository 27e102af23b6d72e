// bfloat16-I/O variants of the selective-scan kernel (lanes per channel >= 8), with the delta bias / softplus / gate options.
#define SSCAN_DISPATCH_IMPL
#include "sscan_dispatch.cuh"

namespace sscan {

using UnitT = bf16;
constexpr int UnitOPT = 1;
SSCAN_DEFINE_UNIT(bf16_b_o, SSCAN_SHAPES_B)

}  // namespace sscan
