// bfloat16-I/O variants of the selective-scan kernel (lanes per channel <= 4), with the options and the zero-order-hold B-bar.
#define SSCAN_DISPATCH_IMPL
#include "sscan_dispatch.cuh"

namespace sscan {

using UnitT = bf16;
constexpr int UnitOPT = 2;
SSCAN_DEFINE_UNIT(bf16_a_z, SSCAN_SHAPES_A)

}  // namespace sscan
