// bfloat16-I/O variants of the selective-scan kernel (lanes per channel <= 4), the plain scan.
#define SSCAN_DISPATCH_IMPL
#include "sscan_dispatch.cuh"

namespace sscan {

using UnitT = bf16;
constexpr int UnitOPT = 0;
SSCAN_DEFINE_UNIT(bf16_a_e, SSCAN_SHAPES_A)

}  // namespace sscan
