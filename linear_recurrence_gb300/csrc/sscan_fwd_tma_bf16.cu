// bf16-I/O instantiations of the TMA-fed selective-scan kernel.
#define SSCAN_TMA_IMPL
#include "sscan_fwd_tma.cuh"

namespace sscan {

using UnitT = bf16;
SSCAN_DEFINE_TMA_UNIT(bf16)

}  // namespace sscan
