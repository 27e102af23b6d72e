// bf16-I/O variants of the selective-scan kernels (fp32 state and accumulation).
#define SSCAN_DISPATCH_IMPL
#include "sscan_dispatch.cuh"

namespace sscan {

cudaError_t fwd_launch_bf16(FwdKernel k, const FwdParams& p, Shape sh, bool vec, int grid,
                            cudaStream_t stream) {
    return launch_dtype<bf16>(k, p, sh, vec, grid, stream);
}

int fwd_occupancy_bf16(Shape sh, bool vec) { return occupancy_dtype<bf16>(sh, vec); }

}  // namespace sscan
