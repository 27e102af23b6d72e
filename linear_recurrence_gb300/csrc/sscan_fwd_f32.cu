// float32-I/O variants of the selective-scan kernels.
#define SSCAN_DISPATCH_IMPL
#include "sscan_dispatch.cuh"

namespace sscan {

cudaError_t fwd_launch_f32(FwdKernel k, const FwdParams& p, Shape sh, bool vec, int grid,
                           cudaStream_t stream) {
    return launch_dtype<float>(k, p, sh, vec, grid, stream);
}

int fwd_occupancy_f32(Shape sh, bool vec) { return occupancy_dtype<float>(sh, vec); }

}  // namespace sscan
