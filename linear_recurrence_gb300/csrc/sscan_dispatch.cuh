// Host-side dispatch from a runtime launch plan to the compiled kernel
// variants.  Each I/O dtype is instantiated in its own translation unit so the
// variants compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include "sscan_fwd_kernel.cuh"

namespace sscan {

// (lanes per channel P, state slots per lane NS) combinations that are compiled.
struct Shape {
    int P;
    int NS;
};
constexpr Shape kShapes[] = {{1, 4}, {1, 8}, {1, 16}, {2, 4}, {2, 8}, {4, 4}, {4, 8}, {4, 16}};
constexpr int kMaxDstate = 64;

enum class FwdKernel { Chunked };

// Per-dtype entry points (defined in sscan_fwd_f32.cu / sscan_fwd_bf16.cu).
// launch: enqueue one kernel on `stream`; returns the launch error, or
// cudaErrorInvalidValue for a shape that is not compiled.
cudaError_t fwd_launch_f32(FwdKernel k, const FwdParams& p, Shape sh, bool vec, int grid,
                           cudaStream_t stream);
cudaError_t fwd_launch_bf16(FwdKernel k, const FwdParams& p, Shape sh, bool vec, int grid,
                            cudaStream_t stream);
// Resident CTAs per SM of the chunked kernel (0 on error).
int fwd_occupancy_f32(Shape sh, bool vec);
int fwd_occupancy_bf16(Shape sh, bool vec);
// Channels per CTA and steps per chunk of a shape.
inline int fwd_channels_per_cta(Shape sh) { return 2 * 2 * (32 / sh.P); }
// Time segments are multiples of this many steps (a multiple of every shape's chunk).
constexpr int kChunkSteps = 32;

// Shared implementation, included by the per-dtype translation units only.
#ifdef SSCAN_DISPATCH_IMPL
template <typename T, int NS, int P, bool VEC>
static cudaError_t launch_variant(FwdKernel k, const FwdParams& p, int grid, cudaStream_t stream) {
    using Cfg = FwdCfg<T, NS, P>;
    (void)k;
    auto kern = sscan_fwd_chunked<T, NS, P, VEC>;
    // opting in to more than 48 KB of dynamic shared memory is per device
    static unsigned long long configured = 0;  // bit per device ordinal (< 64)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured, bit, __ATOMIC_ACQ_REL);
    }
    kern<<<grid, Cfg::kThreads, Cfg::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

template <typename T, int NS, int P, bool VEC>
static int occupancy_variant() {
    using Cfg = FwdCfg<T, NS, P>;
    auto kern = sscan_fwd_chunked<T, NS, P, VEC>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Cfg::kThreads, Cfg::SMEM_BYTES) !=
        cudaSuccess)
        return 0;
    return n;
}

#define SSCAN_FOR_SHAPES(X) X(1, 4) X(1, 8) X(1, 16) X(2, 4) X(2, 8) X(4, 4) X(4, 8) X(4, 16)

template <typename T>
static cudaError_t launch_dtype(FwdKernel k, const FwdParams& p, Shape sh, bool vec, int grid,
                                cudaStream_t stream) {
#define SSCAN_CASE(P_, NS_)                                                        \
    if (sh.P == P_ && sh.NS == NS_)                                                \
        return vec ? launch_variant<T, NS_, P_, true>(k, p, grid, stream)          \
                   : launch_variant<T, NS_, P_, false>(k, p, grid, stream);
    SSCAN_FOR_SHAPES(SSCAN_CASE)
#undef SSCAN_CASE
    return cudaErrorInvalidValue;
}

template <typename T>
static int occupancy_dtype(Shape sh, bool vec) {
#define SSCAN_CASE(P_, NS_)                                                        \
    if (sh.P == P_ && sh.NS == NS_)                                                \
        return vec ? occupancy_variant<T, NS_, P_, true>() : occupancy_variant<T, NS_, P_, false>();
    SSCAN_FOR_SHAPES(SSCAN_CASE)
#undef SSCAN_CASE
    return 0;
}
#endif  // SSCAN_DISPATCH_IMPL

}  // namespace sscan
