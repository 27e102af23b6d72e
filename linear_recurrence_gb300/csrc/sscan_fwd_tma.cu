// Host side of the TMA-fed selective-scan kernel: tensor-map encoding through
// the driver's cuTensorMapEncodeTiled (looked up once through the runtime, so
// nothing links against libcuda) and the dispatch to the per-dtype units.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "sscan_dispatch.cuh"

namespace sscan {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    static std::mutex mu;
    PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
    if (f != nullptr) return f;
    std::lock_guard<std::mutex> lock(mu);
    f = fn.load(std::memory_order_relaxed);
    if (f == nullptr) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

}  // namespace

// 3-D map {L, rows, batch} over a contiguous [batch, rows, L] array with a
// box of {box_l, box_rows, 1}; zeros outside the array.
bool tma_encode_3d(CUtensorMap* map, const void* base, bool f32, long long L, long long rows, long long batch,
               int box_l, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 f = encode_fn();
    if (f == nullptr) return false;
    const cuuint64_t esz = f32 ? 4 : 2;
    const cuuint64_t dims[3] = {(cuuint64_t)L, (cuuint64_t)rows, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)L * esz, (cuuint64_t)(L * rows) * esz};
    const cuuint32_t box[3] = {(cuuint32_t)box_l, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = f(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tma_has_shape(Shape sh) {
#define SSCAN_TMA_HAS(P_, NS_, CPL_) \
    if (sh.P == P_ && sh.NS == NS_ && sh.CPL == CPL_) return true;
    SSCAN_TMA_SHAPES(SSCAN_TMA_HAS)
#undef SSCAN_TMA_HAS
    return false;
}

cudaError_t fwd_tma_launch(bool f32, const FwdParams& p, Shape sh, int grid, cudaStream_t stream) {
    if (!p.vec) return cudaErrorInvalidValue;
    switch (fwd_variant(p)) {
        case 2: return f32 ? fwd_tma_launch_f32_z(p, sh, grid, stream) : fwd_tma_launch_bf16_z(p, sh, grid, stream);
        case 1: return f32 ? fwd_tma_launch_f32_o(p, sh, grid, stream) : fwd_tma_launch_bf16_o(p, sh, grid, stream);
        default: return f32 ? fwd_tma_launch_f32_e(p, sh, grid, stream) : fwd_tma_launch_bf16_e(p, sh, grid, stream);
    }
}

bool shfl_has_shape(Shape sh) {
#define SSCAN_SHFL_HAS(P_, NS_, CPL_) \
    if (sh.P == P_ && sh.NS == NS_ && sh.CPL == CPL_) return true;
    SSCAN_TMA_SHFL_SHAPES(SSCAN_SHFL_HAS)
#undef SSCAN_SHFL_HAS
    return false;
}

cudaError_t fwd_shfl_launch(bool f32, const FwdParams& p, Shape sh, int grid, cudaStream_t stream) {
    if (!p.vec) return cudaErrorInvalidValue;
    return f32 ? fwd_shfl_launch_f32(p, sh, grid, stream) : fwd_shfl_launch_bf16(p, sh, grid, stream);
}

int fwd_shfl_occupancy(bool f32, Shape sh) { return f32 ? fwd_shfl_occupancy_f32(sh) : fwd_shfl_occupancy_bf16(sh); }

int fwd_tma_occupancy(bool f32, Shape sh, int variant) {
    switch (variant) {
        case 2: return f32 ? fwd_tma_occupancy_f32_z(sh) : fwd_tma_occupancy_bf16_z(sh);
        case 1: return f32 ? fwd_tma_occupancy_f32_o(sh) : fwd_tma_occupancy_bf16_o(sh);
        default: return f32 ? fwd_tma_occupancy_f32_e(sh) : fwd_tma_occupancy_bf16_e(sh);
    }
}

}  // namespace sscan
