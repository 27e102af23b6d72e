// Host-side dispatch from a runtime launch plan to the compiled kernel
// variants, and the launch planner shared by the entry points.  The variants
// are instantiated in twelve translation units so that they compile in
// parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "sscan_fwd_kernel.cuh"

namespace sscan {

// (lanes per channel P, state slots per lane NS, channels per lane CPL).
struct Shape {
    int P;
    int NS;
    int CPL;
};
// Every compiled shape.  The first group (P <= 4) lives in the *_a units, the
// second (P >= 8) in the *_b units.
#ifndef SSCAN_SHAPES_A
#define SSCAN_SHAPES_A(X) X(1, 4, 1) X(2, 4, 1) X(4, 4, 1) X(4, 16, 2) X(2, 8, 1)
#endif
#ifndef SSCAN_SHAPES_B
#define SSCAN_SHAPES_B(X) X(8, 2, 1) X(8, 2, 2) X(8, 4, 1) X(8, 8, 1) X(16, 4, 1)
#endif
#define SSCAN_SHAPE_INIT(P_, NS_, CPL_) {P_, NS_, CPL_},
constexpr Shape kShapes[] = {SSCAN_SHAPES_A(SSCAN_SHAPE_INIT) SSCAN_SHAPES_B(SSCAN_SHAPE_INIT)};
constexpr int kMaxDstate = 64;

inline int shape_warps(Shape sh) { return warps_for(sh.P, sh.CPL); }
inline int shape_channels(Shape sh) { return shape_warps(sh) * (32 / sh.P) * sh.CPL; }

// Per-unit entry points: enqueue one kernel on `stream` (returns the launch
// error, or cudaErrorInvalidValue for a shape the unit does not hold), and the
// resident CTAs per SM of a shape (0 if unknown).  Units: I/O dtype x shape
// group (a: P <= 4, b: P >= 8) x variant (e: the plain scan; o: with the
// delta bias / softplus / gate options; z: options and the zero-order hold).
#define SSCAN_DECLARE_UNIT(SUFFIX)                                                               \
    cudaError_t fwd_launch_##SUFFIX(const FwdParams& p, Shape sh, int grid, cudaStream_t stream); \
    int fwd_occupancy_##SUFFIX(Shape sh);
SSCAN_DECLARE_UNIT(f32_a_e)
SSCAN_DECLARE_UNIT(f32_b_e)
SSCAN_DECLARE_UNIT(bf16_a_e)
SSCAN_DECLARE_UNIT(bf16_b_e)
SSCAN_DECLARE_UNIT(f32_a_o)
SSCAN_DECLARE_UNIT(f32_b_o)
SSCAN_DECLARE_UNIT(bf16_a_o)
SSCAN_DECLARE_UNIT(bf16_b_o)
SSCAN_DECLARE_UNIT(f32_a_z)
SSCAN_DECLARE_UNIT(f32_b_z)
SSCAN_DECLARE_UNIT(bf16_a_z)
SSCAN_DECLARE_UNIT(bf16_b_z)
#undef SSCAN_DECLARE_UNIT

// Kernel variant of a launch: 0 plain, 1 options, 2 options + zero-order hold.
inline int fwd_variant(const FwdParams& p) {
    if (p.zoh) return 2;
    return (p.z != nullptr || p.delta_bias != nullptr || p.delta_softplus) ? 1 : 0;
}
inline cudaError_t fwd_launch(bool f32, const FwdParams& p, Shape sh, int grid, cudaStream_t stream) {
    const bool a = sh.P <= 4;
    switch (fwd_variant(p)) {
        case 2:
            if (f32) return a ? fwd_launch_f32_a_z(p, sh, grid, stream) : fwd_launch_f32_b_z(p, sh, grid, stream);
            return a ? fwd_launch_bf16_a_z(p, sh, grid, stream) : fwd_launch_bf16_b_z(p, sh, grid, stream);
        case 1:
            if (f32) return a ? fwd_launch_f32_a_o(p, sh, grid, stream) : fwd_launch_f32_b_o(p, sh, grid, stream);
            return a ? fwd_launch_bf16_a_o(p, sh, grid, stream) : fwd_launch_bf16_b_o(p, sh, grid, stream);
        default:
            if (f32) return a ? fwd_launch_f32_a_e(p, sh, grid, stream) : fwd_launch_f32_b_e(p, sh, grid, stream);
            return a ? fwd_launch_bf16_a_e(p, sh, grid, stream) : fwd_launch_bf16_b_e(p, sh, grid, stream);
    }
}
inline int fwd_occupancy(bool f32, Shape sh) {
    if (sh.P <= 4) return f32 ? fwd_occupancy_f32_a_e(sh) : fwd_occupancy_bf16_a_e(sh);
    return f32 ? fwd_occupancy_f32_b_e(sh) : fwd_occupancy_bf16_b_e(sh);
}

// Shapes of the TMA-fed kernel (sscan_fwd_tma.cuh): four warps per CTA, so
// DT = 4 * (32 / P) * CPL channels per CTA.  It serves the scan (plain or
// with the options) with 16-byte aligned rows in every mode (single, local,
// carry correction), for 8 < N <= 16 ((8,2,2), (4,4,2)) and 32 < N <= 64
// ((4,16,2)); the cp.async kernel takes the other state counts (measured on
// GB300 where both apply: the TMA kernel as fast or faster).
#ifndef SSCAN_TMA_SHAPES
#define SSCAN_TMA_SHAPES(X) X(8, 2, 2) X(4, 4, 2) X(4, 16, 2)
#endif
inline int tma_channels(Shape sh) { return 4 * (32 / sh.P) * sh.CPL; }
// Shapes of the shuffle kernels (the TMA-fed kernel's plain scan with
// outputs summed by shuffles): 16 state slots as 2 lanes x 8 states, two
// channels per lane; with one channel per lane for the carry correction only.
#ifndef SSCAN_TMA_SHFL_SHAPES
#define SSCAN_TMA_SHFL_SHAPES(X) X(2, 8, 2) X(2, 8, 1)
#endif
bool shfl_has_shape(Shape sh);
cudaError_t fwd_shfl_launch(bool f32, const FwdParams& p, Shape sh, int grid, cudaStream_t stream);
int fwd_shfl_occupancy(bool f32, Shape sh);
cudaError_t fwd_shfl_launch_f32(const FwdParams& p, Shape sh, int grid, cudaStream_t stream);
cudaError_t fwd_shfl_launch_bf16(const FwdParams& p, Shape sh, int grid, cudaStream_t stream);
int fwd_shfl_occupancy_f32(Shape sh);
int fwd_shfl_occupancy_bf16(Shape sh);
bool tma_has_shape(Shape sh);
cudaError_t fwd_tma_launch(bool f32, const FwdParams& p, Shape sh, int grid, cudaStream_t stream);
// resident CTAs per SM of a shape and variant (0 plain, 1 options, 2 zero-order hold)
int fwd_tma_occupancy(bool f32, Shape sh, int variant);
#define SSCAN_DECLARE_TMA_UNIT(SUFFIX)                                                                \
    cudaError_t fwd_tma_launch_##SUFFIX(const FwdParams& p, Shape sh, int grid, cudaStream_t stream); \
    int fwd_tma_occupancy_##SUFFIX(Shape sh);
SSCAN_DECLARE_TMA_UNIT(f32_e)
SSCAN_DECLARE_TMA_UNIT(f32_o)
SSCAN_DECLARE_TMA_UNIT(f32_z)
SSCAN_DECLARE_TMA_UNIT(bf16_e)
SSCAN_DECLARE_TMA_UNIT(bf16_o)
SSCAN_DECLARE_TMA_UNIT(bf16_z)
#undef SSCAN_DECLARE_TMA_UNIT
// Encode a 3-D tensor map {L, rows, batch} of a contiguous [batch, rows, L]
// fp32 or bf16 array with box {box_l, box_rows, 1} (false on failure).
bool tma_encode_3d(CUtensorMap* map, const void* base, bool f32, long long L, long long rows, long long batch,
                   int box_l, int box_rows);

// The fold pass of a time split into more than kFoldInCorrectionMaxSegments
// segments (sscan_fold.cu): from the local pass's aggregates, the state
// entering each segment s >= 1, written over aggregate slot s - 1; launched as
// a programmatic dependent of the local pass.
cudaError_t fwd_fold_launch(const FwdParams& p, cudaStream_t stream);
// Splits of up to this many segments skip the fold pass: each correction CTA
// folds the earlier segments' aggregates itself (O(S) per CTA, a few loads in
// flight at a time), which saves one launch on the critical path (512
// channels x 8192 steps in 19 segments: 47.1 us either way, one launch fewer).
// Beyond it the pass is cheaper (1536 x 65536 in 25 segments: 453 us with the
// pass, 464 us with the fold in the correction).
constexpr long long kFoldInCorrectionMaxSegments = 24;
// Scratch floats per (channel, segment) of a time split: the end state (N),
// the sum of delta and min(0, smallest delta).
inline long long split_floats_per_segment(long long N) { return N + 2; }

// Stream-ordered scratch of the time-split passes (defined in sscan_abi.cu):
// from a per-device pool of this library that keeps up to
// kScratchRetainBytes mapped while idle, so that a call after a host
// synchronisation does not map its scratch again.
constexpr unsigned long long kScratchRetainBytes = 1ull << 30;
cudaError_t scratch_alloc(void** ptr, size_t bytes, cudaStream_t stream);

// A launch plan of the forward pass (defined in sscan_abi.cu).
struct FwdPlan {
    Shape sh;
    long long tiles_per_batch;
    long long tiles;  // channel tiles (CTAs per segment)
    long long S;      // time segments
    long long Tseg;   // steps per segment
    bool tma;         // the single/local pass runs on the TMA-fed kernel
    bool shfl;        // ... in its shuffle variant (plain scan)
    Shape corr_sh;    // shape of the carry correction
    bool corr_tma;    // the correction runs on the TMA-fed kernel (else cp.async)
    bool corr_shfl;   // ... in its shuffle variant
    long long corr_tiles_per_batch;
    long long corr_tiles;
};
// Choose the shape and time split.  lanes: 0 = automatic, else P; segments:
// 0 = automatic, else S; max_segments (>= 1) caps an automatic split.
// Returns SSCAN_OK, SSCAN_ERR_INVALID or SSCAN_ERR_CUDA.
int plan_fwd(bool f32, long long batch, long long dim, long long seqlen, long long N, int segments,
             int lanes, long long max_segments, FwdPlan* out);
// The plan of the TMA-fed kernel (aligned rows, 8 < N <= 16; lanes 0, 4 or
// 8; variant as fwd_variant), or SSCAN_ERR_INVALID when it does not apply.
// plan_fwd_shfl: the plan of its shuffle variant (plain scan, aligned rows,
// 8 < N <= 16, lanes 0 or 2).
int plan_fwd_shfl(bool f32, long long batch, long long dim, long long seqlen, long long N, int segments,
                  int lanes, long long max_segments, FwdPlan* out);
int plan_fwd_tma(bool f32, int variant, long long batch, long long dim, long long seqlen, long long N,
                 int segments, int lanes, FwdPlan* out);

// Shared implementation, included by the per-unit translation units only.
#ifdef SSCAN_DISPATCH_IMPL
template <typename T, int NS, int P, int CPL, int OPT>
static cudaError_t launch_variant(const FwdParams& p, int grid, cudaStream_t stream) {
    using Cfg = FwdCfg<T, NS, P, CPL, OPT>;
    const bool corr = p.mode == MODE_CORR;
    auto kern = corr ? sscan_fwd_chunked<T, NS, P, CPL, OPT, true> : sscan_fwd_chunked<T, NS, P, CPL, OPT, false>;
    // the state slots of a shape must cover every state: the kernel stages
    // B/C rows n < N into NSP slots
    if (p.N < 1 || p.N > (long long)Cfg::NSP) return cudaErrorInvalidValue;
    // opting in to more than 48 KB of dynamic shared memory is per device and
    // kernel (one bit per device and kernel)
    static unsigned long long configured[2] = {0, 0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&configured[corr ? 1 : 0], __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured[corr ? 1 : 0], bit, __ATOMIC_ACQ_REL);
    }
    if (!corr) {
        kern<<<grid, Cfg::kThreads, Cfg::SMEM_BYTES, stream>>>(p);
        return cudaGetLastError();
    }
    // the correction follows the local pass on the same stream as a
    // programmatic dependent: its CTAs may be resident before the pass ends
    // and wait (griddepcontrol.wait) for its results
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int NS, int P, int CPL, int OPT>
static int occupancy_variant() {
    using Cfg = FwdCfg<T, NS, P, CPL, OPT>;
    auto kern = sscan_fwd_chunked<T, NS, P, CPL, OPT, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Cfg::kThreads, Cfg::SMEM_BYTES) !=
        cudaSuccess)
        return 0;
    return n;
}

// A unit sets `using UnitT = float;` (or bf16) and `constexpr int UnitOPT`, then
// expands SSCAN_DEFINE_UNIT(f32_a_e, SSCAN_SHAPES_A) and so on.
#define SSCAN_LAUNCH_CASE(P_, NS_, CPL_)                                   \
    if (sh.P == P_ && sh.NS == NS_ && sh.CPL == CPL_)                      \
        return launch_variant<UnitT, NS_, P_, CPL_, UnitOPT>(p, grid, st);
#define SSCAN_OCC_CASE(P_, NS_, CPL_)                                      \
    if (sh.P == P_ && sh.NS == NS_ && sh.CPL == CPL_) return occupancy_variant<UnitT, NS_, P_, CPL_, UnitOPT>();
#define SSCAN_DEFINE_UNIT(SUFFIX, SHAPES)                                                       \
    cudaError_t fwd_launch_##SUFFIX(const FwdParams& p, Shape sh, int grid, cudaStream_t st) { \
        SHAPES(SSCAN_LAUNCH_CASE)                                                               \
        return cudaErrorInvalidValue;                                                           \
    }                                                                                           \
    int fwd_occupancy_##SUFFIX(Shape sh) {                                                      \
        SHAPES(SSCAN_OCC_CASE)                                                                  \
        return 0;                                                                               \
    }
#endif  // SSCAN_DISPATCH_IMPL

}  // namespace sscan
