// sscan_fwd_noalloc: the selective-scan forward pass without any device
// allocation, for callers that cannot allocate device memory while they run.
//
// Some hosts must never allocate during their own execution path: an
// inference engine calling a plugin's per-request hook under a fixed memory
// budget, a real-time loop where an allocation may synchronise the device or
// stall on the allocator, or an embedding runtime whose memory is handed out
// up front.  sscan_fwd may need a little scratch (the per-segment carry of a
// time-split launch) and takes it from CUDA's stream-ordered pool; this entry
// point instead keeps that scratch in a fixed array in device memory that
// every GPU which loads libsscan.so holds until the process exits.
//
// Setup: the first call on each device looks up the array's device address
// with cudaGetSymbolAddress (with that device current) and caches it.  That
// lookup may load the module, so make the first call on a device before any
// stream capture.
//
// Sharing: every call uses the same array.  Everything a call reads from it
// is written earlier in the same call, so nothing needs clearing between
// calls, but two calls whose kernels overlap on the GPU (different streams,
// no ordering between them) race on the array and may corrupt each other's
// results.  Order such calls on one stream, or use sscan_fwd.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include <stdio.h>

#include "../../include/sscan.h"
#include "sscan_dispatch.cuh"

namespace sscan {
// call record and device status word of the entry points (sscan_abi.cu)
void record_call(int launches, cudaStream_t stream, const char* plan);
int* device_status_word();
}  // namespace sscan

namespace {

constexpr size_t kScratchBytes = SSCAN_NOALLOC_SCRATCH_BYTES;  // carry scratch per GPU
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[64] = {nullptr};  // per device ordinal

// Device address of the scratch array on the current device (set up once).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

inline bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaError_t launch(bool f32, const sscan::FwdParams& p, sscan::Shape sh, long long grid,
                   cudaStream_t st) {
    if (grid <= 0) return cudaSuccess;
    return sscan::fwd_launch(f32, p, sh, (int)grid, st);
}

}  // namespace

extern "C" int sscan_fwd_noalloc(const void* u, const void* delta, const float* A, const void* B,
                                 const void* C, const float* D, const float* h0, void* out,
                                 float* final_state, int64_t batch, int64_t dim, int64_t seqlen,
                                 int64_t dstate, int dtype, int segments, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    sscan::record_call(0, st, "rejected");
    if (dtype != SSCAN_F32 && dtype != SSCAN_BF16) return SSCAN_ERR_INVALID;
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1 || dstate > sscan::kMaxDstate ||
        segments < 0)
        return SSCAN_ERR_INVALID;
    const long long big = (long long)1 << 46;
    if (batch > big || dim > big || seqlen > big || (batch && dim > big / batch) ||
        (batch * dim && seqlen > big / (batch * dim)))
        return SSCAN_ERR_INVALID;
    if (batch == 0 || dim == 0) {
        sscan::record_call(0, st, "empty");
        return SSCAN_OK;
    }
    if (seqlen == 0) {
        sscan::record_call(0, st, "seqlen 0: final_state = h0");
        if (final_state) {
            const size_t bytes = (size_t)(batch * dim * dstate) * sizeof(float);
            cudaError_t e = h0 ? cudaMemcpyAsync(final_state, h0, bytes, cudaMemcpyDeviceToDevice, st)
                               : cudaMemsetAsync(final_state, 0, bytes, st);
            if (e != cudaSuccess) return SSCAN_ERR_CUDA;
        }
        return SSCAN_OK;
    }
    if (!u || !delta || !A || !B || !C || !out) return SSCAN_ERR_INVALID;

    const bool f32 = dtype == SSCAN_F32;
    const int esz = f32 ? 4 : 2;
    const bool vec = (seqlen % (16 / esz)) == 0 && is_aligned16(u) && is_aligned16(delta) &&
                     is_aligned16(B) && is_aligned16(C) && is_aligned16(out);
    // carry scratch of a plan with S segments: batch*dim*S*(dstate+2) floats
    const long long per_segment =
        batch * dim * sscan::split_floats_per_segment(dstate) * (long long)sizeof(float);
    const long long max_segments = (long long)kScratchBytes / per_segment;  // may be 0 or 1
    sscan::FwdPlan pl;
    const int prc = sscan::plan_fwd(f32, batch, dim, seqlen, dstate, segments, 0,
                                    std::max(1LL, max_segments), &pl);
    if (prc != SSCAN_OK) return prc;
    const sscan::Shape sh = pl.sh;
    const long long S = pl.S, tiles = pl.tiles, Tseg = pl.Tseg, tiles_per_batch = pl.tiles_per_batch;
    if (S > 1 && S > max_segments) return SSCAN_ERR_INVALID;  // would overflow the fixed scratch

    int* status = sscan::device_status_word();
    if (status == nullptr) return SSCAN_ERR_CUDA;
    sscan::FwdParams p{};
    p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.h0 = h0;
    p.out = out; p.final_state = final_state;
    p.batch = batch; p.dim = dim; p.L = seqlen; p.N = dstate;
    p.Tseg = Tseg; p.S = (int)S; p.tiles_per_batch = (int)tiles_per_batch;
    p.vec = vec ? 1 : 0;
    p.status = status;
    char plan[160];
    snprintf(plan, sizeof(plan), "noalloc %s P=%d NS=%d CPL=%d vec=%d tiles=%lld S=%lld Tseg=%lld cp.async %s",
             f32 ? "f32" : "bf16", sh.P, sh.NS, sh.CPL, (int)vec, tiles, S, Tseg,
             S == 1 ? "single" : S <= sscan::kFoldInCorrectionMaxSegments ? "local+correct" : "local+fold+correct");

    cudaError_t e;
    if (S == 1) {
        p.mode = sscan::MODE_SINGLE;
        p.seg_count = 1;
        e = launch(f32, p, sh, tiles, st);
        sscan::record_call(1, st, plan);
        return e == cudaSuccess ? SSCAN_OK : SSCAN_ERR_CUDA;
    }
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return SSCAN_ERR_CUDA;
    const size_t nseg = (size_t)(batch * dim) * (size_t)S;
    p.seg_state = static_cast<float*>(scratch);
    p.seg_dsum = p.seg_state + nseg * (size_t)dstate;
    p.seg_dmin = p.seg_dsum + nseg;
    // pass 1: every segment from its local start, writing y and its aggregate;
    // pass 2 (more than kFoldInCorrectionMaxSegments segments): fold the
    // aggregates into the state entering each segment; pass 3: add the carried
    // state's decaying contribution (folding the aggregates itself when pass 2
    // did not run) and compose the final state (bf16 outputs are rounded
    // twice, the second time with the carry added)
    p.mode = sscan::MODE_LOCAL;
    p.seg_count = (int)S;
    e = launch(f32, p, sh, tiles * S, st);
    p.fold_in_corr = S <= sscan::kFoldInCorrectionMaxSegments ? 1 : 0;
    if (e == cudaSuccess && S > 2 && !p.fold_in_corr) e = sscan::fwd_fold_launch(p, st);
    if (e == cudaSuccess) {
        p.mode = sscan::MODE_CORR;
        p.seg_count = (int)(S - 1);
        e = launch(f32, p, sh, tiles * (S - 1), st);
    }
    sscan::record_call(S > sscan::kFoldInCorrectionMaxSegments ? 3 : 2, st, plan);
    return e == cudaSuccess ? SSCAN_OK : SSCAN_ERR_CUDA;
}
