// Throughput probes behind the roofline of the selective scan.  The exponent
// unit (MUFU ex2): every element of the scan takes one 2^x (one per channel
// and step when a channel has a single rate); the probe runs independent
// chains x <- 2^-x (values stay in [0.5, 1]) so that only the unit's issue
// rate limits it.  The element probe runs the whole arithmetic of an element
// (the exponent and the FP32 operations together), which one issue slot per
// scheduler and clock bounds below the two units' separate peaks.
#include <cuda_runtime.h>

#include "../../include/sscan.h"
#include "device_utils.cuh"

namespace sscan {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeChains = 16;

__global__ void __launch_bounds__(kProbeThreads) ex2_probe_kernel(float* sink, int iters) {
    float x[kProbeChains];
#pragma unroll
    for (int i = 0; i < kProbeChains; ++i) x[i] = 0.5f + 0.01f * (float)((threadIdx.x + i) & 31);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kProbeChains; ++i) x[i] = ex2(-x[i]);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kProbeChains; ++i) s += x[i];
    // never true (x stays in [0.5, 1]); keeps the chains from being removed
    if (s < 0.f) sink[blockIdx.x * kProbeThreads + threadIdx.x] = s;
}

// The arithmetic of one scan element at the highest rate the SM sustains:
// every thread runs K independent state chains, and per step and chain
//   a = 2^(delta * A log2e)        (FMUL, MUFU; once per step when the
//                                   chains share one rate)
//   h = a * h + (delta u) * B      (FMUL, FFMA)
//   y = C * h + y                  (FFMA)
// with delta and delta*u advanced once per step (two FADD).  The exponent
// and the FP32 instructions draw on the same issue slots, so this is the
// peak element rate of the scan's arithmetic, below both the MUFU's and the
// FP32 pipe's separate peaks.
template <bool SHARED>
__global__ void __launch_bounds__(kProbeThreads, 2) element_probe_kernel(float* sink, int iters) {
    constexpr int K = SHARED ? 32 : 16;
    const float f = 1.0f + 1e-3f * (float)(threadIdx.x & 31);
    float h[K], al[K], b[K], c[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        h[k] = 0.01f * (float)k * f;
        al[k] = -0.1f * (float)(k + 1) * f;
        b[k] = 0.5f + 0.03f * (float)k * f;
        c[k] = 0.25f - 0.01f * (float)k * f;
    }
    float d = 0.01f * f, du = 0.02f * f;
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    for (int it = 0; it < iters; ++it) {
        d += 1e-7f;
        du += 1e-7f;
        const float as = SHARED ? ex2(d * al[0]) : 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const float a = SHARED ? as : ex2(d * al[k]);
            h[k] = fmaf(a, h[k], du * b[k]);
            y[k & 3] = fmaf(c[k], h[k], y[k & 3]);
        }
    }
    const float s = (y[0] + y[1]) + (y[2] + y[3]);
    // never true for these values; keeps the chains from being removed
    if (s == -1.2345e-7f) sink[blockIdx.x * kProbeThreads + threadIdx.x] = s;
}

}  // namespace
}  // namespace sscan

extern "C" int sscan_probe_ex2(float* sink, int blocks, int iters, void* stream) {
    if (sink == nullptr || blocks < 1 || iters < 1) return SSCAN_ERR_INVALID;
    sscan::ex2_probe_kernel<<<blocks, sscan::kProbeThreads, 0, static_cast<cudaStream_t>(stream)>>>(sink, iters);
    return cudaGetLastError() == cudaSuccess ? SSCAN_OK : SSCAN_ERR_CUDA;
}

extern "C" long long sscan_probe_ex2_count(int blocks, int iters) {
    return (long long)blocks * sscan::kProbeThreads * sscan::kProbeChains * (long long)iters;
}

extern "C" int sscan_probe_element(float* sink, int blocks, int iters, int shared_rate, void* stream) {
    if (sink == nullptr || blocks < 1 || iters < 1) return SSCAN_ERR_INVALID;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (shared_rate)
        sscan::element_probe_kernel<true><<<blocks, sscan::kProbeThreads, 0, st>>>(sink, iters);
    else
        sscan::element_probe_kernel<false><<<blocks, sscan::kProbeThreads, 0, st>>>(sink, iters);
    return cudaGetLastError() == cudaSuccess ? SSCAN_OK : SSCAN_ERR_CUDA;
}

extern "C" long long sscan_probe_element_count(int blocks, int iters, int shared_rate) {
    return (long long)blocks * sscan::kProbeThreads * (shared_rate ? 32 : 16) * (long long)iters;
}
