// Throughput probe of the exponent unit (MUFU ex2), the denominator of the
// exponent-bound roofline of the selective scan: every element of the scan
// takes one 2^x (one per channel and step when a channel has a single rate).
// The probe runs independent chains x <- 2^-x (values stay in [0.5, 1]) so
// that only the unit's issue rate limits it.
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
