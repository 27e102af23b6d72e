// Fold pass of a time-split forward scan: the state entering every segment.
//
// The local pass leaves, per channel and segment s, the end state e_s of the
// segment's recurrence started from zero (segment 0 from h0) and the sum of
// delta over the segment.  Across a whole segment the recurrence is the affine
// map h -> 2^(A log2e sum_t delta_t) h + e_s (the chunk-carry identity of
// "为什么Mamba的“并行扫描”不是真并行" section 3, with the product of the
// step decays exp(delta_t A) written as one exponential), so the state
// entering segment s + 1 is that map applied to the state entering s: the
// segments' aggregates composed in order with the operator
// (a1, b1) o (a2, b2) = (a2 a1, a2 b1 + b2) of "并行扫描与硬件感知优化"
// section 2.2.  One thread per (channel, state) walks the segments in order
// and writes the state entering segment s over slot s - 1 of the aggregates
// (whose end state it has already read).  The carry correction then reads its
// entry state from slot s - 1, and the last segment's correction composes the
// final state from its entry state and its own aggregate (slot S - 1, which
// this pass leaves as it is).  With two segments slot 0 already holds the
// state entering segment 1, and the pass is not launched.
#include <cuda_runtime.h>

#include <climits>

#include "sscan_dispatch.cuh"

namespace sscan {

namespace {

constexpr int kFoldThreads = 256;
constexpr int kFoldBatch = 8;  // segments whose loads are issued together

// (64 registers at most: four CTAs per SM, since a fold over few segments is
// a single load round trip per thread and its speed is the number in flight)
__global__ void __launch_bounds__(kFoldThreads, 4) sscan_fold_kernel(const FwdParams p) {
    // the correction, launched as this pass's programmatic dependent, may
    // start its CTAs (it waits for this pass before reading the entry states)
    griddep_launch_dependents();
    // the host guarantees batch * dim * N < 2^31 (32-bit index arithmetic)
    const int chains = (int)(p.batch * p.dim * p.N);
    const int idx = (int)blockIdx.x * kFoldThreads + (int)threadIdx.x;
    const int N = (int)p.N, dim = (int)p.dim;
    int ch = 0, n = 0;
    float al2 = 0.f;
    if (idx < chains) {
        ch = idx / N;
        n = idx - ch * N;
        al2 = p.A[(ch % dim) * N + n] * kLog2e;
    }
    griddep_wait();  // the local pass's aggregates are complete and visible
    if (idx >= chains) return;
    float* st = p.seg_state + (long long)ch * p.S * N + n;  // slot s at st[s * N]
    const float* ds = p.seg_dsum + (long long)ch * p.S;
    float h = st[0];  // segment 0 started from h0: its end state is the true one
    for (int s0 = 1; s0 < p.S; s0 += kFoldBatch) {
        float e[kFoldBatch], dv[kFoldBatch];
#pragma unroll
        for (int q = 0; q < kFoldBatch; ++q) {
            const int s = s0 + q;
            e[q] = s < p.S ? st[(long long)s * N] : 0.f;
            dv[q] = s < p.S ? ds[s] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kFoldBatch; ++q) {
            const int s = s0 + q;
            if (s < p.S) {
                st[(long long)(s - 1) * N] = h;          // the state entering segment s
                h = fmaf(ex2(al2 * dv[q]), h, e[q]);  // ... and entering s + 1
            }
        }
    }
}

}  // namespace

cudaError_t fwd_fold_launch(const FwdParams& p, cudaStream_t stream) {
    const long long chains = p.batch * p.dim * p.N;
    const long long grid = (chains + kFoldThreads - 1) / kFoldThreads;
    if (grid <= 0) return cudaSuccess;
    if (chains >= (long long)INT_MAX - kFoldThreads) return cudaErrorInvalidValue;
    // a programmatic dependent of the local pass: its CTAs may become resident
    // while the pass runs and wait (griddepcontrol.wait) for its results
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kFoldThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, sscan_fold_kernel, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace sscan
