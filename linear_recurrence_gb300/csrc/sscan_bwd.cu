// C ABI of the selective-scan backward pass (declared in include/sscan.h):
// validation, the checkpoint scratch and the launch of sscan_bwd_chunked.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>

#include "../../include/sscan.h"
#include "sscan_bwd_kernel.cuh"

namespace sscan {
void record_call(int launches, cudaStream_t stream, const char* plan);
void record_error(cudaError_t e);
cudaError_t scratch_alloc(void** ptr, size_t bytes, cudaStream_t stream);  // sscan_abi.cu
}  // namespace sscan

namespace {

using sscan::BwdCfg;
using sscan::BwdParams;

template <typename T, int NS, int P>
cudaError_t launch_bwd(const BwdParams& p, long long grid, cudaStream_t st) {
    using Cfg = BwdCfg<T, NS, P>;
    auto kern = sscan::sscan_bwd_chunked<T, NS, P>;
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
    kern<<<(unsigned)grid, Cfg::kThreads, Cfg::SMEM_BYTES, st>>>(p);
    return cudaGetLastError();
}

// (states per lane, lanes per channel) by state count
struct BwdShape {
    int NS, P;
};
BwdShape bwd_shape(long long N) {
    if (N <= 4) return {1, 4};
    if (N <= 8) return {2, 4};
    if (N <= 16) return {2, 8};
    if (N <= 32) return {4, 8};
    return {4, 16};
}
int bwd_channels(BwdShape s) { return 4 * (32 / s.P); }

template <typename T>
cudaError_t launch_dtype(const BwdParams& p, BwdShape s, long long grid, cudaStream_t st) {
    if (s.NS == 1 && s.P == 4) return launch_bwd<T, 1, 4>(p, grid, st);
    if (s.NS == 2 && s.P == 4) return launch_bwd<T, 2, 4>(p, grid, st);
    if (s.NS == 2 && s.P == 8) return launch_bwd<T, 2, 8>(p, grid, st);
    if (s.NS == 4 && s.P == 8) return launch_bwd<T, 4, 8>(p, grid, st);
    if (s.NS == 4 && s.P == 16) return launch_bwd<T, 4, 16>(p, grid, st);
    return cudaErrorInvalidValue;
}

template <typename T, int NS, int P>
int occupancy_bwd() {
    using Cfg = BwdCfg<T, NS, P>;
    auto kern = sscan::sscan_bwd_chunked<T, NS, P>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Cfg::kThreads, Cfg::SMEM_BYTES) != cudaSuccess)
        return 0;
    return n;
}

// Resident CTAs per SM of the backward kernel of a shape, queried once per
// device and dtype.
template <typename T>
int occupancy_dtype(BwdShape s) {
    static std::atomic<int> cache[64][5] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int idx = s.P == 16 ? 4 : s.NS == 4 ? 3 : s.P == 8 ? 2 : s.NS == 2 ? 1 : 0;
    std::atomic<int>& c = cache[dev & 63][idx];
    int v = c.load(std::memory_order_relaxed);
    if (v == 0) {
        if (s.NS == 1 && s.P == 4) v = occupancy_bwd<T, 1, 4>();
        else if (s.NS == 2 && s.P == 4) v = occupancy_bwd<T, 2, 4>();
        else if (s.NS == 2 && s.P == 8) v = occupancy_bwd<T, 2, 8>();
        else if (s.NS == 4 && s.P == 8) v = occupancy_bwd<T, 4, 8>();
        else v = occupancy_bwd<T, 4, 16>();
        c.store(v, std::memory_order_relaxed);
    }
    return v;
}

inline bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

}  // namespace

extern "C" int sscan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                         const float* D, const float* h0, const void* dy, const float* dfinal_state,
                         void* du, void* ddelta, float* dA, float* dB, float* dC, float* dD, float* dh0,
                         int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int dtype,
                         void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    sscan::record_call(0, st, "rejected");
    if (dtype != SSCAN_F32 && dtype != SSCAN_BF16) return SSCAN_ERR_INVALID;
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1 || dstate > sscan_max_dstate())
        return SSCAN_ERR_INVALID;
    const long long big = (long long)1 << 46;
    if (batch > big || dim > big || seqlen > big || (batch && dim > big / batch) ||
        (batch * dim && seqlen > big / (batch * dim)))
        return SSCAN_ERR_INVALID;
    if (batch == 0 || dim == 0) {
        sscan::record_call(0, st, "empty");
        return SSCAN_OK;
    }
    if (!A || !dA) return SSCAN_ERR_INVALID;
    // gradients that no step feeds are zero; dh0 takes the final state's gradient
    cudaError_t e = cudaMemsetAsync(dA, 0, (size_t)(dim * dstate) * sizeof(float), st);
    if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, (size_t)dim * sizeof(float), st);
    if (seqlen == 0) {
        if (e == cudaSuccess && dh0) {
            const size_t bytes = (size_t)(batch * dim * dstate) * sizeof(float);
            e = dfinal_state ? cudaMemcpyAsync(dh0, dfinal_state, bytes, cudaMemcpyDeviceToDevice, st)
                             : cudaMemsetAsync(dh0, 0, bytes, st);
        }
        if (e != cudaSuccess) {
            sscan::record_error(e);
            return SSCAN_ERR_CUDA;
        }
        sscan::record_call(0, st, "seqlen 0");
        return SSCAN_OK;
    }
    if (!u || !delta || !B || !C || !dy || !du || !ddelta || !dB || !dC) return SSCAN_ERR_INVALID;
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, (size_t)(batch * dstate * seqlen) * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dC, 0, (size_t)(batch * dstate * seqlen) * sizeof(float), st);
    if (e != cudaSuccess) {
        sscan::record_error(e);
        return SSCAN_ERR_CUDA;
    }
    const BwdShape s = bwd_shape(dstate);
    const long long DT = bwd_channels(s);
    const long long tiles_per_batch = (dim + DT - 1) / DT;
    const long long grid = batch * tiles_per_batch;
    if (grid > (1LL << 30)) return SSCAN_ERR_INVALID;
    const int vece = dtype == SSCAN_F32 ? 4 : 8;
    const bool vec = (seqlen % vece) == 0 && aligned16(u) && aligned16(delta) && aligned16(B) &&
                     aligned16(C) && aligned16(dy) && aligned16(du) && aligned16(ddelta);
    const long long TC = sscan::kBwdChunk;
    const long long nchunks = (seqlen + TC - 1) / TC;
    // time split: about 12 warps per SM (4 per CTA), segments of 8 chunks or more
    // few channels: split time so that the grid fills one wave of the
    // resident CTA slots (a partial second wave would double the time of the
    // CTAs in it)
    long long S = 1;
    {
        int dev = 0, nsm = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && nsm > 0) {
            const int occ = dtype == SSCAN_F32 ? occupancy_dtype<float>(s) : occupancy_dtype<sscan::bf16>(s);
            const long long slots = (long long)nsm * std::max(occ, 1);
            if (grid < slots) S = slots / grid;
            S = std::min(S, std::max(1LL, nchunks / 8));
        }
    }
    const long long Tseg = ((nchunks + S - 1) / S) * TC;
    S = (seqlen + Tseg - 1) / Tseg;
    if (grid * S > (1LL << 30)) return SSCAN_ERR_INVALID;
    const size_t nckpt = (size_t)(batch * dim) * (size_t)nchunks * (size_t)dstate;
    const size_t nseg = (size_t)(batch * dim) * (size_t)S;
    const size_t scratch_floats = nckpt + (S > 1 ? nseg * (2 * (size_t)dstate + 1) : 0);
    void* scratch = nullptr;
    e = sscan::scratch_alloc(&scratch, scratch_floats * sizeof(float), st);
    if (e != cudaSuccess) {
        sscan::record_error(e);
        return SSCAN_ERR_CUDA;
    }
    BwdParams p{};
    p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.h0 = h0;
    p.dy = dy; p.dhT = dfinal_state;
    p.du = du; p.ddelta = ddelta; p.dA = dA; p.dB = dB; p.dC = dC; p.dD = D ? dD : nullptr; p.dh0 = dh0;
    p.ckpt = static_cast<float*>(scratch);
    p.seg_h = p.ckpt + nckpt;
    p.seg_g = p.seg_h + nseg * (size_t)dstate;
    p.seg_dsum = p.seg_g + nseg * (size_t)dstate;
    p.batch = batch; p.dim = dim; p.L = seqlen; p.N = dstate;
    p.Tseg = Tseg; p.S = (int)S;
    p.tiles_per_batch = (int)tiles_per_batch;
    p.vec = vec ? 1 : 0;
    char plan[160];
    snprintf(plan, sizeof(plan), "bwd %s P=%d NS=%d vec=%d tiles=%lld chunks=%lld S=%lld Tseg=%lld",
             dtype == SSCAN_F32 ? "f32" : "bf16", s.P, s.NS, (int)vec, grid, nchunks, S, Tseg);
    sscan::record_call(S > 1 ? 2 : 1, st, plan);
    e = cudaSuccess;
    if (S > 1) {  // per-segment aggregates first
        p.mode = 1;
        e = dtype == SSCAN_F32 ? launch_dtype<float>(p, s, grid * S, st)
                               : launch_dtype<sscan::bf16>(p, s, grid * S, st);
    }
    if (e == cudaSuccess) {
        p.mode = 0;
        e = dtype == SSCAN_F32 ? launch_dtype<float>(p, s, grid * S, st)
                               : launch_dtype<sscan::bf16>(p, s, grid * S, st);
    }
    const cudaError_t ef = cudaFreeAsync(scratch, st);
    if (e == cudaSuccess) e = ef;
    if (e != cudaSuccess) {
        sscan::record_error(e);
        return SSCAN_ERR_CUDA;
    }
    return SSCAN_OK;
}
