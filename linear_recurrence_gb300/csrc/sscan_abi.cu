// C ABI of libsscan.so (declared in include/sscan.h): argument validation,
// launch planning and stream-ordered scratch for the selective-scan and pscan
// kernels.  Nothing here computes on the host; every step of the scan runs in
// the kernels it launches.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <algorithm>

#include "../../include/sscan.h"
#include "pscan_kernel.cuh"
#include "sscan_dispatch.cuh"

namespace {

using sscan::FwdKernel;
using sscan::FwdParams;
using sscan::Shape;

struct CallRecord {
    int launches = 0;
    cudaStream_t stream = nullptr;
    int pending_error = SSCAN_OK;
    char plan[256] = "none";
};
thread_local CallRecord g_rec;

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int& c = cached[dev & 63];
    if (c == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        c = n;
    }
    return c;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

int fail_cuda(cudaError_t e) {
    g_rec.pending_error = SSCAN_ERR_CUDA;
    snprintf(g_rec.plan, sizeof(g_rec.plan), "cuda error: %s", cudaGetErrorString(e));
    return SSCAN_ERR_CUDA;
}

// Smallest compiled shape for dstate N with the requested lanes per channel
// (0 = the default for N).
bool choose_shape(long long N, int lanes, Shape* out) {
    if (lanes == 0) {
        if (N <= 4) lanes = 1;
        else if (N <= 8) lanes = 2;
        else lanes = 4;
    }
    for (const Shape& s : sscan::kShapes)
        if (s.P == lanes && (long long)s.NS * s.P >= N) {
            *out = s;
            return true;
        }
    return false;
}

cudaError_t launch_fwd(int dtype, FwdKernel k, const FwdParams& p, Shape sh, bool vec, long long grid,
                       cudaStream_t st) {
    if (grid <= 0) return cudaSuccess;
    ++g_rec.launches;
    return dtype == SSCAN_F32 ? sscan::fwd_launch_f32(k, p, sh, vec, (int)grid, st)
                              : sscan::fwd_launch_bf16(k, p, sh, vec, (int)grid, st);
}

}  // namespace

namespace sscan {
// Call record of an entry point defined in another translation unit.
void record_call(int launches, cudaStream_t stream, const char* plan) {
    g_rec.launches = launches;
    g_rec.stream = stream;
    snprintf(g_rec.plan, sizeof(g_rec.plan), "%s", plan);
}
void record_error(cudaError_t e) { fail_cuda(e); }
}  // namespace sscan

extern "C" {

const char* sscan_status_string(int status) {
    switch (status) {
        case SSCAN_OK: return "SSCAN_OK";
        case SSCAN_ERR_INVALID: return "SSCAN_ERR_INVALID: invalid argument";
        case SSCAN_ERR_CUDA: return "SSCAN_ERR_CUDA: CUDA call failed";
        case SSCAN_ERR_TIMEOUT: return "SSCAN_ERR_TIMEOUT: a bounded device wait gave up";
        default: return "SSCAN_ERR_UNKNOWN: unknown status code";
    }
}

int sscan_max_dstate(void) { return sscan::kMaxDstate; }

int sscan_last_launch_count(void) { return g_rec.launches; }

const char* sscan_last_plan(void) { return g_rec.plan; }

int sscan_get_last_error(void) {
    int status = g_rec.pending_error;
    cudaError_t e = cudaStreamSynchronize(g_rec.stream);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess && status == SSCAN_OK) status = SSCAN_ERR_CUDA;
    g_rec.pending_error = SSCAN_OK;
    return status;
}

int sscan_fwd_ex(const void* u, const void* delta, const float* A, const void* B, const void* C,
                 const float* D, const float* h0, void* out, float* final_state, int64_t batch,
                 int64_t dim, int64_t seqlen, int64_t dstate, int dtype, int segments, int lanes,
                 void* stream) {
    g_rec.launches = 0;
    snprintf(g_rec.plan, sizeof(g_rec.plan), "rejected");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    g_rec.stream = st;
    if (dtype != SSCAN_F32 && dtype != SSCAN_BF16) return SSCAN_ERR_INVALID;
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1 || dstate > sscan::kMaxDstate)
        return SSCAN_ERR_INVALID;
    if (segments < 0 || lanes < 0) return SSCAN_ERR_INVALID;
    // every element index of every array must fit comfortably in int64 and
    // every grid in a 32-bit grid dimension
    const long long big = (long long)1 << 46;
    if (batch > big || dim > big || seqlen > big || (batch && dim > big / batch) ||
        (batch * dim && seqlen > big / (batch * dim)))
        return SSCAN_ERR_INVALID;
    Shape sh;
    if (!choose_shape(dstate, lanes, &sh)) return SSCAN_ERR_INVALID;

    // empty problems: arrays with no elements may be NULL
    if (batch == 0 || dim == 0) {
        snprintf(g_rec.plan, sizeof(g_rec.plan), "empty");
        return SSCAN_OK;
    }
    if (seqlen == 0) {
        snprintf(g_rec.plan, sizeof(g_rec.plan), "seqlen 0: final_state = h0");
        if (final_state) {
            const size_t bytes = (size_t)(batch * dim * dstate) * sizeof(float);
            cudaError_t e = h0 ? cudaMemcpyAsync(final_state, h0, bytes, cudaMemcpyDeviceToDevice, st)
                               : cudaMemsetAsync(final_state, 0, bytes, st);
            if (e != cudaSuccess) return fail_cuda(e);
        }
        return SSCAN_OK;
    }
    if (!u || !delta || !A || !B || !C || !out) return SSCAN_ERR_INVALID;

    const int esz = dtype == SSCAN_F32 ? 4 : 2;
    const int vece = 16 / esz;
    const bool vec = (seqlen % vece) == 0 && aligned16(u) && aligned16(delta) && aligned16(B) &&
                     aligned16(C) && aligned16(out);
    const int DT = sscan::fwd_channels_per_cta(sh);
    const int TC = sscan::kChunkSteps;
    const long long tiles_per_batch = ceil_div(dim, DT);
    const long long tiles = batch * tiles_per_batch;
    if (tiles > (1LL << 30)) return SSCAN_ERR_INVALID;

    // time split: about two CTAs per SM (measured best on GB300 for the
    // few-channel workloads), each segment at least 8 chunks long
    long long S = segments;
    if (S == 0) {
        const int nsm = sm_count();
        const int occ = dtype == SSCAN_F32 ? sscan::fwd_occupancy_f32(sh, vec)
                                           : sscan::fwd_occupancy_bf16(sh, vec);
        // fp32 splits cost a short carry pass; bf16 splits re-run every segment,
        // so bf16 splits only when there are fewer tiles than SMs
        const long long per_sm = dtype == SSCAN_F32 ? std::min(std::max(occ, 1), 2) : 1;
        const long long target = (long long)std::max(nsm, 1) * per_sm;
        S = tiles >= target ? 1 : ceil_div((long long)std::max(nsm, 1) * std::min(std::max(occ, 1), 2), tiles);
        S = std::min(S, std::max(1LL, seqlen / (8LL * TC)));
    }
    S = std::max(1LL, std::min(S, ceil_div(seqlen, TC)));
    const long long Tseg = ceil_div(ceil_div(seqlen, S), TC) * TC;
    S = ceil_div(seqlen, Tseg);
    if (tiles * S > (1LL << 30)) return SSCAN_ERR_INVALID;

    FwdParams p{};
    p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.h0 = h0;
    p.out = out; p.final_state = final_state;
    p.batch = batch; p.dim = dim; p.L = seqlen; p.N = dstate;
    p.Tseg = Tseg; p.S = (int)S; p.tiles_per_batch = (int)tiles_per_batch;

    snprintf(g_rec.plan, sizeof(g_rec.plan),
             "sscan %s P=%d NS=%d vec=%d tiles=%lld S=%lld Tseg=%lld %s", esz == 4 ? "f32" : "bf16",
             sh.P, sh.NS, (int)vec, tiles, S, Tseg,
             S == 1 ? "single" : (dtype == SSCAN_F32 ? "local+correct" : "agg+fold"));

    cudaError_t e;
    if (S == 1) {
        p.mode = sscan::MODE_SINGLE;
        p.seg_count = 1;
        e = launch_fwd(dtype, FwdKernel::Chunked, p, sh, vec, tiles, st);
        if (e != cudaSuccess) return fail_cuda(e);
        return SSCAN_OK;
    }

    const size_t nseg = (size_t)(batch * dim) * (size_t)S;
    const size_t scratch_bytes = nseg * (size_t)(dstate + 1) * sizeof(float);
    void* scratch = nullptr;
    e = cudaMallocAsync(&scratch, scratch_bytes, st);
    if (e != cudaSuccess) return fail_cuda(e);
    p.seg_state = static_cast<float*>(scratch);
    p.seg_dsum = p.seg_state + nseg * (size_t)dstate;
    if (dtype == SSCAN_F32) {
        // pass 1: every segment from its local start, writing y and its aggregate;
        // pass 2: add the carried state's decaying contribution
        p.mode = sscan::MODE_LOCAL;
        p.seg_count = (int)S;
        e = launch_fwd(dtype, FwdKernel::Chunked, p, sh, vec, tiles * S, st);
        if (e == cudaSuccess) {
            p.mode = sscan::MODE_CORR;
            p.seg_count = (int)(S - 1);
            e = launch_fwd(dtype, FwdKernel::Chunked, p, sh, vec, tiles * (S - 1), st);
        }
    } else {
        // bf16 output is written once: aggregates first, then every segment from
        // its exact entry state
        p.mode = sscan::MODE_AGG;
        p.seg_count = (int)(S - 1);
        e = launch_fwd(dtype, FwdKernel::Chunked, p, sh, vec, tiles * (S - 1), st);
        if (e == cudaSuccess) {
            p.mode = sscan::MODE_FOLD;
            p.seg_count = (int)S;
            e = launch_fwd(dtype, FwdKernel::Chunked, p, sh, vec, tiles * S, st);
        }
    }
    cudaError_t ef = cudaFreeAsync(scratch, st);
    if (e != cudaSuccess) return fail_cuda(e);
    if (ef != cudaSuccess) return fail_cuda(ef);
    return SSCAN_OK;
}

int sscan_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
              const float* D, const float* h0, void* out, float* final_state, int64_t batch,
              int64_t dim, int64_t seqlen, int64_t dstate, int dtype, void* stream) {
    return sscan_fwd_ex(u, delta, A, B, C, D, h0, out, final_state, batch, dim, seqlen, dstate,
                        dtype, 0, 0, stream);
}

int pscan(const float* a, const float* b, float* h, const float* h0, int64_t rows, int64_t len,
          void* stream) {
    g_rec.launches = 0;
    snprintf(g_rec.plan, sizeof(g_rec.plan), "rejected");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    g_rec.stream = st;
    if (!a || !b || !h) return SSCAN_ERR_INVALID;
    const long long big = (long long)1 << 46;
    if (rows < 0 || len < 0 || rows > big || len > big || (rows && len > big / rows))
        return SSCAN_ERR_INVALID;
    if (rows == 0 || len == 0) {
        snprintf(g_rec.plan, sizeof(g_rec.plan), "empty");
        return SSCAN_OK;
    }
    const bool vec = (len % 4) == 0 && aligned16(a) && aligned16(b) && aligned16(h);
    const long long block = 128LL * sscan::kPscanUnroll;
    const long long target = (long long)std::max(sm_count(), 1) * 32;  // warps
    long long S = rows >= target ? 1 : ceil_div(target, rows);
    S = std::max(1LL, std::min(S, len / (4 * block)));
    const long long Tseg = ceil_div(ceil_div(len, S), block) * block;
    S = ceil_div(len, Tseg);
    if (ceil_div(rows * S, 4) > (1LL << 30)) return SSCAN_ERR_INVALID;

    sscan::PscanParams p{};
    p.a = a; p.b = b; p.h = h; p.h0 = h0;
    p.rows = rows; p.len = len; p.Tseg = Tseg; p.S = (int)S;
    snprintf(g_rec.plan, sizeof(g_rec.plan), "pscan vec=%d S=%lld Tseg=%lld", (int)vec, S, Tseg);

    auto launch = [&](long long units) -> cudaError_t {
        const long long grid = ceil_div(units, 4);
        ++g_rec.launches;
        if (vec) sscan::pscan_kernel<true><<<(unsigned)grid, 128, 0, st>>>(p);
        else sscan::pscan_kernel<false><<<(unsigned)grid, 128, 0, st>>>(p);
        return cudaGetLastError();
    };
    cudaError_t e;
    if (S == 1) {
        p.mode = sscan::PS_SINGLE;
        p.seg_count = 1;
        e = launch(rows);
        return e == cudaSuccess ? SSCAN_OK : fail_cuda(e);
    }
    void* scratch = nullptr;
    e = cudaMallocAsync(&scratch, (size_t)(rows * S) * 2 * sizeof(float), st);
    if (e != cudaSuccess) return fail_cuda(e);
    p.agg_a = static_cast<float*>(scratch);
    p.agg_b = p.agg_a + rows * S;
    p.mode = sscan::PS_AGG;
    p.seg_count = (int)(S - 1);
    e = launch(rows * (S - 1));
    if (e == cudaSuccess) {
        p.mode = sscan::PS_FOLD;
        p.seg_count = (int)S;
        e = launch(rows * S);
    }
    cudaError_t ef = cudaFreeAsync(scratch, st);
    if (e != cudaSuccess) return fail_cuda(e);
    if (ef != cudaSuccess) return fail_cuda(ef);
    return SSCAN_OK;
}

}  // extern "C"
