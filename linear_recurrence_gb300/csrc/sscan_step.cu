// Single-step selective-scan update (autoregressive decode) on sm_103a.
//
// One token per sequence: the cached state of every (batch, channel) is
// advanced by one step and read out, the recurrent inference step that the
// state cache of "Mamba 状态空间模型：从理论到生产级推理的 CUDA 内核优化实战"
// (section 5.1) keeps between tokens:
//     h[b,d,n] <- exp(delta[b,d]*A[d,n]) * h[b,d,n] + delta[b,d]*B[b,n]*u[b,d]
//     y[b,d]    = sum_n C[b,n]*h[b,d,n] + D[d]*u[b,d]
// The work is a streaming read-modify-write of the float32 state, so the
// kernel is bound by HBM bandwidth: a thread owns one or two groups of 4
// consecutive states of one channel (16-byte loads and stores), the threads of
// a channel sum their partial outputs with warp shuffles, and B/C rows come
// from L1/L2.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sscan.h"
#include "device_utils.cuh"

namespace sscan {
void record_call(int launches, cudaStream_t stream, const char* plan);
void record_error(cudaError_t e);
}  // namespace sscan

namespace {

using sscan::bf16;

constexpr float kLog2eStep = 1.4426950408889634f;

// Four B (or C) values starting at a 4-aligned state index: one 16-byte load
// for float, one 8-byte load for bf16 (the row start is aligned accordingly).
__device__ __forceinline__ void load4_row(const float* p, float v[4]) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void load4_row(const bf16* p, float v[4]) {
    const uint2 x = __ldg(reinterpret_cast<const uint2*>(p));
    v[0] = __uint_as_float(x.x << 16); v[1] = __uint_as_float(x.x & 0xffff0000u);
    v[2] = __uint_as_float(x.y << 16); v[3] = __uint_as_float(x.y & 0xffff0000u);
}

// Q threads per channel; each owns G groups of 4 consecutive states
// (states 4*(q + Q*g) .. +3), so a thread keeps G 16-byte state loads in
// flight.  VEC: N % 4 == 0 and every row 16-byte (B/C: element-) aligned.
template <typename T, int Q, int G, bool VEC>
__global__ void __launch_bounds__(256) sscan_step_kernel(const T* __restrict__ u, const T* __restrict__ delta,
                                                         const float* __restrict__ A,
                                                         const T* __restrict__ Bm, const T* __restrict__ Cm,
                                                         const float* __restrict__ D, float* __restrict__ state,
                                                         T* __restrict__ out, long long b0, int dim,
                                                         int N) {
    // grid: x over (channel, q) of one batch row, y over batch rows from b0
    const int tid = blockIdx.x * blockDim.x + threadIdx.x;
    const int dd = tid / Q;  // channel
    const int q = tid % Q;
    const bool valid = dd < dim;
    const long long b = b0 + blockIdx.y;
    const long long d = valid ? dd : 0;
    const long long chc = b * dim + d;  // flat (b, d)
    const float dt = valid ? sscan::to_f32(delta[chc]) : 0.f;
    const float uu = valid ? sscan::to_f32(u[chc]) : 0.f;
    const float du = dt * uu;
    float* hrow = state + chc * N;
    const float* Arow = A + d * N;
    const T* Brow = Bm + b * N;
    const T* Crow = Cm + b * N;
    float acc = 0.f;
    if (VEC) {
        float4 h4[G];
        bool on[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {       // issue every state load first
            const int n0 = 4 * (q + Q * g);
            on[g] = valid && n0 < N;
            if (on[g]) h4[g] = *reinterpret_cast<const float4*>(hrow + n0);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int n0 = 4 * (q + Q * g);
            if (!on[g]) continue;
            const float4 a4 = __ldg(reinterpret_cast<const float4*>(Arow + n0));
            float bv[4], cv[4];
            load4_row(Brow + n0, bv);
            load4_row(Crow + n0, cv);
            float4 h = h4[g];
            h.x = fmaf(sscan::ex2(dt * a4.x * kLog2eStep), h.x, du * bv[0]);
            h.y = fmaf(sscan::ex2(dt * a4.y * kLog2eStep), h.y, du * bv[1]);
            h.z = fmaf(sscan::ex2(dt * a4.z * kLog2eStep), h.z, du * bv[2]);
            h.w = fmaf(sscan::ex2(dt * a4.w * kLog2eStep), h.w, du * bv[3]);
            acc = fmaf(cv[0], h.x, fmaf(cv[1], h.y, fmaf(cv[2], h.z, fmaf(cv[3], h.w, acc))));
            *reinterpret_cast<float4*>(hrow + n0) = h;
        }
    } else {
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = 4 * (q + Q * g) + j;
                if (valid && n < N) {
                    const float a = sscan::ex2(dt * Arow[n] * kLog2eStep);
                    const float hn = fmaf(a, hrow[n], du * sscan::to_f32(Brow[n]));
                    hrow[n] = hn;
                    acc = fmaf(sscan::to_f32(Crow[n]), hn, acc);
                }
            }
        }
    }
#pragma unroll
    for (int off = Q / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, Q);
    if (valid && q == 0) {
        const float y = fmaf(D != nullptr ? D[d] : 0.f, uu, acc);
        out[chc] = sscan::from_f32<T>(y);
    }
}

// G = 2 groups per thread once N > 4 (two 16-byte state loads in flight per
// thread); Q = the smallest power of two with 4*G*Q >= N (1 .. 8 for N <= 64).
template <typename T>
cudaError_t launch_step(const void* u, const void* delta, const float* A, const void* B, const void* C,
                        const float* D, float* state, void* out, long long batch, long long dim, int N,
                        bool vec, cudaStream_t st) {
    const int G = N > 4 ? 2 : 1;
    int Q = 1;
    while (Q * 4 * G < N) Q *= 2;
    if (dim * Q > (1LL << 30)) return cudaErrorInvalidValue;
    const unsigned gx = (unsigned)((dim * Q + 255) / 256);
    const T* tu = static_cast<const T*>(u);
    const T* td = static_cast<const T*>(delta);
    const T* tB = static_cast<const T*>(B);
    const T* tC = static_cast<const T*>(C);
    T* to = static_cast<T*>(out);
    // batch rows go to grid.y, at most 65535 per launch
#define SSCAN_STEP_CASE(QQ, GG)                                                                     \
    if (Q == QQ && G == GG) {                                                                       \
        for (long long b0 = 0; b0 < batch; b0 += 65535) {                                           \
            const dim3 grid(gx, (unsigned)(batch - b0 < 65535 ? batch - b0 : 65535));              \
            if (vec)                                                                                \
                sscan_step_kernel<T, QQ, GG, true><<<grid, 256, 0, st>>>(tu, td, A, tB, tC, D, state, to, b0, (int)dim, N); \
            else                                                                                    \
                sscan_step_kernel<T, QQ, GG, false><<<grid, 256, 0, st>>>(tu, td, A, tB, tC, D, state, to, b0, (int)dim, N); \
            const cudaError_t e = cudaGetLastError();                                               \
            if (e != cudaSuccess) return e;                                                         \
        }                                                                                           \
        return cudaSuccess;                                                                         \
    }
    SSCAN_STEP_CASE(1, 1) SSCAN_STEP_CASE(1, 2) SSCAN_STEP_CASE(2, 2) SSCAN_STEP_CASE(4, 2)
    SSCAN_STEP_CASE(8, 2)
#undef SSCAN_STEP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

extern "C" int sscan_step(const void* u, const void* delta, const float* A, const void* B, const void* C,
                          const float* D, float* state, void* out, int64_t batch, int64_t dim,
                          int64_t dstate, int dtype, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    sscan::record_call(0, st, "rejected");
    if (dtype != SSCAN_F32 && dtype != SSCAN_BF16) return SSCAN_ERR_INVALID;
    if (batch < 0 || dim < 0 || dstate < 1 || dstate > sscan_max_dstate()) return SSCAN_ERR_INVALID;
    const long long big = (long long)1 << 40;
    if (batch > big || dim > big || (batch && dim > big / batch)) return SSCAN_ERR_INVALID;
    if (batch == 0 || dim == 0) {
        sscan::record_call(0, st, "empty");
        return SSCAN_OK;
    }
    if (!u || !delta || !A || !B || !C || !state || !out) return SSCAN_ERR_INVALID;
    const uintptr_t rows_align = dtype == SSCAN_F32 ? 15u : 7u;
    const bool vec = (dstate % 4) == 0 && (reinterpret_cast<uintptr_t>(state) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(A) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(B) & rows_align) == 0 &&
                     (reinterpret_cast<uintptr_t>(C) & rows_align) == 0;
    sscan::record_call((int)((batch + 65534) / 65535), st, vec ? "step vec=1" : "step vec=0");
    const cudaError_t e =
        dtype == SSCAN_F32
            ? launch_step<float>(u, delta, A, B, C, D, state, out, batch, dim, (int)dstate, vec, st)
            : launch_step<bf16>(u, delta, A, B, C, D, state, out, batch, dim, (int)dstate, vec, st);
    if (e != cudaSuccess) {
        sscan::record_error(e);
        return SSCAN_ERR_CUDA;
    }
    return SSCAN_OK;
}
