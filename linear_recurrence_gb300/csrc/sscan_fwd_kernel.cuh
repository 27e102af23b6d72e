// Fused selective-scan forward kernels for sm_103a.
//
// What is computed (the selective_scan pseudocode of "Mamba 状态空间模型：从理论
// 到生产级推理的 CUDA 内核优化实战", section 2.3, with the initial/final state of
// its section 7.1): per batch b, channel d, state n and step t
//     h_t[n] = exp(delta_t * A[d,n]) * h_{t-1}[n] + (delta_t * u_t) * B[b,n,t]
//     y_t    = sum_n C[b,n,t] * h_t[n] + D[d] * u_t
//
// Work decomposition (diagonal A makes every (b, d, n) an independent chain,
// "为什么Mamba的“并行扫描”不是真并行" section 1):
//   * a lane owns one channel and NS of its states (P lanes share a channel;
//     lane g of the group owns states n = k*P + g), keeping h in registers;
//   * a warp covers 32/P channels, a CTA of 4 warps covers DT channels and
//     walks time in chunks of TC steps; u/delta tiles [DT x TC] and the B/C
//     tile [N x TC] of the chunk are staged in shared memory by cp.async
//     (multi-stage ring) and the B/C tile is reused by every channel of the CTA
//     (the fusion of discretisation, scan and C-contraction of "并行扫描与硬件
//     感知优化 (mhpq.cn/news/1077344)" section 3.2, with the double buffering
//     of the CUDA page's section 4.3 generalised to a ring);
//   * the C-contraction's partial sums of the P lanes of a channel are
//     combined by a shuffle reduce-scatter over 4 steps, so each lane writes
//     one output; outputs are staged in shared memory and stored as 16-byte
//     vectors;
//   * long sequences with few channels are split into S time segments
//     (the chunked scan of "并行扫描与硬件感知优化" section 2.4).  Segments carry
//     their aggregate (prod_t exp(delta_t A) = 2^(A log2e * sum_t delta_t),
//     h_end) -- the chunk-carry identity of "为什么Mamba的“并行扫描”不是真并行"
//     section 3 -- and the state entering a segment is the fold of the
//     aggregates before it, i.e. the associative operator
//     (a1,b1) o (a2,b2) = (a2 a1, a2 b1 + b2) applied in order.
#pragma once

#include "device_utils.cuh"

namespace sscan {

enum FwdMode : int {
    MODE_SINGLE = 0,  // one segment: start from h0, write y and final_state
    MODE_LOCAL = 1,   // segment s starts from h0 (s = 0) or 0; write y and the
                      // segment aggregate; a MODE_CORR launch adds the carry
    MODE_AGG = 2,     // like MODE_LOCAL but only the aggregate (no y)
    MODE_FOLD = 3,    // segment s starts from the fold of segments < s; write y;
                      // the last segment writes final_state
    MODE_CORR = 4     // after MODE_LOCAL: segment s >= 1 adds the decaying carry of
                      // its entry state to the outputs already written (read back
                      // through the u slot), until the carry has decayed below
                      // 2^-24 of its entry magnitude; the last segment writes
                      // final_state
};

struct FwdParams {
    const void* u;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const float* h0;
    void* out;
    float* final_state;
    float* seg_state;  // [batch*dim, S, N]  state at the end of each segment
    float* seg_dsum;   // [batch*dim, S]     sum of delta over each segment
    long long batch, dim, L, N;
    long long Tseg;    // steps per segment (multiple of TC)
    int S;             // segments per channel
    int tiles_per_batch;
    int mode;
    int seg_count;     // segments covered by this grid: grid = tiles * seg_count
};

constexpr float kLog2e = 1.4426950408889634f;

#ifndef SSCAN_STEP_UNROLL
#define SSCAN_STEP_UNROLL 8
#endif
// Steps per unrolled iteration of the inner loop (a multiple of 4).
constexpr int kStepUnroll = SSCAN_STEP_UNROLL;
#ifndef SSCAN_MAX_CHUNK
#define SSCAN_MAX_CHUNK 32
#endif
// Largest number of steps staged per chunk (16 or 32).
constexpr int kMaxChunk = SSCAN_MAX_CHUNK;

template <typename T, int NS_, int P_>
struct FwdCfg {
    static constexpr int NS = NS_;
    static constexpr int P = P_;
    static constexpr int kWarps = 2;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int PPW = 32 / P;                // channel pairs per warp
    static constexpr int CPW = 2 * PPW;               // channels per warp
    static constexpr int DT = kWarps * CPW;           // channels per CTA
    static constexpr int NSP = NS * P;                // state slots per channel
    static constexpr int TC = (DT > 64 || kMaxChunk < 32) ? 16 : 32;  // steps per chunk
    static constexpr int VECE = 16 / (int)sizeof(T);  // elements per 16 bytes
    static constexpr int RROW = TC + VECE;            // raw smem row (T), padded by 16 B
    static constexpr int PPR = TC / VECE;             // 16-byte pieces per raw row
    static constexpr int UROW = 2 * TC + 4;           // interleaved u/delta row of a channel pair
    static constexpr int GS = NS + ((P == 4 && NS >= 16) ? 4 : 0);  // floats per state group
    static constexpr int RB = P * GS;                 // floats per B/C work row (one step)
    static constexpr int RAW_ELEMS = (2 * DT + 2 * NSP) * RROW;
    static constexpr int RAW_BYTES = RAW_ELEMS * (int)sizeof(T);
    static constexpr int UW_FLOATS = (DT / 2) * UROW;  // one of u, delta
    static constexpr int BW_FLOATS = TC * RB;          // one of B, C
    static constexpr int WORK_FLOATS = 2 * UW_FLOATS + 2 * BW_FLOATS;
    static constexpr int Y_ELEMS = DT * RROW;
    static constexpr int FIXED_BYTES = 2 * WORK_FLOATS * 4 + 2 * Y_ELEMS * (int)sizeof(T);
    static constexpr int STAGES = (RAW_BYTES * 4 + FIXED_BYTES <= 48 * 1024) ? 4
                                  : (RAW_BYTES * 3 + FIXED_BYTES <= 72 * 1024) ? 3
                                                                               : 2;
    static constexpr int SMEM_BYTES = STAGES * RAW_BYTES + FIXED_BYTES;
    static_assert(32 % P == 0, "lanes per channel must divide the warp");
    static_assert(NS % 4 == 0, "state slots are read 4 at a time");
    static_assert(TC % VECE == 0 && TC % 4 == 0, "chunk must hold whole vectors");
    static_assert((RROW * sizeof(T)) % 16 == 0, "smem rows must stay 16-byte aligned");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// State entering segment s (s >= 1) for states n = g*NS + k of one channel: the
// fold of the aggregates of segments 0 .. s-1 (segment 0's entry holds its true
// end state because it started from h0).
template <int NS>
__device__ __forceinline__ void fold_segments(const FwdParams& p, long long ch, int s, int g,
                                              const float (&Al2)[NS], float (&h)[NS]) {
    const float* st = p.seg_state + ch * p.S * p.N;
    const float* ds = p.seg_dsum + ch * p.S;
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        const long long n = (long long)g * NS + k;
        h[k] = n < p.N ? st[n] : 0.f;
    }
    for (int sp = 1; sp < s; ++sp) {
        const float dsum = ds[sp];
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const long long n = (long long)g * NS + k;
            const float bagg = n < p.N ? st[(long long)sp * p.N + n] : 0.f;
            h[k] = fmaf(ex2(Al2[k] * dsum), h[k], bagg);
        }
    }
}

// Shared-memory layout of the chunked kernel:
//   raw ring [STAGES]: u [DT][RROW], delta [DT][RROW], B [NSP][RROW], C [NSP][RROW]
//                      (type T, copied verbatim from global by cp.async)
//   work [2]:          u, delta [DT/2][UROW]: the two channels of a pair interleaved
//                        per step (u0[t], u1[t], u0[t+1], ...), fp32;
//                      B, C [TC][RB]: fp32, transposed so that a lane's NS states at
//                        one step are contiguous, group g at g*GS
//   ybuf [2]:          y [DT][RROW] (type T)
template <typename T, int NS, int P>
struct Smem {
    using Cfg = FwdCfg<T, NS, P>;
    T* raw;
    float* work;
    T* ybuf;
    __device__ __forceinline__ explicit Smem(unsigned char* base)
        : raw(reinterpret_cast<T*>(base)),
          work(reinterpret_cast<float*>(base + Cfg::STAGES * Cfg::RAW_BYTES)),
          ybuf(reinterpret_cast<T*>(base + Cfg::STAGES * Cfg::RAW_BYTES + 2 * Cfg::WORK_FLOATS * 4)) {}
    __device__ __forceinline__ T* stage(int i) const { return raw + (i % Cfg::STAGES) * Cfg::RAW_ELEMS; }
    __device__ __forceinline__ float* wk(int i) const { return work + (i & 1) * Cfg::WORK_FLOATS; }
    __device__ __forceinline__ T* yb(int i) const { return ybuf + (i & 1) * Cfg::Y_ELEMS; }
};

// B/C work-tile column of state n: group n / NS, slot n % NS.
template <int NS, int GS>
__device__ __forceinline__ int work_col(int n) { return (n / NS) * GS + (n % NS); }

// VEC path, step 1: issue this thread's 16-byte cp.async pieces of chunk [t0, t0+TC).
// A thread owns the same piece of both rows of a channel pair, and whole B/C
// pieces.  Out-of-range pieces are zero-filled (delta = 0 keeps the state).
template <typename T, int NS, int P, bool LOAD_C, bool LOAD_B = true>
__device__ __forceinline__ void issue_chunk(const FwdParams& p, T* st, long long b, long long d0,
                                            long long t0, long long t_end, int tid) {
    using Cfg = FwdCfg<T, NS, P>;
    constexpr int DT = Cfg::DT, RROW = Cfg::RROW, NSP = Cfg::NSP, PPR = Cfg::PPR, VE = Cfg::VECE;
    const T* gu = static_cast<const T*>(p.u);
    const T* gd = static_cast<const T*>(p.delta);
    const T* gB = static_cast<const T*>(p.B);
    const T* gC = static_cast<const T*>(p.C);
    T* su = st;
    T* sd = st + DT * RROW;
    T* sB = st + 2 * DT * RROW;
    T* sC = sB + NSP * RROW;
    for (int q = tid; q < (DT / 2) * PPR; q += Cfg::kThreads) {
        const int pr = q / PPR, pc = q % PPR;
        const long long t = t0 + (long long)pc * VE;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 2 * pr + e;
            const long long dd = d0 + r;
            const bool ok = dd < p.dim && t < t_end;
            const long long off = (b * p.dim + (ok ? dd : 0)) * p.L + (ok ? t : 0);
            cp_async16(su + r * RROW + pc * VE, gu + off, ok ? 16 : 0);
            cp_async16(sd + r * RROW + pc * VE, gd + off, ok ? 16 : 0);
        }
    }
    const int N = (int)p.N;
    for (int q = tid; q < N * PPR; q += Cfg::kThreads) {
        const int n = q / PPR, pc = q % PPR;
        const long long t = t0 + (long long)pc * VE;
        const bool ok = t < t_end;
        const long long off = (b * p.N + n) * p.L + (ok ? t : 0);
        if (LOAD_B) cp_async16(sB + n * RROW + pc * VE, gB + off, ok ? 16 : 0);
        if (LOAD_C) cp_async16(sC + n * RROW + pc * VE, gC + off, ok ? 16 : 0);
    }
}

// VEC path, step 2 (after this thread's copies of the chunk landed): widen the
// pieces this same thread copied into the fp32 work tiles (u/delta interleaved
// by channel pair, B/C transposed).  Only own pieces are touched, so no barrier
// is needed between the copy and the conversion.
template <typename T, int NS, int P, bool LOAD_C, bool LOAD_B = true>
__device__ __forceinline__ void convert_own_pieces(const FwdParams& p, const T* st, float* wk, int tid) {
    using Cfg = FwdCfg<T, NS, P>;
    constexpr int DT = Cfg::DT, RROW = Cfg::RROW, NSP = Cfg::NSP, PPR = Cfg::PPR, VE = Cfg::VECE;
    constexpr int UROW = Cfg::UROW, RB = Cfg::RB, GS = Cfg::GS;
    const T* su = st;
    const T* sd = st + DT * RROW;
    const T* sB = st + 2 * DT * RROW;
    const T* sC = sB + NSP * RROW;
    float* wu = wk;
    float* wd = wk + Cfg::UW_FLOATS;
    float* wB = wk + 2 * Cfg::UW_FLOATS;
    float* wC = wB + Cfg::BW_FLOATS;
    for (int q = tid; q < (DT / 2) * PPR; q += Cfg::kThreads) {
        const int pr = q / PPR, pc = q % PPR;
#pragma unroll
        for (int e = 0; e < VE; e += 4) {
            float a0[4], a1[4];
            load4_smem(su + (2 * pr) * RROW + pc * VE + e, a0);
            load4_smem(su + (2 * pr + 1) * RROW + pc * VE + e, a1);
            float* o = wu + pr * UROW + 2 * (pc * VE + e);
            *reinterpret_cast<float4*>(o) = make_float4(a0[0], a1[0], a0[1], a1[1]);
            *reinterpret_cast<float4*>(o + 4) = make_float4(a0[2], a1[2], a0[3], a1[3]);
            load4_smem(sd + (2 * pr) * RROW + pc * VE + e, a0);
            load4_smem(sd + (2 * pr + 1) * RROW + pc * VE + e, a1);
            o = wd + pr * UROW + 2 * (pc * VE + e);
            *reinterpret_cast<float4*>(o) = make_float4(a0[0], a1[0], a0[1], a1[1]);
            *reinterpret_cast<float4*>(o + 4) = make_float4(a0[2], a1[2], a0[3], a1[3]);
        }
    }
    const int N = (int)p.N;
    for (int q = tid; q < N * PPR; q += Cfg::kThreads) {
        const int n = q / PPR, pc = q % PPR;
        const int col = work_col<NS, GS>(n);
#pragma unroll
        for (int e = 0; e < VE; e += 4) {
            float v[4];
            if (LOAD_B) {
                load4_smem(sB + n * RROW + pc * VE + e, v);
#pragma unroll
                for (int j = 0; j < 4; ++j) wB[(pc * VE + e + j) * RB + col] = v[j];
            }
            if (LOAD_C) {
                load4_smem(sC + n * RROW + pc * VE + e, v);
#pragma unroll
                for (int j = 0; j < 4; ++j) wC[(pc * VE + e + j) * RB + col] = v[j];
            }
        }
    }
}

// Non-VEC path (rows not 16-byte aligned): synchronous element loads with bounds
// checks straight into the fp32 work tiles.
template <typename T, int NS, int P, bool LOAD_C, bool LOAD_B = true>
__device__ __forceinline__ void load_chunk_scalar(const FwdParams& p, float* wk, long long b,
                                                  long long d0, long long t0, long long t_end, int tid) {
    using Cfg = FwdCfg<T, NS, P>;
    constexpr int DT = Cfg::DT, TC = Cfg::TC, UROW = Cfg::UROW, RB = Cfg::RB, GS = Cfg::GS;
    const T* gu = static_cast<const T*>(p.u);
    const T* gd = static_cast<const T*>(p.delta);
    const T* gB = static_cast<const T*>(p.B);
    const T* gC = static_cast<const T*>(p.C);
    float* wu = wk;
    float* wd = wk + Cfg::UW_FLOATS;
    float* wB = wk + 2 * Cfg::UW_FLOATS;
    float* wC = wB + Cfg::BW_FLOATS;
    for (int q = tid; q < DT * TC; q += Cfg::kThreads) {
        const int r = q / TC, tt = q % TC;
        const long long dd = d0 + r, t = t0 + tt;
        const bool ok = dd < p.dim && t < t_end;
        const long long off = (b * p.dim + dd) * p.L + t;
        wu[(r / 2) * UROW + 2 * tt + (r & 1)] = ok ? to_f32(gu[off]) : 0.f;
        wd[(r / 2) * UROW + 2 * tt + (r & 1)] = ok ? to_f32(gd[off]) : 0.f;
    }
    const int N = (int)p.N;
    for (int q = tid; q < N * TC; q += Cfg::kThreads) {
        const int n = q % N, tt = q / N;
        const long long t = t0 + tt;
        const bool ok = t < t_end;
        const long long off = (b * p.N + n) * p.L + t;
        const int col = work_col<NS, GS>(n);
        if (LOAD_B) wB[tt * RB + col] = ok ? to_f32(gB[off]) : 0.f;
        if (LOAD_C) wC[tt * RB + col] = ok ? to_f32(gC[off]) : 0.f;
    }
}

// Write a staged output chunk [DT x TC] to global memory.
template <typename T, int NS, int P, bool VEC>
__device__ __forceinline__ void store_chunk(const FwdParams& p, const T* ys, long long b,
                                            long long d0, long long t0, long long t_end, int tid) {
    using Cfg = FwdCfg<T, NS, P>;
    constexpr int DT = Cfg::DT, RROW = Cfg::RROW;
    T* go = static_cast<T*>(p.out);
    if constexpr (VEC) {
        constexpr int PPR = Cfg::PPR, VE = Cfg::VECE;
        for (int q = tid; q < DT * PPR; q += Cfg::kThreads) {
            const int r = q / PPR, pc = q % PPR;
            const long long dd = d0 + r, t = t0 + (long long)pc * VE;
            if (dd < p.dim && t < t_end)
                *reinterpret_cast<uint4*>(go + (b * p.dim + dd) * p.L + t) =
                    *reinterpret_cast<const uint4*>(ys + r * RROW + pc * VE);
        }
    } else {
        constexpr int TC = Cfg::TC;
        for (int q = tid; q < DT * TC; q += Cfg::kThreads) {
            const int r = q / TC, tt = q % TC;
            const long long dd = d0 + r, t = t0 + tt;
            if (dd < p.dim && t < t_end) go[(b * p.dim + dd) * p.L + t] = ys[r * RROW + tt];
        }
    }
}

// Combine the P lanes' partial outputs of 4 consecutive steps (a shuffle
// reduce-scatter).  Afterwards lane g of a 4-lane group holds step g in v[0];
// lane g of a 2-lane group holds steps 2g, 2g+1 in v[0], v[1]; a lone lane
// holds all four.
template <int P>
__device__ __forceinline__ void reduce4(const float (&y)[4], int g, float (&v)[4]) {
    constexpr unsigned FULL = 0xffffffffu;
    if constexpr (P == 4) {
        const bool hi = (g & 2) != 0;
        const float k0 = hi ? y[2] : y[0], k1 = hi ? y[3] : y[1];
        const float s0 = hi ? y[0] : y[2], s1 = hi ? y[1] : y[3];
        const float r0 = k0 + __shfl_xor_sync(FULL, s0, 2);
        const float r1 = k1 + __shfl_xor_sync(FULL, s1, 2);
        const bool odd = (g & 1) != 0;
        const float kv = odd ? r1 : r0;
        const float sv = odd ? r0 : r1;
        v[0] = kv + __shfl_xor_sync(FULL, sv, 1);
    } else if constexpr (P == 2) {
        const bool hi = (g & 1) != 0;
        const float k0 = hi ? y[2] : y[0], k1 = hi ? y[3] : y[1];
        const float s0 = hi ? y[0] : y[2], s1 = hi ? y[1] : y[3];
        v[0] = k0 + __shfl_xor_sync(FULL, s0, 1);
        v[1] = k1 + __shfl_xor_sync(FULL, s1, 1);
    } else {
        v[0] = y[0]; v[1] = y[1]; v[2] = y[2]; v[3] = y[3];
    }
}

// Reduce-scatter one channel's 4 partial outputs, add the skip term D*u once
// (by the lane that owns each step), and write the lane's share of the staged
// output row (yrow points at the first of the 4 steps).
template <typename T, int P>
__device__ __forceinline__ void reduce_write4(const float (&y)[4], const float (&u)[4], float Dd, int g,
                                              T* yrow) {
    float v[4];
    reduce4<P>(y, g, v);
    if constexpr (P == 4) {
        const float ug = (g & 2) ? ((g & 1) ? u[3] : u[2]) : ((g & 1) ? u[1] : u[0]);
        yrow[g] = from_f32<T>(fmaf(Dd, ug, v[0]));
    } else if constexpr (P == 2) {
        const float u0 = g ? u[2] : u[0], u1 = g ? u[3] : u[1];
        yrow[2 * g] = from_f32<T>(fmaf(Dd, u0, v[0]));
        yrow[2 * g + 1] = from_f32<T>(fmaf(Dd, u1, v[1]));
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) yrow[j] = from_f32<T>(fmaf(Dd, u[j], v[j]));
    }
}

// One chunk of the recurrence for the calling lane: channel pair pr (rows 2pr,
// 2pr+1 of the tile; index e below), states n = g*NS + k.  Each B/C value read
// from shared memory serves both channels of the pair.  Software-pipelined:
// step t+1's loads and exponentials are issued before step t's state updates,
// so the dependent FMA chain overlaps independent work.  Arithmetic is scalar
// FP32 (on this part two scalar FFMAs outrun one packed f32x2 FFMA).  SCALAR:
// every state of a channel shares its decay rate (one exponent per channel and
// step).  Returns the chunk's sum of delta per channel when DSUM.  NO_B: the
// homogeneous recurrence h = a*h (the carry correction), B is not read.
template <typename T, int NS, int P, bool WRITE_Y, bool SCALAR, bool DSUM, bool NO_B = false>
__device__ __forceinline__ float2 compute_chunk(const float* wk, T* yb, int pr, int g,
                                                const float (&A)[2][NS], const float (&As)[2],
                                                float (&h)[2][NS], const float (&Dd)[2]) {
    using Cfg = FwdCfg<T, NS, P>;
    constexpr int TC = Cfg::TC, UROW = Cfg::UROW, RB = Cfg::RB, GS = Cfg::GS, RROW = Cfg::RROW;
    const float* ur = wk + pr * UROW;
    const float* dr = wk + Cfg::UW_FLOATS + pr * UROW;
    const float* bb = wk + 2 * Cfg::UW_FLOATS + g * GS;
    const float* cb = bb + Cfg::BW_FLOATS;
    T* yrow0 = yb + (2 * pr) * RROW;
    T* yrow1 = yrow0 + RROW;

    // Two register sets (ping-pong): while step t is applied from one set, step
    // t+1 is fetched into the other, so no values are copied between steps.
    struct StepRegs {
        float a[2][NS];
        float du[2], u[2];
        float4 b[NS / 4], c[NS / 4];
    };
    StepRegs r0, r1;
    float2 csum = make_float2(0.f, 0.f);
    auto fetch = [&](StepRegs& r, int t) {
        const float2 u2 = *reinterpret_cast<const float2*>(ur + 2 * t);
        const float2 d2 = *reinterpret_cast<const float2*>(dr + 2 * t);
        if (DSUM) { csum.x += d2.x; csum.y += d2.y; }
        r.u[0] = u2.x; r.u[1] = u2.y;
        r.du[0] = d2.x * u2.x; r.du[1] = d2.y * u2.y;
#pragma unroll
        for (int q = 0; q < NS / 4; ++q) {
            if (!NO_B) r.b[q] = *reinterpret_cast<const float4*>(bb + t * RB + 4 * q);
            if (WRITE_Y) r.c[q] = *reinterpret_cast<const float4*>(cb + t * RB + 4 * q);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float dt = e ? d2.y : d2.x;
            if (SCALAR) {
                const float a = ex2(dt * As[e]);
#pragma unroll
                for (int k = 0; k < NS; ++k) r.a[e][k] = a;
            } else {
#pragma unroll
                for (int k = 0; k < NS; ++k) r.a[e][k] = ex2(dt * A[e][k]);
            }
        }
    };
    float y[2][4], uu[2][4];
    auto apply = [&](const StepRegs& r, int t) {
        float acc[2] = {0.f, 0.f};
#pragma unroll
        for (int q = 0; q < NS / 4; ++q) {
            float bv[4] = {0.f, 0.f, 0.f, 0.f};
            if (!NO_B) { bv[0] = r.b[q].x; bv[1] = r.b[q].y; bv[2] = r.b[q].z; bv[3] = r.b[q].w; }
            float cv[4] = {0.f, 0.f, 0.f, 0.f};
            if (WRITE_Y) { cv[0] = r.c[q].x; cv[1] = r.c[q].y; cv[2] = r.c[q].z; cv[3] = r.c[q].w; }
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = 4 * q + j;
                    if (NO_B) h[e][k] = r.a[e][k] * h[e][k];
                    else h[e][k] = fmaf(r.a[e][k], h[e][k], r.du[e] * bv[j]);
                    if (WRITE_Y) acc[e] = fmaf(cv[j], h[e][k], acc[e]);
                }
        }
        if (WRITE_Y) {
            y[0][t & 3] = acc[0];
            y[1][t & 3] = acc[1];
            uu[0][t & 3] = r.u[0];
            uu[1][t & 3] = r.u[1];
            if ((t & 3) == 3) {
                reduce_write4<T, P>(y[0], uu[0], Dd[0], g, yrow0 + (t & ~3));
                reduce_write4<T, P>(y[1], uu[1], Dd[1], g, yrow1 + (t & ~3));
            }
        }
    };
    fetch(r0, 0);
#pragma unroll kStepUnroll / 2
    for (int t = 0; t < TC; t += 2) {
        fetch(r1, t + 1);  // TC is even
        apply(r0, t);
        if (t + 2 < TC) fetch(r0, t + 2);
        apply(r1, t + 1);
    }
    return csum;
}

template <typename T, int NS, int P, bool VEC>
__global__ void __launch_bounds__(FwdCfg<T, NS, P>::kThreads) sscan_fwd_chunked(const FwdParams p) {
    using Cfg = FwdCfg<T, NS, P>;
    constexpr int DT = Cfg::DT, TC = Cfg::TC, RB = Cfg::RB, GS = Cfg::GS, NSP = Cfg::NSP;
    constexpr int STAGES = Cfg::STAGES;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const Smem<T, NS, P> sm(smem_raw);

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int g = lane % P;
    const int pr = w * Cfg::PPW + lane / P;  // channel pair within the tile
    const bool corr = p.mode == MODE_CORR;
    const int tile = blockIdx.x / p.seg_count;
    const int s = (corr ? 1 : 0) + blockIdx.x % p.seg_count;
    const long long b = tile / p.tiles_per_batch;
    const long long d0 = (long long)(tile % p.tiles_per_batch) * DT;
    const long long t_begin = (long long)s * p.Tseg;
    const long long t_end = min(p.L, t_begin + p.Tseg);
    const int nchunks = t_end > t_begin ? (int)((t_end - t_begin + TC - 1) / TC) : 0;
    const bool write_y = p.mode != MODE_AGG;
    const bool dsum_on = p.mode == MODE_LOCAL || p.mode == MODE_AGG;
    // the correction reads back the local outputs through the u slot
    FwdParams q = p;
    if (corr) q.u = p.out;

    // the lane's two channels and their decay rates (A * log2 e); a warp whose
    // channels each have a single rate takes the one-exponent-per-step path
    long long dch[2], ch[2];
    bool dval[2];
    float A[2][NS], As[2], Dd[2], h[2][NS];
    bool uniform_rate = true;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        dch[e] = d0 + 2 * pr + e;
        dval[e] = dch[e] < p.dim;
        ch[e] = b * p.dim + (dval[e] ? dch[e] : 0);
        const float a_first = dval[e] ? p.A[dch[e] * p.N] : 0.f;
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const long long n = (long long)g * NS + k;
            const bool nv = dval[e] && n < p.N;
            const float a = nv ? p.A[dch[e] * p.N + n] : a_first;
            uniform_rate &= (a == a_first);
            A[e][k] = nv ? a * kLog2e : 0.f;
        }
        As[e] = a_first * kLog2e;
        Dd[e] = corr ? 1.f : ((p.D != nullptr && dval[e]) ? p.D[dch[e]] : 0.f);
        if ((p.mode == MODE_FOLD || corr) && s > 0) {
            fold_segments<NS>(p, ch[e], s, g, A[e], h[e]);
            if (!dval[e]) {
#pragma unroll
                for (int k = 0; k < NS; ++k) h[e][k] = 0.f;
            }
        } else {
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const long long n = (long long)g * NS + k;
                h[e][k] = (s == 0 && p.h0 != nullptr && dval[e] && n < p.N) ? p.h0[ch[e] * p.N + n] : 0.f;
            }
        }
    }
    const bool scalar = __all_sync(FULL, uniform_rate);

    // correction: the last segment's final state is the carry decayed over the
    // segment plus its local end state; the carry is followed until every
    // state of the CTA has fallen below 2^-24 of its entry magnitude
    float thr[2] = {0.f, 0.f};
    if (corr) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float m = 0.f;
#pragma unroll
            for (int k = 0; k < NS; ++k) m = fmaxf(m, fabsf(h[e][k]));
            thr[e] = m * 0x1p-24f;
            if (dval[e] && s == p.S - 1 && p.final_state != nullptr) {
                const float ds = p.seg_dsum[ch[e] * p.S + s];
                const float* sst = p.seg_state + (ch[e] * p.S + s) * p.N;
#pragma unroll
                for (int k = 0; k < NS; ++k) {
                    const long long n = (long long)g * NS + k;
                    if (n < p.N) p.final_state[ch[e] * p.N + n] = fmaf(ex2(A[e][k] * ds), h[e][k], sst[n]);
                }
            }
        }
    }

    // B/C columns of state slots >= N stay zero for the whole kernel
    if ((int)p.N < NSP) {
        const int nz = NSP - (int)p.N;
        for (int q = tid; q < 2 * 2 * TC * nz; q += Cfg::kThreads) {
            const int n = (int)p.N + q % nz;
            const int row = q / nz;  // [buf][B|C][t]
            const int buf = row / (2 * TC), rr = row % (2 * TC);
            float* wbase = sm.work + buf * Cfg::WORK_FLOATS + 2 * Cfg::UW_FLOATS;
            wbase[rr * RB + work_col<NS, GS>(n)] = 0.f;
        }
    }

    // prologue: chunks 0 .. STAGES-2 in flight, chunk 0 converted
    if constexpr (VEC) {
#pragma unroll
        for (int j = 0; j < STAGES - 1; ++j) {
            if (j < nchunks) {
                if (corr) issue_chunk<T, NS, P, true, false>(q, sm.stage(j), b, d0, t_begin + (long long)j * TC, t_end, tid);
                else if (write_y) issue_chunk<T, NS, P, true>(q, sm.stage(j), b, d0, t_begin + (long long)j * TC, t_end, tid);
                else issue_chunk<T, NS, P, false>(q, sm.stage(j), b, d0, t_begin + (long long)j * TC, t_end, tid);
            }
            cp_async_commit();
        }
        cp_async_wait<STAGES - 2>();
        if (nchunks > 0) {
            if (corr) convert_own_pieces<T, NS, P, true, false>(q, sm.stage(0), sm.wk(0), tid);
            else if (write_y) convert_own_pieces<T, NS, P, true>(q, sm.stage(0), sm.wk(0), tid);
            else convert_own_pieces<T, NS, P, false>(q, sm.stage(0), sm.wk(0), tid);
        }
    } else {
        if (nchunks > 0) {
            if (corr) load_chunk_scalar<T, NS, P, true, false>(q, sm.wk(0), b, d0, t_begin, t_end, tid);
            else if (write_y) load_chunk_scalar<T, NS, P, true>(q, sm.wk(0), b, d0, t_begin, t_end, tid);
            else load_chunk_scalar<T, NS, P, false>(q, sm.wk(0), b, d0, t_begin, t_end, tid);
        }
    }

    float2 dsum = make_float2(0.f, 0.f), dcomp = make_float2(0.f, 0.f);  // Kahan sums of delta
    int done = 0;  // chunks computed (the correction may stop early)
    for (int i = 0; i < nchunks; ++i) {
        if (corr) {
            bool live = false;
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int k = 0; k < NS; ++k) live |= fabsf(h[e][k]) > thr[e];
            if (!__syncthreads_or(live)) break;
        } else {
            __syncthreads();
        }
        const long long t0 = t_begin + (long long)i * TC;
        if (write_y && i > 0) store_chunk<T, NS, P, VEC>(p, sm.yb(i - 1), b, d0, t0 - TC, t_end, tid);
        if constexpr (VEC) {
            const int nx = i + STAGES - 1;
            if (nx < nchunks) {
                if (corr) issue_chunk<T, NS, P, true, false>(q, sm.stage(nx), b, d0, t_begin + (long long)nx * TC, t_end, tid);
                else if (write_y) issue_chunk<T, NS, P, true>(q, sm.stage(nx), b, d0, t_begin + (long long)nx * TC, t_end, tid);
                else issue_chunk<T, NS, P, false>(q, sm.stage(nx), b, d0, t_begin + (long long)nx * TC, t_end, tid);
            }
            cp_async_commit();
        }
        float2 csum = make_float2(0.f, 0.f);
        if (corr) {
            if (scalar) compute_chunk<T, NS, P, true, true, false, true>(sm.wk(i), sm.yb(i), pr, g, A, As, h, Dd);
            else compute_chunk<T, NS, P, true, false, false, true>(sm.wk(i), sm.yb(i), pr, g, A, As, h, Dd);
        } else if (write_y) {
            if (scalar) {
                if (dsum_on) csum = compute_chunk<T, NS, P, true, true, true>(sm.wk(i), sm.yb(i), pr, g, A, As, h, Dd);
                else compute_chunk<T, NS, P, true, true, false>(sm.wk(i), sm.yb(i), pr, g, A, As, h, Dd);
            } else {
                if (dsum_on) csum = compute_chunk<T, NS, P, true, false, true>(sm.wk(i), sm.yb(i), pr, g, A, As, h, Dd);
                else compute_chunk<T, NS, P, true, false, false>(sm.wk(i), sm.yb(i), pr, g, A, As, h, Dd);
            }
        } else {
            if (scalar) csum = compute_chunk<T, NS, P, false, true, true>(sm.wk(i), sm.yb(i), pr, g, A, As, h, Dd);
            else csum = compute_chunk<T, NS, P, false, false, true>(sm.wk(i), sm.yb(i), pr, g, A, As, h, Dd);
        }
        if (dsum_on) {
            const float2 yk = make_float2(csum.x - dcomp.x, csum.y - dcomp.y);
            const float2 tk = make_float2(dsum.x + yk.x, dsum.y + yk.y);
            dcomp = make_float2((tk.x - dsum.x) - yk.x, (tk.y - dsum.y) - yk.y);
            dsum = tk;
        }
        done = i + 1;
        if (i + 1 < nchunks) {
            if constexpr (VEC) {
                cp_async_wait<STAGES - 2>();
                if (corr) convert_own_pieces<T, NS, P, true, false>(q, sm.stage(i + 1), sm.wk(i + 1), tid);
                else if (write_y) convert_own_pieces<T, NS, P, true>(q, sm.stage(i + 1), sm.wk(i + 1), tid);
                else convert_own_pieces<T, NS, P, false>(q, sm.stage(i + 1), sm.wk(i + 1), tid);
            } else {
                if (corr) load_chunk_scalar<T, NS, P, true, false>(q, sm.wk(i + 1), b, d0, t0 + TC, t_end, tid);
                else if (write_y) load_chunk_scalar<T, NS, P, true>(q, sm.wk(i + 1), b, d0, t0 + TC, t_end, tid);
                else load_chunk_scalar<T, NS, P, false>(q, sm.wk(i + 1), b, d0, t0 + TC, t_end, tid);
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    if (write_y && done > 0)
        store_chunk<T, NS, P, VEC>(p, sm.yb(done - 1), b, d0, t_begin + (long long)(done - 1) * TC, t_end, tid);
    if (corr) return;

#pragma unroll
    for (int e = 0; e < 2; ++e) {
        if (!dval[e]) continue;
        if (p.mode == MODE_LOCAL || p.mode == MODE_AGG) {
            float* sst = p.seg_state + (ch[e] * p.S + s) * p.N;
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const long long n = (long long)g * NS + k;
                if (n < p.N) sst[n] = h[e][k];
            }
            if (g == 0) p.seg_dsum[ch[e] * p.S + s] = e ? dsum.y : dsum.x;
        } else if (p.final_state != nullptr && (p.mode == MODE_SINGLE || s == p.S - 1)) {
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const long long n = (long long)g * NS + k;
                if (n < p.N) p.final_state[ch[e] * p.N + n] = h[e][k];
            }
        }
    }
}

}  // namespace sscan
