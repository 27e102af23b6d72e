// Fused selective-scan forward kernel for sm_103a.
//
// What is computed (the selective_scan pseudocode of "Mamba 状态空间模型：从理论
// 到生产级推理的 CUDA 内核优化实战", section 2.3, with the initial/final state of
// its section 7.1): per batch b, channel d, state n and step t
//     h_t[n] = exp(delta_t * A[d,n]) * h_{t-1}[n] + (delta_t * u_t) * B[b,n,t]
//     y_t    = sum_n C[b,n,t] * h_t[n] + D[d] * u_t
//
// Work decomposition (diagonal A makes every (b, d, n) an independent chain,
// "为什么Mamba的“并行扫描”不是真并行" section 1):
//   * P lanes share a channel; lane g owns the NS states n = k*P + g and keeps
//     their h in registers; a lane serves CPL channels, so every B/C value it
//     reads from shared memory feeds CPL chains;
//   * a CTA of W warps covers DT channels and walks its time range in chunks
//     of TC steps.  The u/delta rows of its channels and the B/C rows of the
//     batch are staged per chunk in shared memory by cp.async in a 3-stage ring
//     (rows keep time contiguous, so every read is a 16-byte vector of 4
//     steps); bf16 tiles are widened to fp32 once per chunk by the whole CTA.
//     The B/C tile is reused by all DT channels (the fusion of discretisation,
//     scan and C-contraction of "并行扫描与硬件感知优化 (mhpq.cn/news/1077344)"
//     section 3.2, with the double buffering of the CUDA page's section 4.3
//     generalised to a ring);
//   * each lane writes its partial C-contraction of 4 steps to shared memory;
//     after the chunk the CTA sums the P partials of every output and stores
//     the outputs as vectors.  The skip term D*u enters through lane 0's
//     partial;
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
    MODE_CORR = 2     // after MODE_LOCAL: segment s >= 1 adds the decaying carry of
                      // its entry state to the outputs already written, until the
                      // carry has decayed below 2^-24 of its entry magnitude; the
                      // last segment writes final_state
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
    float* seg_dmin;   // [batch*dim, S]     min(0, smallest delta of the segment): a carry
                       //                    may grow where it is negative
    long long batch, dim, L, N;
    long long Tseg;    // steps per segment (multiple of the chunk)
    int S;             // segments per channel
    int tiles_per_batch;
    int mode;
    int seg_count;     // segments covered by this grid: grid = tiles * seg_count
    int vec;           // rows are 16-byte aligned: cp.async staging, vector stores
    const void* z;            // [batch, dim, L] output gate (out *= silu(z)), or NULL
    const float* delta_bias;  // [dim] added to delta, or NULL
    int delta_softplus;       // delta <- softplus(delta (+ bias)) inside the op
    int zoh;                  // zero-order-hold B-bar (the kernel's ZOH variant)
    int* status;              // device status word: a bounded wait that gives up
                              // stores SSCAN_ERR_TIMEOUT there
    int fold_in_corr;  // the correction folds the aggregates itself (few segments; no fold pass)
    // test aid (TMA-fed kernels): when set, each bounded wait gives up after
    // wait_ns, and the first B/C stage's barrier expects 16 bytes that no copy
    // delivers, so that its waits run out and the timeout path runs
    unsigned long long wait_ns;
    int expire_wait;
};

// softplus(x) = log(1 + e^x) from the MUFU exponent and logarithm: with
// e = e^x, log1p(e) is taken from its Maclaurin series e - e^2/2 + e^3/3 where
// e < 1/64 (truncation below 2^-26 relative), else as ln2 * log2(1 + e), whose
// absolute error (2^-22) is then below 1e-5 of the result; x > 20 gives x.
// Both branches are computed and the result selected, so that lanes with
// different arguments do not diverge.
__device__ __forceinline__ float softplus_f(float x) {
    const float e = ex2(x * 1.4426950408889634f);
    const float series = e * fmaf(e, fmaf(e, 1.f / 3.f, -0.5f), 1.f);
    float l;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l) : "f"(1.f + e));
    const float r = e < 0.015625f ? series : l * 0.69314718055994531f;
    return x > 20.f ? x : r;
}

// delta as the scan uses it: delta + bias, then softplus when asked for
__device__ __forceinline__ float delta_in(float x, float bias, bool softplus) {
    x += bias;
    return softplus ? softplus_f(x) : x;
}

// Zero-order-hold B-bar per unit B, (exp(delta*A) - 1) / A, given the exponent
// argument y = delta*A*log2(e), a = 2^y and invA = 1/A (0 when A = 0).  Where
// |delta*A| < 1/16 the difference a - 1 would cancel, so there the series
// delta*(1 + x/2 + x^2/6 + x^3/24), x = delta*A, is used (truncation below
// 2e-7 relative); A = 0 gives delta, the Euler value.
// Both forms are computed and one selected (no divergent branch in the
// element loop).
__device__ __forceinline__ float zoh_coef(float dt, float y, float a, float invA) {
    const float x = y * 0.69314718055994531f;
    const float series = dt * fmaf(x, fmaf(x, fmaf(x, 1.f / 24.f, 1.f / 6.f), 0.5f), 1.f);
    const float direct = (a - 1.f) * invA;
    return fabsf(x) < 0.0625f ? series : direct;
}

// silu(z) = z * sigmoid(z), the output gate
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + ex2(-z * 1.4426950408889634f)); }

constexpr float kLog2e = 1.4426950408889634f;
#ifndef SSCAN_CHUNK_STEPS
#define SSCAN_CHUNK_STEPS 32
#endif
constexpr int kChunkSteps = SSCAN_CHUNK_STEPS;  // steps per chunk (TC); segments are multiples of it
#ifndef SSCAN_BLOCK_UNROLL
#define SSCAN_BLOCK_UNROLL 2
#endif
// 4-step blocks unrolled per iteration of the chunk loop: a partial unroll keeps
// the loop body small enough for the instruction cache at every shape
constexpr int kBlockUnroll = SSCAN_BLOCK_UNROLL;

#ifndef SSCAN_CP_STAGES
#define SSCAN_CP_STAGES 3
#endif
constexpr int kCpStages = SSCAN_CP_STAGES;  // depth of the cp.async ring

constexpr int warps_for(int P, int CPL) {
    return (16 * P) / (32 * CPL) < 2 ? 2 : ((16 * P) / (32 * CPL) > 8 ? 8 : (16 * P) / (32 * CPL));
}

template <typename T, int NS_, int P_, int CPL_, int OPT_ = 0>
struct FwdCfg {
    static constexpr int NS = NS_;
    static constexpr int P = P_;
    static constexpr int CPL = CPL_;
    static constexpr int GPW = 32 / P;                // channel groups per warp
    static constexpr int kWarps = warps_for(P, CPL);  // at least 16 channels per CTA
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int CPW = GPW * CPL;             // channels per warp
    static constexpr int DT = kWarps * CPW;           // channels per CTA
    static constexpr int NSP = NS * P;                // state slots per channel
    static constexpr int TC = kChunkSteps;
    static constexpr bool kF32 = sizeof(T) == 4;
    static constexpr int VECE = 16 / (int)sizeof(T);  // elements per 16 bytes
    static constexpr int RROW = TC + VECE;            // raw row (T), padded by 16 bytes
    static constexpr int FROW = TC + 4;               // fp32 row, padded by 16 bytes
    static constexpr int PPR = TC / VECE;             // 16-byte pieces per row
    static constexpr int OPT = OPT_;                  // 0 plain; 1 options; 2 options + zero-order hold
    static constexpr int ROWS = (OPT > 0 ? 3 : 2) * DT + 2 * NSP;  // u, delta, B, C (, z)
    static constexpr int ZROW0 = 2 * DT + 2 * NSP;    // first z row (options only)
    static constexpr int RAW_ELEMS = ROWS * RROW;
    static constexpr int RAW_BYTES = RAW_ELEMS * (int)sizeof(T);
    static constexpr int STAGES = kCpStages;
    // fp32 rows the lanes read: the raw stage itself for fp32 I/O (RROW == FROW),
    // a widened copy for bf16
    static constexpr int WORK_FLOATS = kF32 ? 0 : ROWS * FROW;
    // partial outputs [DT][P][FROW]; the channel stride RS keeps RS/4 odd so the
    // rows a quarter-warp reads in the epilogue fall in distinct banks
    static constexpr int RS = ((P * FROW / 4) % 2 == 1) ? P * FROW : P * FROW + 4;
    static constexpr int YP_FLOATS = DT * RS;
    // epilogue items (4 steps of one channel) per thread
    static constexpr int IPT = (DT * (TC / 4) + kThreads - 1) / kThreads;
    static constexpr int SMEM_BYTES = STAGES * RAW_BYTES + (WORK_FLOATS + YP_FLOATS) * 4;
    static_assert(32 % P == 0, "lanes per channel must divide the warp");
    static_assert(TC % 4 == 0 && TC % VECE == 0, "chunk must hold whole vectors");
    static_assert(RROW * sizeof(T) % 16 == 0, "smem rows must stay 16-byte aligned");
    static_assert(!kF32 || RROW == FROW, "fp32 lanes read the raw rows");
    static_assert((DT * TC / 4) % kThreads == 0 || (DT * TC / 4) < kThreads, "epilogue items");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// State entering segment s (s >= 1) for the lane's states n = k*P + g of one
// channel, when a split has few segments and the fold pass is not launched
// (FwdParams::fold_in_corr): the fold of the aggregates of segments 0 .. s-1
// (segment 0's entry holds its true end state because it started from h0),
// the same composition in the same order as the fold pass.  FB segments'
// loads are issued before their folds so the chain waits on memory once per FB.
template <int NS, int P>
__device__ __forceinline__ void fold_segments(const FwdParams& p, long long ch, int s, int g,
                                              const float (&Al2)[NS], float (&h)[NS]) {
    constexpr int FB = NS <= 2 ? 16 : NS <= 4 ? 8 : 4;
    const float* st = p.seg_state + ch * p.S * p.N;
    const float* ds = p.seg_dsum + ch * p.S;
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        const long long n = (long long)k * P + g;
        h[k] = n < p.N ? st[n] : 0.f;
    }
    for (int sp = 1; sp < s; sp += FB) {
        float dv[FB], bv[FB][NS];
#pragma unroll
        for (int q = 0; q < FB; ++q) {
            const bool on = sp + q < s;
            dv[q] = on ? ds[sp + q] : 0.f;
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const long long n = (long long)k * P + g;
                bv[q][k] = (on && n < p.N) ? st[(long long)(sp + q) * p.N + n] : 0.f;
            }
        }
#pragma unroll
        for (int q = 0; q < FB; ++q) {
            if (sp + q < s) {
#pragma unroll
                for (int k = 0; k < NS; ++k) h[k] = fmaf(ex2(Al2[k] * dv[q]), h[k], bv[q][k]);
            }
        }
    }
}

// Shared memory: raw ring [STAGES][ROWS][RROW] (T, cp.async targets), then the
// fp32 work rows [ROWS][FROW] (bf16 only), then the partial outputs [DT][RS].
// Rows: u [0, DT), delta [DT, 2DT), B [2DT, 2DT+NSP), C [2DT+NSP, 2DT+2NSP).
template <typename T, int NS, int P, int CPL, int OPT>
struct Smem {
    using Cfg = FwdCfg<T, NS, P, CPL, OPT>;
    T* raw;
    float* work;
    float* yp;
    __device__ __forceinline__ explicit Smem(unsigned char* base)
        : raw(reinterpret_cast<T*>(base)),
          work(reinterpret_cast<float*>(base + Cfg::STAGES * Cfg::RAW_BYTES)),
          yp(reinterpret_cast<float*>(base + Cfg::STAGES * Cfg::RAW_BYTES) + Cfg::WORK_FLOATS) {}
    __device__ __forceinline__ T* stage(int i) const { return raw + (i % Cfg::STAGES) * Cfg::RAW_ELEMS; }
    // fp32 rows the lanes compute from for chunk i
    __device__ __forceinline__ float* rows(int i) const {
        if constexpr (Cfg::kF32) return reinterpret_cast<float*>(stage(i));
        else return work;
    }
};

// Vector path: issue this thread's 16-byte cp.async pieces of chunk [t0, t0+TC)
// into stage st.  Out-of-range pieces are zero-filled (delta = 0 keeps the state).
// load_d = false leaves out the delta (and z) rows.
template <typename T, int NS, int P, int CPL, int OPT>
__device__ __forceinline__ void issue_chunk(const FwdParams& p, T* st, long long b, long long d0,
                                            long long t0, long long t_end, int tid, bool load_u,
                                            bool load_b, bool load_c, bool load_d = true) {
    using Cfg = FwdCfg<T, NS, P, CPL, OPT>;
    constexpr int DT = Cfg::DT, RROW = Cfg::RROW, NSP = Cfg::NSP, PPR = Cfg::PPR, VE = Cfg::VECE;
    const T* gu = static_cast<const T*>(p.u);
    const T* gd = static_cast<const T*>(p.delta);
    const T* gB = static_cast<const T*>(p.B);
    const T* gC = static_cast<const T*>(p.C);
    const T* gz = static_cast<const T*>(p.z);
    for (int q = tid; q < DT * PPR; q += Cfg::kThreads) {
        const int r = q / PPR, pc = q % PPR;
        const long long t = t0 + (long long)pc * VE;
        const long long dd = d0 + r;
        const bool ok = dd < p.dim && t < t_end;
        const long long off = (b * p.dim + (ok ? dd : 0)) * p.L + (ok ? t : 0);
        if (load_u) cp_async16(st + r * RROW + pc * VE, gu + off, ok ? 16 : 0);
        if (!load_d) continue;
        cp_async16(st + (DT + r) * RROW + pc * VE, gd + off, ok ? 16 : 0);
        if constexpr (OPT > 0)
            if (gz != nullptr) cp_async16(st + (Cfg::ZROW0 + r) * RROW + pc * VE, gz + off, ok ? 16 : 0);
    }
    const int N = (int)p.N;
    for (int q = tid; q < N * PPR; q += Cfg::kThreads) {
        const int n = q / PPR, pc = q % PPR;
        const long long t = t0 + (long long)pc * VE;
        const bool ok = t < t_end;
        const long long off = (b * p.N + n) * p.L + (ok ? t : 0);
        if (load_b) cp_async16(st + (2 * DT + n) * RROW + pc * VE, gB + off, ok ? 16 : 0);
        if (load_c) cp_async16(st + (2 * DT + NSP + n) * RROW + pc * VE, gC + off, ok ? 16 : 0);
    }
}

// bf16 vector path: widen a landed stage to the fp32 work rows (after a barrier,
// since a thread widens pieces other threads copied), one 16-byte piece (8
// values) per item.  Rows: u and delta [0, 2DT), B [2DT, 2DT+N),
// C [2DT+NSP, 2DT+NSP+N), z [ZROW0, ZROW0+DT) when gated.
__device__ __forceinline__ void widen8(const bf16* src, float* dst) {
    const uint4 q = *reinterpret_cast<const uint4*>(src);
    *reinterpret_cast<float4*>(dst) = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u),
                                                  __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
    *reinterpret_cast<float4*>(dst + 4) = make_float4(__uint_as_float(q.z << 16), __uint_as_float(q.z & 0xffff0000u),
                                                      __uint_as_float(q.w << 16), __uint_as_float(q.w & 0xffff0000u));
}

template <typename T, int NS, int P, int CPL, int OPT>
__device__ __forceinline__ void widen_stage(const FwdParams& p, const T* st, float* wk, long long d0,
                                            long long t0, long long t_end, int tid) {
    using Cfg = FwdCfg<T, NS, P, CPL, OPT>;
    constexpr int DT = Cfg::DT, RROW = Cfg::RROW, FROW = Cfg::FROW, TC = Cfg::TC, NSP = Cfg::NSP;
    constexpr int Q8 = TC / 8;  // 16-byte pieces per row
    const int N = (int)p.N;
    // u and delta rows; with the options, delta is transformed (bias,
    // softplus) on the way, except in padding
    const bool xform = OPT > 0 && (p.delta_softplus != 0 || p.delta_bias != nullptr);
    for (int q = tid; q < 2 * DT * Q8; q += Cfg::kThreads) {
        const int r = q / Q8, c = (q % Q8) * 8;
        widen8(st + r * RROW + c, wk + r * FROW + c);
        if (xform && r >= DT) {
            const long long dd = d0 + (r - DT);
            if (dd < p.dim) {
                const float bias = p.delta_bias != nullptr ? p.delta_bias[dd] : 0.f;
                float* v = wk + r * FROW + c;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (t0 + c + e < t_end) v[e] = delta_in(v[e], bias, p.delta_softplus != 0);
            }
        }
    }
    // B and C rows of the N states
    for (int q = tid; q < 2 * N * Q8; q += Cfg::kThreads) {
        const int k = q / Q8, c = (q % Q8) * 8;
        const int r = 2 * DT + (k < N ? k : NSP + (k - N));
        widen8(st + r * RROW + c, wk + r * FROW + c);
    }
    if constexpr (OPT > 0) {
        if (p.z != nullptr)
            for (int q = tid; q < DT * Q8; q += Cfg::kThreads) {
                const int r = Cfg::ZROW0 + q / Q8, c = (q % Q8) * 8;
                widen8(st + r * RROW + c, wk + r * FROW + c);
            }
    }
}

// delta transform (bias, softplus) of a chunk's delta rows in place in an fp32
// stage (bf16 stages are transformed as they are widened);
// padding (channels beyond dim, steps beyond the segment) stays 0 so that it
// keeps the state.  Runs after the rows are visible to every thread.
template <typename T, int NS, int P, int CPL, int OPT>
__device__ __forceinline__ void transform_delta_rows(const FwdParams& p, float* rows, long long d0,
                                                     long long t0, long long t_end, int tid) {
    using Cfg = FwdCfg<T, NS, P, CPL, OPT>;
    constexpr int DT = Cfg::DT, FROW = Cfg::FROW, TC = Cfg::TC;
    for (int q = tid; q < DT * TC; q += Cfg::kThreads) {
        const int r = q / TC, tt = q % TC;
        const long long dd = d0 + r;
        if (dd < p.dim && t0 + tt < t_end) {
            const float bias = p.delta_bias != nullptr ? p.delta_bias[dd] : 0.f;
            float& v = rows[(DT + r) * FROW + tt];
            v = delta_in(v, bias, p.delta_softplus != 0);
        }
    }
}

// Scalar path (rows not 16-byte aligned): element loads with bounds checks
// straight into the fp32 rows the lanes read.
template <typename T, int NS, int P, int CPL, int OPT>
__device__ __forceinline__ void load_chunk_scalar(const FwdParams& p, float* rows, long long b,
                                                  long long d0, long long t0, long long t_end, int tid,
                                                  bool load_u, bool load_b, bool load_c) {
    using Cfg = FwdCfg<T, NS, P, CPL, OPT>;
    constexpr int DT = Cfg::DT, TC = Cfg::TC, FROW = Cfg::FROW, NSP = Cfg::NSP;
    const T* gu = static_cast<const T*>(p.u);
    const T* gd = static_cast<const T*>(p.delta);
    const T* gB = static_cast<const T*>(p.B);
    const T* gC = static_cast<const T*>(p.C);
    for (int q = tid; q < DT * TC; q += Cfg::kThreads) {
        const int r = q / TC, tt = q % TC;
        const long long dd = d0 + r, t = t0 + tt;
        const bool ok = dd < p.dim && t < t_end;
        const long long off = (b * p.dim + dd) * p.L + t;
        if (load_u) rows[r * FROW + tt] = ok ? to_f32(gu[off]) : 0.f;
        float dv = 0.f;
        if (ok) {
            dv = to_f32(gd[off]);
            if (OPT > 0 && (p.delta_softplus != 0 || p.delta_bias != nullptr))
                dv = delta_in(dv, p.delta_bias != nullptr ? p.delta_bias[dd] : 0.f, p.delta_softplus != 0);
        }
        rows[(DT + r) * FROW + tt] = dv;
        if constexpr (OPT > 0)
            if (p.z != nullptr)
                rows[(Cfg::ZROW0 + r) * FROW + tt] = ok ? to_f32(static_cast<const T*>(p.z)[off]) : 0.f;
    }
    const int N = (int)p.N;
    for (int q = tid; q < N * TC; q += Cfg::kThreads) {
        const int n = q / TC, tt = q % TC;
        const long long t = t0 + tt;
        const bool ok = t < t_end;
        const long long off = (b * p.N + n) * p.L + t;
        if (load_b) rows[(2 * DT + n) * FROW + tt] = ok ? to_f32(gB[off]) : 0.f;
        if (load_c) rows[(2 * DT + NSP + n) * FROW + tt] = ok ? to_f32(gC[off]) : 0.f;
    }
}

// One chunk of the recurrence for the calling lane: channels at tile rows
// rr[j], states n = k*P + g.  For every block of 4 steps the lane reads its
// channels' u/delta as 16-byte vectors, then walks its states in quads: the
// B/C rows of 4 states (4 steps each) are read as 16-byte vectors and the quad
// is advanced 4 steps for all CPL channels.  The 4 partial outputs of each
// channel are stored at the end of the block (the skip term D*u is added by
// the epilogue).  SCALAR: every state of a channel shares one decay rate (one
// exponent per channel and step).  NO_B: the homogeneous recurrence h = a*h of
// the carry correction (u and B are not read).
template <typename T, int NS, int P, int CPL, int OPT, bool WRITE_Y, bool SCALAR, bool NO_B, bool ZOH>
__device__ __forceinline__ void compute_chunk(const float* rows, float* yp, const int (&rr)[CPL], int g,
                                              const float (&Al2)[CPL][NS], const float (&As)[CPL],
                                              const float (&invA)[CPL][NS], const float (&invAs)[CPL],
                                              float (&h)[CPL][NS]) {
    using Cfg = FwdCfg<T, NS, P, CPL, OPT>;
    constexpr int DT = Cfg::DT, TC = Cfg::TC, FROW = Cfg::FROW, NSP = Cfg::NSP, RS = Cfg::RS;
    constexpr int QS = NS < 4 ? NS : 4;  // states per quad
    constexpr int NQ = NS / QS;
    static_assert(NS % QS == 0, "states come in whole quads");
    const float* su = rows;
    const float* sd = rows + DT * FROW;
    const float* sB = rows + (2 * DT + g) * FROW;
    const float* sC = rows + (2 * DT + NSP + g) * FROW;
#pragma unroll kBlockUnroll
    for (int t4 = 0; t4 < TC; t4 += 4) {
        float uu[CPL][4], dd[CPL][4];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            if (!NO_B) load4_smem(su + rr[j] * FROW + t4, uu[j]);
            load4_smem(sd + rr[j] * FROW + t4, dd[j]);
        }
        // terms of a (channel, step) shared by all its states.  du is the
        // input factor of B: delta*u (Euler), u (general zero-order hold, whose
        // factor is per state) or B-bar/B * u (zero-order hold, shared rate)
        float du[CPL][4], as[CPL][4], y[CPL][4];
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const float ys = dd[j][s] * As[j];
                as[j][s] = SCALAR ? ex2(ys) : 0.f;
                if (NO_B) du[j][s] = 0.f;
                else if (!ZOH) du[j][s] = dd[j][s] * uu[j][s];
                else if (SCALAR) du[j][s] = zoh_coef(dd[j][s], ys, as[j][s], invAs[j]) * uu[j][s];
                else du[j][s] = uu[j][s];
                y[j][s] = 0.f;
            }
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            float bb[QS][4], cc[QS][4];
#pragma unroll
            for (int kk = 0; kk < QS; ++kk) {
                const int k = q * QS + kk;
                if (!NO_B) load4_smem(sB + k * P * FROW + t4, bb[kk]);
                if (WRITE_Y) load4_smem(sC + k * P * FROW + t4, cc[kk]);
            }
#pragma unroll
            for (int s = 0; s < 4; ++s)
#pragma unroll
                for (int j = 0; j < CPL; ++j)
#pragma unroll
                    for (int kk = 0; kk < QS; ++kk) {
                        const int k = q * QS + kk;
                        const float yk = dd[j][s] * Al2[j][k];
                        const float a = SCALAR ? as[j][s] : ex2(yk);
                        if (NO_B) {
                            h[j][k] = a * h[j][k];
                        } else if (ZOH && !SCALAR) {
                            const float c = zoh_coef(dd[j][s], yk, a, invA[j][k]);
                            h[j][k] = fmaf(a, h[j][k], (c * du[j][s]) * bb[kk][s]);
                        } else {
                            h[j][k] = fmaf(a, h[j][k], du[j][s] * bb[kk][s]);
                        }
                        if (WRITE_Y) y[j][s] = fmaf(cc[kk][s], h[j][k], y[j][s]);
                    }
        }
        if (WRITE_Y) {
#pragma unroll
            for (int j = 0; j < CPL; ++j)
                *reinterpret_cast<float4*>(yp + rr[j] * RS + g * FROW + t4) =
                    make_float4(y[j][0], y[j][1], y[j][2], y[j][3]);
        }
    }
}

// One chunk of the carry correction for the calling lane: the homogeneous
// recurrence h = exp(delta*A) * h from the carried state, with its
// C-contraction stored as partial outputs exactly as compute_chunk stores
// them.  A state slot k whose carry has fallen below the lane's threshold in
// every lane of the warp at the start of the chunk is frozen for the chunk:
// its term is below 2^-24 of the largest carry component and only keeps
// decaying, so it is skipped (a warp-uniform branch).  SCALAR: one decay rate
// per channel (the states decay together; no per-slot check).
template <typename T, int NS, int P, int CPL, int OPT, bool SCALAR>
__device__ __forceinline__ void decay_chunk(const float* rows, float* yp, const int (&rr)[CPL], int g,
                                            const float (&Al2)[CPL][NS], const float (&As)[CPL],
                                            const float (&thr)[CPL], float (&h)[CPL][NS]) {
    using Cfg = FwdCfg<T, NS, P, CPL, OPT>;
    constexpr int DT = Cfg::DT, TC = Cfg::TC, FROW = Cfg::FROW, NSP = Cfg::NSP, RS = Cfg::RS;
    constexpr unsigned FULL = 0xffffffffu;
    const float* sd = rows + DT * FROW;
    const float* sC = rows + (2 * DT + NSP + g) * FROW;
    bool live[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        if (SCALAR) {  // one rate: the states decay together
            live[k] = true;
            continue;
        }
        bool l = false;
#pragma unroll
        for (int j = 0; j < CPL; ++j) l |= fabsf(h[j][k]) > thr[j];
        live[k] = __any_sync(FULL, l);
    }
#pragma unroll kBlockUnroll
    for (int t4 = 0; t4 < TC; t4 += 4) {
        float dd[CPL][4], as[CPL][4], y[CPL][4];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            load4_smem(sd + rr[j] * FROW + t4, dd[j]);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                as[j][s] = SCALAR ? ex2(dd[j][s] * As[j]) : 0.f;
                y[j][s] = 0.f;
            }
        }
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            if (!live[k]) continue;
            float cc[4];
            load4_smem(sC + k * P * FROW + t4, cc);
#pragma unroll
            for (int s = 0; s < 4; ++s)
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    const float a = SCALAR ? as[j][s] : ex2(dd[j][s] * Al2[j][k]);
                    h[j][k] *= a;
                    y[j][s] = fmaf(cc[s], h[j][k], y[j][s]);
                }
        }
#pragma unroll
        for (int j = 0; j < CPL; ++j)
            *reinterpret_cast<float4*>(yp + rr[j] * RS + g * FROW + t4) = make_float4(y[j][0], y[j][1], y[j][2], y[j][3]);
    }
}

// Sum the P partials of every output of the chunk, add the skip term D*u and
// store it (CORR: add it to the output already written, no skip term).  Item
// q covers 4 steps of tile row q % DT; a thread's items keep their (row,
// steps) slot from chunk to chunk, so with DSUM each thread also keeps a
// running (Kahan) sum of delta per item slot, for the segment aggregate.
template <typename T, int NS, int P, int CPL, int OPT>
__device__ __forceinline__ void store_chunk(const FwdParams& p, const float* yp, const float* rows,
                                            const float* zrows, long long b, long long d0, long long t0,
                                            long long t_end, int tid, bool corr, bool vec, bool dsum_on,
                                            float (&ds)[FwdCfg<T, NS, P, CPL, OPT>::IPT],
                                            float (&dc)[FwdCfg<T, NS, P, CPL, OPT>::IPT],
                                            float (&dm)[FwdCfg<T, NS, P, CPL, OPT>::IPT]) {
    using Cfg = FwdCfg<T, NS, P, CPL, OPT>;
    constexpr int DT = Cfg::DT, TC = Cfg::TC, FROW = Cfg::FROW, RS = Cfg::RS;
    T* go = static_cast<T*>(p.out);
#pragma unroll
    for (int k = 0; k < Cfg::IPT; ++k) {
        const int q = tid + k * Cfg::kThreads;
        if (q >= DT * (TC / 4)) break;
        const int r = q % DT, t4 = (q / DT) * 4;
        const long long dd = d0 + r, t = t0 + t4;
        if (dd >= p.dim || t >= t_end) continue;
        if (dsum_on) {  // padding steps hold delta = 0
            float dv[4];
            load4_smem(rows + (DT + r) * FROW + t4, dv);
            const float yk = ((dv[0] + dv[1]) + (dv[2] + dv[3])) - dc[k];
            const float tk = ds[k] + yk;
            dc[k] = (tk - ds[k]) - yk;
            ds[k] = tk;
            dm[k] = fminf(dm[k], fminf(fminf(dv[0], dv[1]), fminf(dv[2], dv[3])));
        }
        float v[4];
        load4_smem(yp + r * RS + t4, v);
#pragma unroll
        for (int gg = 1; gg < P; ++gg) {
            float w[4];
            load4_smem(yp + r * RS + gg * FROW + t4, w);
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] += w[e];
        }
        if (!corr && p.D != nullptr) {  // the skip term, u from the chunk's rows
            const float Dd = __ldg(p.D + dd);
            float uv[4];
            load4_smem(rows + r * FROW + t4, uv);
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = fmaf(Dd, uv[e], v[e]);
        }
        if (OPT > 0 && zrows != nullptr) {  // out = (y + D*u) * silu(z); a correction is gated alike
            float zv[4];
            load4_smem(zrows + r * FROW + t4, zv);
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] *= silu(zv[e]);
        }
        if (corr) {  // the local outputs of the chunk, staged in the u rows
            float w[4];
            load4_smem(rows + r * FROW + t4, w);
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] += w[e];
        }
        T* o = go + (b * p.dim + dd) * p.L + t;
        // vector rows: t_end is a multiple of 4, so whole groups are in range
        if (vec) {
            if constexpr (Cfg::kF32) {
                *reinterpret_cast<float4*>(o) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
                const unsigned lo = (unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[0])) |
                                    ((unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[1])) << 16);
                const unsigned hi = (unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[2])) |
                                    ((unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[3])) << 16);
                *reinterpret_cast<uint2*>(o) = make_uint2(lo, hi);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (t + e < t_end) o[e] = from_f32<T>(v[e]);
        }
    }
}

// CORR: the carry-correction instantiation (MODE_CORR launches); the single
// and local passes use the other, so that neither path's code shapes the
// other's register allocation and schedule.
template <typename T, int NS, int P, int CPL, int OPT, bool CORR>
__global__ void __launch_bounds__(FwdCfg<T, NS, P, CPL, OPT>::kThreads) sscan_fwd_chunked(const FwdParams p) {
    using Cfg = FwdCfg<T, NS, P, CPL, OPT>;
    constexpr int DT = Cfg::DT, TC = Cfg::TC, NSP = Cfg::NSP, STAGES = Cfg::STAGES;
    constexpr int RROW = Cfg::RROW, FROW = Cfg::FROW;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const Smem<T, NS, P, CPL, OPT> sm(smem_raw);

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int g = lane % P, gi = lane / P;
    const bool vec = p.vec != 0;
    constexpr bool corr = CORR;
    const bool dsum_on = p.mode == MODE_LOCAL;
    // the correction stages the local outputs in the u rows: it reads them
    // through q.u and adds the carry's contribution to them
    FwdParams q = p;
    if (corr) q.u = p.out;
    const bool load_u = true, load_b = !corr, load_c = true;
    const int tile = blockIdx.x / p.seg_count;
    const int s = (corr ? 1 : 0) + blockIdx.x % p.seg_count;
    const long long b = tile / p.tiles_per_batch;
    const long long d0 = (long long)(tile % p.tiles_per_batch) * DT;
    const long long t_begin = (long long)s * p.Tseg;
    const long long t_end = min(p.L, t_begin + p.Tseg);
    const int nchunks = t_end > t_begin ? (int)((t_end - t_begin + TC - 1) / TC) : 0;
    const int N = (int)p.N;

    // a local pass lets the correction (launched as its programmatic
    // dependent) start its CTAs early: they read the decay rates, then wait
    // for the pass's outputs and aggregates
    if constexpr (!CORR) griddep_launch_dependents();

    // the lane's channels and their decay rates (A * log2 e); a warp whose
    // channels each have a single rate takes the one-exponent-per-step path
    int rr[CPL];
    long long ch[CPL];
    bool dval[CPL];
    float Al2[CPL][NS], As[CPL], h[CPL][NS];
    float invA[CPL][NS], invAs[CPL];  // 1/A (0 where A = 0), for the zero-order hold
    bool uniform_rate = true;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        rr[j] = w * Cfg::CPW + j * Cfg::GPW + gi;
        const long long dch = d0 + rr[j];
        dval[j] = dch < p.dim;
        ch[j] = b * p.dim + (dval[j] ? dch : 0);
        const float a_first = dval[j] ? p.A[dch * p.N] : 0.f;
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const int n = k * P + g;
            const bool nv = dval[j] && n < N;
            const float a = nv ? p.A[dch * p.N + n] : a_first;
            uniform_rate &= (a == a_first);
            Al2[j][k] = nv ? a * kLog2e : 0.f;
            invA[j][k] = (nv && a != 0.f) ? 1.f / a : 0.f;
        }
        As[j] = a_first * kLog2e;
        invAs[j] = a_first != 0.f ? 1.f / a_first : 0.f;
    }
    if constexpr (CORR) {
        // the first chunks' inputs (delta, z, C) are in flight before the wait;
        // their local outputs join the same copy groups after it
        if (vec) {
#pragma unroll
            for (int j = 0; j < STAGES - 1; ++j)
                if (j < nchunks)
                    issue_chunk<T, NS, P, CPL, OPT>(q, sm.stage(j), b, d0, t_begin + (long long)j * TC, t_end, tid,
                                                    false, false, load_c);
        }
        griddep_wait();
    }
    // correction: a carried state is dropped once it has decayed below the
    // threshold only while every decay factor exp(delta*A) of the CTA's
    // channels in this segment is at most 1 (every A <= 0, no negative delta)
    bool grows = false;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        if (corr) {
            // the state entering segment s, folded from the aggregates of the
            // segments before it by the fold pass (slot s - 1; with two
            // segments slot 0 holds it already: segment 0 started from h0)
            if (p.fold_in_corr) {
                fold_segments<NS, P>(p, ch[j], s, g, Al2[j], h[j]);
            } else {
                const float* ent = p.seg_state + (ch[j] * p.S + (s - 1)) * p.N;
#pragma unroll
                for (int k = 0; k < NS; ++k) {
                    const int n = k * P + g;
                    h[j][k] = n < N ? ent[n] : 0.f;
                }
            }
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                if (!dval[j]) h[j][k] = 0.f;
                grows |= Al2[j][k] > 0.f;
            }
            if (dval[j]) grows |= p.seg_dmin[ch[j] * p.S + s] < 0.f;
        } else {
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const int n = k * P + g;
                h[j][k] = (s == 0 && p.h0 != nullptr && dval[j] && n < N) ? p.h0[ch[j] * p.N + n] : 0.f;
            }
        }
    }
    const bool scalar = __all_sync(FULL, uniform_rate);

    // correction: the last segment's final state is the carry decayed over the
    // segment plus its local end state; the carry is followed until every
    // state of the CTA has fallen below 2^-24 of its entry magnitude
    float thr[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) thr[j] = 0.f;
    const bool cut = corr && !__syncthreads_or(grows);
    if (corr) {
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            float m = 0.f;
#pragma unroll
            for (int k = 0; k < NS; ++k) m = fmaxf(m, fabsf(h[j][k]));
            thr[j] = cut ? m * 0x1p-24f : 0.f;
            // the last segment's final state: the entry state decayed over the
            // segment plus the segment's local end state
            if (dval[j] && s == p.S - 1 && p.final_state != nullptr) {
                const float dsg = p.seg_dsum[ch[j] * p.S + s];
                const float* sst = p.seg_state + (ch[j] * p.S + s) * p.N;
#pragma unroll
                for (int k = 0; k < NS; ++k) {
                    const int n = k * P + g;
                    if (n < N) p.final_state[ch[j] * p.N + n] = fmaf(ex2(Al2[j][k] * dsg), h[j][k], sst[n]);
                }
            }
        }
    }

    // B/C rows of state slots >= N are never copied: zero them once in every
    // buffer the lanes read
    if (N < NSP) {
        const int nz = NSP - N;
        for (int q = tid; q < 2 * nz * TC; q += Cfg::kThreads) {
            const int rz = q / TC, tt = q % TC;
            const int row = 2 * DT + (rz < nz ? N + rz : NSP + N + (rz - nz));
            if constexpr (Cfg::kF32) {
#pragma unroll
                for (int st = 0; st < STAGES; ++st) sm.stage(st)[row * RROW + tt] = 0.f;
            } else {
                sm.work[row * FROW + tt] = 0.f;
            }
        }
    }

    // prologue: chunks 0 .. STAGES-2 in flight (a correction issued their
    // inputs before its wait and adds the local outputs now)
    if (vec) {
#pragma unroll
        for (int j = 0; j < STAGES - 1; ++j) {
            if (j < nchunks)
                issue_chunk<T, NS, P, CPL, OPT>(q, sm.stage(j), b, d0, t_begin + (long long)j * TC, t_end, tid,
                                           load_u, corr ? false : load_b, corr ? false : load_c, !corr);
            cp_async_commit();
        }
    }

    float ds[Cfg::IPT], dc[Cfg::IPT];  // Kahan sums of delta per epilogue item slot
    float dm[Cfg::IPT];                // and min(0, smallest delta)
#pragma unroll
    for (int k = 0; k < Cfg::IPT; ++k) ds[k] = dc[k] = dm[k] = 0.f;
    for (int i = 0; i < nchunks; ++i) {
        const long long t0 = t_begin + (long long)i * TC;
        if (vec) {
            cp_async_wait<STAGES - 2>();
        } else {
            __syncthreads();  // the previous chunk's readers are done with the rows
            load_chunk_scalar<T, NS, P, CPL, OPT>(q, sm.rows(i), b, d0, t0, t_end, tid, load_u, load_b, load_c);
        }
        if (corr) {
            bool live = !cut;
#pragma unroll
            for (int j = 0; j < CPL; ++j)
#pragma unroll
                for (int k = 0; k < NS; ++k) live |= fabsf(h[j][k]) > thr[j];
            if (!__syncthreads_or(live)) break;
        } else {
            __syncthreads();
        }
        if constexpr (!Cfg::kF32) {
            if (vec) {
                widen_stage<T, NS, P, CPL, OPT>(p, sm.stage(i), sm.work, d0, t0, t_end, tid);
                __syncthreads();
            }
        }
        // (the scalar loader and the bf16 widening apply the delta transform)
        if constexpr (OPT > 0 && Cfg::kF32) {
            if (vec && (p.delta_softplus != 0 || p.delta_bias != nullptr)) {
                transform_delta_rows<T, NS, P, CPL, OPT>(p, sm.rows(i), d0, t0, t_end, tid);
                __syncthreads();
            }
        }
        if (vec) {
            const int nx = i + STAGES - 1;
            if (nx < nchunks)
                issue_chunk<T, NS, P, CPL, OPT>(q, sm.stage(nx), b, d0, t_begin + (long long)nx * TC, t_end, tid,
                                           load_u, load_b, load_c);
            cp_async_commit();
        }
        const float* rows = sm.rows(i);
        if (corr) {
            if (scalar) decay_chunk<T, NS, P, CPL, OPT, true>(rows, sm.yp, rr, g, Al2, As, thr, h);
            else decay_chunk<T, NS, P, CPL, OPT, false>(rows, sm.yp, rr, g, Al2, As, thr, h);
        } else {
            if (scalar) compute_chunk<T, NS, P, CPL, OPT, true, true, false, OPT == 2>(rows, sm.yp, rr, g, Al2, As, invA, invAs, h);
            else compute_chunk<T, NS, P, CPL, OPT, true, false, false, OPT == 2>(rows, sm.yp, rr, g, Al2, As, invA, invAs, h);
        }
        __syncthreads();  // every lane's partials of the chunk are in place
        store_chunk<T, NS, P, CPL, OPT>(p, sm.yp, rows, (OPT > 0 && p.z != nullptr) ? rows + Cfg::ZROW0 * Cfg::FROW : nullptr, b,
                                   d0, t0, t_end, tid, corr, vec, dsum_on, ds, dc, dm);
    }
    cp_async_wait<0>();
    if (corr) return;

    if (dsum_on) {  // the segment's sum of delta per channel: add up the item slots
        __syncthreads();  // the last epilogue is done with the partial buffer
        constexpr int SL = TC / 4;
#pragma unroll
        for (int k = 0; k < Cfg::IPT; ++k) {
            const int q = tid + k * Cfg::kThreads;
            if (q < DT * SL) {
                sm.yp[q] = ds[k];
                sm.yp[DT * SL + q] = dm[k];
            }
        }
        __syncthreads();
        for (int r = tid; r < DT; r += Cfg::kThreads) {
            if (d0 + r >= p.dim) continue;
            float sum = 0.f, mn = 0.f;
#pragma unroll
            for (int j = 0; j < SL; ++j) {
                sum += sm.yp[j * DT + r];
                mn = fminf(mn, sm.yp[DT * SL + j * DT + r]);
            }
            p.seg_dsum[(b * p.dim + d0 + r) * p.S + s] = sum;
            p.seg_dmin[(b * p.dim + d0 + r) * p.S + s] = mn;
        }
    }
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        if (!dval[j]) continue;
        if (p.mode == MODE_LOCAL) {
            float* sst = p.seg_state + (ch[j] * p.S + s) * p.N;
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const int n = k * P + g;
                if (n < N) sst[n] = h[j][k];
            }
        } else if (p.final_state != nullptr) {
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const int n = k * P + g;
                if (n < N) p.final_state[ch[j] * p.N + n] = h[j][k];
            }
        }
    }
}

}  // namespace sscan
