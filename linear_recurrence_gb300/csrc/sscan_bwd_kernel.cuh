// Backward pass of the selective scan for sm_103a, with chunk-boundary
// recompute: only the state at every chunk boundary is kept, and the states
// inside a chunk are recomputed from it when the reverse sweep reaches the
// chunk (the recompute strategy of "并行扫描与硬件感知优化
// (mhpq.cn/news/1077344)" section 3.3).
//
// For the loss gradients dy = dL/dy and dhT = dL/d(final state), per batch b,
// channel d, state n and step t (a_t = exp(delta_t*A[d,n])):
//   g_t      = C_t*dy_t + a_{t+1}*g_{t+1},  g_{L-1} = C*dy + dhT   (dL/dh_t)
//   ddelta_t = sum_n g_t*(h_{t-1}*a_t*A + u_t*B_t)
//   du_t     = sum_n g_t*delta_t*B_t + D*dy_t
//   dB_t    += g_t*delta_t*u_t,  dC_t += dy_t*h_t        (summed over channels)
//   dA      += g_t*h_{t-1}*a_t*delta_t,  dD += dy_t*u_t  (summed over batch, time)
//   dh0      = a_0*g_0
//
// One CTA of 4 warps owns DT channels of one batch for the whole sequence.
// P lanes share a channel, lane g owning states n = k*P + g (NS of them).
// Phase 1 runs the forward recurrence once and writes the state at every
// chunk boundary to global scratch.  Phase 2 walks the chunks backwards: it
// stages u, delta, dy, B and C of the chunk in shared memory (cp.async, two
// stages, in reverse order), recomputes the chunk's states from its boundary
// state into lane-private shared memory, then sweeps the chunk in reverse,
// carrying G = a_{t+1}*g_{t+1} in registers.  Per-step sums over a channel's
// states (du, ddelta) and over the CTA's channels (dB, dC) go through shared
// memory partials; dB and dC are accumulated into float32 outputs with one
// vector reduction per (tile, state, 4 steps), dA and dD with atomic adds once
// per lane at the end.
//
// Few channels and long sequences are split into S time segments, each its
// own CTA.  A first launch (mode 1) computes per segment the forward
// aggregate (its end state from a zero start, and sum(delta), whose decay is
// 2^(A log2e sum(delta))) and the reverse one (dL/dh at its start from a zero
// gradient at its end).  The gradient launch (mode 0) then folds the forward
// aggregates of the earlier segments into its entry state and the reverse
// aggregates of the later segments (with dL/d(final state)) into its exit
// gradient, both in order under (a1,b1) o (a2,b2) = (a2 a1, a2 b1 + b2), and
// runs the exact backward of its segment.
#pragma once

#include "device_utils.cuh"

namespace sscan {

struct BwdParams {
    const void* u;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;      // [dim] or NULL
    const float* h0;     // [batch, dim, N] or NULL
    const void* dy;      // [batch, dim, L]
    const float* dhT;    // [batch, dim, N] or NULL
    void* du;            // [batch, dim, L]  I/O dtype
    void* ddelta;        // [batch, dim, L]  I/O dtype
    float* dA;           // [dim, N]       accumulated (zeroed by the host)
    float* dB;           // [batch, N, L]  accumulated (zeroed by the host)
    float* dC;           // [batch, N, L]  accumulated (zeroed by the host)
    float* dD;           // [dim] or NULL, accumulated (zeroed by the host)
    float* dh0;          // [batch, dim, N] or NULL
    float* ckpt;         // [batch*dim, nchunks, N]: state before each chunk
    float* seg_h;        // [batch*dim, S, N] local end state of each segment (time split)
    float* seg_g;        // [batch*dim, S, N] local dL/dh entering each segment from its end
    float* seg_dsum;     // [batch*dim, S]    sum of delta over each segment
    long long batch, dim, L, N;
    long long Tseg;      // steps per segment (multiple of the chunk)
    int S;               // time segments
    int mode;            // 0: gradients of a segment; 1: its aggregates (time split)
    int tiles_per_batch;
    int vec;             // rows 16-byte aligned: cp.async staging, vector stores
};

constexpr int kBwdChunk = 16;  // steps per chunk (and checkpoint spacing)

template <typename T, int NS_, int P_>
struct BwdCfg {
    static constexpr int NS = NS_;
    static constexpr int P = P_;
    static constexpr int kWarps = 4;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int GPW = 32 / P;
    static constexpr int DT = kWarps * GPW;           // channels per CTA
    static constexpr int NSP = NS * P;                // state slots per channel
    static constexpr int TC = kBwdChunk;
    static constexpr bool kF32 = sizeof(T) == 4;
    static constexpr int VECE = 16 / (int)sizeof(T);
    static constexpr int RROW = TC + VECE;            // raw row (T), padded by 16 bytes
    static constexpr int FROW = TC + 4;               // fp32 row, padded by 16 bytes
    static constexpr int PPR = TC / VECE;             // 16-byte pieces per row
    // rows: u [0,DT), delta [DT,2DT), dy [2DT,3DT), B [3DT,3DT+NSP), C [3DT+NSP, 3DT+2NSP)
    static constexpr int ROWS = 3 * DT + 2 * NSP;
    static constexpr int RAW_ELEMS = ROWS * RROW;
    static constexpr int RAW_BYTES = RAW_ELEMS * (int)sizeof(T);
    static constexpr int STAGES = 2;
    static constexpr int WORK_FLOATS = kF32 ? 0 : ROWS * FROW;
    // recomputed states of a chunk: in registers for up to two states per
    // lane (32 registers), else lane-private shared memory
    static constexpr bool kHReg = NS <= 2;
#ifndef SSCAN_BWD_MIN_BLOCKS
#define SSCAN_BWD_MIN_BLOCKS 3
#endif
    // resident CTAs per SM asked of the compiler (register cap) where the
    // shared memory allows them
    static constexpr int kMinBlocks = kHReg ? SSCAN_BWD_MIN_BLOCKS : 1;
    static constexpr int HB_FLOATS = kHReg ? 0 : TC * NS * kThreads;
    // per-step partial sums: du, ddelta over the P lanes of a channel
    // [2][DT][P][FROW] (channel stride RS), dB, dC over the channels
    // [2][NSP][DT][FROW] (state stride RSB); RS/4 and RSB/4 odd keep the
    // epilogue's quarter-warp reads in distinct banks
    static constexpr int RS = ((P * FROW / 4) % 2 == 1) ? P * FROW : P * FROW + 4;
    static constexpr int RSB = ((DT * FROW / 4) % 2 == 1) ? DT * FROW : DT * FROW + 4;
    static constexpr int PU_FLOATS = 2 * DT * RS;
    static constexpr int PB_FLOATS = 2 * NSP * RSB;
    static constexpr int SMEM_BYTES =
        STAGES * RAW_BYTES + (WORK_FLOATS + HB_FLOATS + PU_FLOATS + PB_FLOATS) * 4;
    static_assert(RROW * sizeof(T) % 16 == 0, "smem rows must stay 16-byte aligned");
    static_assert(!kF32 || RROW == FROW, "fp32 lanes read the raw rows");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// Stage chunk [t0, t0+TC) of one CTA.  Phase 1 needs only u, delta and B.
template <typename T, int NS, int P>
__device__ __forceinline__ void bwd_issue(const BwdParams& p, T* st, long long b, long long d0,
                                          long long t0, int tid, bool full) {
    using Cfg = BwdCfg<T, NS, P>;
    constexpr int DT = Cfg::DT, RROW = Cfg::RROW, NSP = Cfg::NSP, PPR = Cfg::PPR, VE = Cfg::VECE;
    const T* gu = static_cast<const T*>(p.u);
    const T* gd = static_cast<const T*>(p.delta);
    const T* gy = static_cast<const T*>(p.dy);
    const T* gB = static_cast<const T*>(p.B);
    const T* gC = static_cast<const T*>(p.C);
    for (int q = tid; q < DT * PPR; q += Cfg::kThreads) {
        const int r = q / PPR, pc = q % PPR;
        const long long t = t0 + (long long)pc * VE;
        const long long dd = d0 + r;
        const bool ok = dd < p.dim && t < p.L;
        const long long off = (b * p.dim + (ok ? dd : 0)) * p.L + (ok ? t : 0);
        cp_async16(st + r * RROW + pc * VE, gu + off, ok ? 16 : 0);
        cp_async16(st + (DT + r) * RROW + pc * VE, gd + off, ok ? 16 : 0);
        if (full) cp_async16(st + (2 * DT + r) * RROW + pc * VE, gy + off, ok ? 16 : 0);
    }
    const int N = (int)p.N;
    for (int q = tid; q < N * PPR; q += Cfg::kThreads) {
        const int n = q / PPR, pc = q % PPR;
        const long long t = t0 + (long long)pc * VE;
        const bool ok = t < p.L;
        const long long off = (b * p.N + n) * p.L + (ok ? t : 0);
        cp_async16(st + (3 * DT + n) * RROW + pc * VE, gB + off, ok ? 16 : 0);
        if (full) cp_async16(st + (3 * DT + NSP + n) * RROW + pc * VE, gC + off, ok ? 16 : 0);
    }
}

// Element loads with bounds checks straight into fp32 rows (unaligned rows).
template <typename T, int NS, int P>
__device__ __forceinline__ void bwd_load_scalar(const BwdParams& p, float* rows, long long b, long long d0,
                                                long long t0, int tid, bool full) {
    using Cfg = BwdCfg<T, NS, P>;
    constexpr int DT = Cfg::DT, TC = Cfg::TC, FROW = Cfg::FROW, NSP = Cfg::NSP;
    const T* gu = static_cast<const T*>(p.u);
    const T* gd = static_cast<const T*>(p.delta);
    const T* gy = static_cast<const T*>(p.dy);
    const T* gB = static_cast<const T*>(p.B);
    const T* gC = static_cast<const T*>(p.C);
    for (int q = tid; q < DT * TC; q += Cfg::kThreads) {
        const int r = q / TC, tt = q % TC;
        const long long dd = d0 + r, t = t0 + tt;
        const bool ok = dd < p.dim && t < p.L;
        const long long off = (b * p.dim + dd) * p.L + t;
        rows[r * FROW + tt] = ok ? to_f32(gu[off]) : 0.f;
        rows[(DT + r) * FROW + tt] = ok ? to_f32(gd[off]) : 0.f;
        if (full) rows[(2 * DT + r) * FROW + tt] = ok ? to_f32(gy[off]) : 0.f;
    }
    const int N = (int)p.N;
    for (int q = tid; q < N * TC; q += Cfg::kThreads) {
        const int n = q / TC, tt = q % TC;
        const long long t = t0 + tt;
        const bool ok = t < p.L;
        const long long off = (b * p.N + n) * p.L + t;
        rows[(3 * DT + n) * FROW + tt] = ok ? to_f32(gB[off]) : 0.f;
        if (full) rows[(3 * DT + NSP + n) * FROW + tt] = ok ? to_f32(gC[off]) : 0.f;
    }
}

// bf16: widen a landed stage (all rows but the unused B/C slots >= N)
template <typename T, int NS, int P>
__device__ __forceinline__ void bwd_widen(const T* st, float* wk, int N, int tid) {
    using Cfg = BwdCfg<T, NS, P>;
    constexpr int DT = Cfg::DT, RROW = Cfg::RROW, FROW = Cfg::FROW, TC = Cfg::TC, NSP = Cfg::NSP;
    constexpr int Q4 = TC / 4;
    const int nr = 3 * DT + 2 * N;
    for (int q = tid; q < nr * Q4; q += Cfg::kThreads) {
        int r = q / Q4;
        const int c = (q % Q4) * 4;
        if (r >= 3 * DT + N) r += NSP - N;
        float v[4];
        load4_smem(st + r * RROW + c, v);
        *reinterpret_cast<float4*>(wk + r * FROW + c) = make_float4(v[0], v[1], v[2], v[3]);
    }
}

template <typename T, int NS, int P>
__global__ void __launch_bounds__(BwdCfg<T, NS, P>::kThreads, BwdCfg<T, NS, P>::kMinBlocks)
    sscan_bwd_chunked(const BwdParams p) {
    using Cfg = BwdCfg<T, NS, P>;
    constexpr int DT = Cfg::DT, TC = Cfg::TC, NSP = Cfg::NSP, FROW = Cfg::FROW, RROW = Cfg::RROW;
    constexpr int STAGES = Cfg::STAGES, NT = Cfg::kThreads, RS = Cfg::RS, RSB = Cfg::RSB;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* raw = reinterpret_cast<T*>(smem_raw);
    float* work = reinterpret_cast<float*>(smem_raw + STAGES * Cfg::RAW_BYTES);
    float* hb = work + Cfg::WORK_FLOATS;
    float* pu = hb + Cfg::HB_FLOATS;   // [du|ddelta][DT][RS]
    float* pb = pu + Cfg::PU_FLOATS;   // [dB|dC][NSP][RSB]
    auto stage = [&](int i) { return raw + (i % STAGES) * Cfg::RAW_ELEMS; };
    auto rows_of = [&](int i) -> float* {
        if constexpr (Cfg::kF32) return reinterpret_cast<float*>(stage(i));
        else return work;
    };

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int g = lane % P, gi = lane / P;
    const int r = w * Cfg::GPW + gi;  // the lane's channel row in the tile
    const bool vec = p.vec != 0;
    const int seg = blockIdx.x % p.S;
    const int tile = blockIdx.x / p.S;
    const long long b = tile / p.tiles_per_batch;
    const long long d0 = (long long)(tile % p.tiles_per_batch) * DT;
    const long long dch = d0 + r;
    const bool dval = dch < p.dim;
    const long long ch = b * p.dim + (dval ? dch : 0);
    const int N = (int)p.N;
    const int nchunks = (int)((p.L + TC - 1) / TC);
    const int cps = (int)(p.Tseg / TC);  // chunks per segment
    const int c_begin = seg * cps;
    const int c_end = min(nchunks, c_begin + cps);
    const bool agg = p.mode == 1;

    float A[NS], Al2[NS], h[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        const int n = k * P + g;
        const bool nv = dval && n < N;
        A[k] = nv ? p.A[dch * p.N + n] : 0.f;
        Al2[k] = A[k] * 1.4426950408889634f;
        h[k] = (nv && seg == 0 && p.h0 != nullptr) ? p.h0[ch * p.N + n] : 0.f;
    }
    const float Dd = (dval && p.D != nullptr) ? p.D[dch] : 0.f;
    // entry state of a later segment of the gradient launch: the fold of the
    // forward aggregates of segments 0 .. seg-1 (four segments' loads at a time)
    if (!agg && seg > 0 && dval) {
        const float* sh = p.seg_h + ch * p.S * p.N;
        const float* sd = p.seg_dsum + ch * p.S;
#pragma unroll
        for (int k = 0; k < NS; ++k) h[k] = (k * P + g < N) ? sh[k * P + g] : 0.f;
        for (int sp = 1; sp < seg; sp += 4) {
            float dv[4], hv[4][NS];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool on = sp + q < seg;
                dv[q] = on ? sd[sp + q] : 0.f;
#pragma unroll
                for (int k = 0; k < NS; ++k)
                    hv[q][k] = (on && k * P + g < N) ? sh[(long long)(sp + q) * p.N + k * P + g] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (sp + q < seg) {
#pragma unroll
                    for (int k = 0; k < NS; ++k) h[k] = fmaf(ex2(Al2[k] * dv[q]), h[k], hv[q][k]);
                }
        }
    }

    // B/C rows of state slots >= N are never copied: zero them once
    if (N < NSP) {
        const int nz = NSP - N;
        for (int q = tid; q < 2 * nz * TC; q += NT) {
            const int rz = q / TC, tt = q % TC;
            const int row = 3 * DT + (rz < nz ? N + rz : NSP + N + (rz - nz));
            if constexpr (Cfg::kF32) {
#pragma unroll
                for (int st = 0; st < STAGES; ++st) stage(st)[row * RROW + tt] = 0.f;
            } else {
                work[row * FROW + tt] = 0.f;
            }
        }
    }

    // ---- phase 1: forward sweep over the segment, state before every chunk ->
    // ckpt (the aggregate launch keeps only the end state and sum(delta))
    float* ck = p.ckpt + ch * (long long)nchunks * p.N;
    float dsum = 0.f, dcomp = 0.f;  // Kahan sum of delta (aggregate launch)
    if (vec) {
        if (c_begin < c_end) bwd_issue<T, NS, P>(p, stage(c_begin), b, d0, (long long)c_begin * TC, tid, false);
        cp_async_commit();
    }
    for (int c = c_begin; c < c_end; ++c) {
        if (vec) {
            if (c + 1 < c_end) bwd_issue<T, NS, P>(p, stage(c + 1), b, d0, (long long)(c + 1) * TC, tid, false);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            bwd_load_scalar<T, NS, P>(p, rows_of(c), b, d0, (long long)c * TC, tid, false);
        }
        __syncthreads();
        if constexpr (!Cfg::kF32) {
            if (vec) {
                bwd_widen<T, NS, P>(stage(c), work, N, tid);
                __syncthreads();
            }
        }
        if (dval && !agg) {
#pragma unroll
            for (int k = 0; k < NS; ++k)
                if (k * P + g < N) ck[(long long)c * p.N + k * P + g] = h[k];
        }
        const float* rows = rows_of(c);
        const float* su = rows + r * FROW;
        const float* sd = rows + (DT + r) * FROW;
        const float* sB = rows + (3 * DT + g) * FROW;
        float csum = 0.f;
#pragma unroll 2
        for (int t4 = 0; t4 < TC; t4 += 4) {
            float uu[4], dd[4];
            load4_smem(su + t4, uu);
            load4_smem(sd + t4, dd);
            csum += (dd[0] + dd[1]) + (dd[2] + dd[3]);
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                float bb[4];
                load4_smem(sB + k * P * FROW + t4, bb);
#pragma unroll
                for (int s = 0; s < 4; ++s) h[k] = fmaf(ex2(dd[s] * Al2[k]), h[k], (dd[s] * uu[s]) * bb[s]);
            }
        }
        const float yk = csum - dcomp;
        const float tk = dsum + yk;
        dcomp = (tk - dsum) - yk;
        dsum = tk;
        __syncthreads();  // the rows of chunk c are free for the next copy
    }
    cp_async_wait<0>();
    __syncthreads();
    if (agg && dval) {
#pragma unroll
        for (int k = 0; k < NS; ++k)
            if (k * P + g < N) p.seg_h[(ch * p.S + seg) * p.N + k * P + g] = h[k];
        if (g == 0) p.seg_dsum[ch * p.S + seg] = dsum;
    }

    // ---- phase 2: reverse sweep over the segment's chunks.  The exit gradient
    // G is dL/d(final state) for the last segment, else the reverse fold of
    // the later segments' aggregates; the aggregate launch starts from zero.
    float G[NS], dAacc[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        const int n = k * P + g;
        G[k] = (!agg && dval && n < N && p.dhT != nullptr) ? p.dhT[ch * p.N + n] : 0.f;
        dAacc[k] = 0.f;
    }
    if (!agg && seg < p.S - 1 && dval) {
        const float* sg = p.seg_g + ch * p.S * p.N;
        const float* sd = p.seg_dsum + ch * p.S;
        for (int sp = p.S - 1; sp > seg; sp -= 4) {
            float dv[4], gv[4][NS];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool on = sp - q > seg;
                dv[q] = on ? sd[sp - q] : 0.f;
#pragma unroll
                for (int k = 0; k < NS; ++k)
                    gv[q][k] = (on && k * P + g < N) ? sg[(long long)(sp - q) * p.N + k * P + g] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (sp - q > seg) {
#pragma unroll
                    for (int k = 0; k < NS; ++k) G[k] = fmaf(ex2(Al2[k] * dv[q]), G[k], gv[q][k]);
                }
        }
    }
    float dDacc = 0.f;
    if (vec) {
        if (c_begin < c_end) bwd_issue<T, NS, P>(p, stage(c_end - 1), b, d0, (long long)(c_end - 1) * TC, tid, true);
        cp_async_commit();
    }
    for (int c = c_end - 1; c >= c_begin; --c) {
        const long long t0 = (long long)c * TC;
        if (vec) {
            if (c > c_begin) bwd_issue<T, NS, P>(p, stage(c - 1), b, d0, t0 - TC, tid, true);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            bwd_load_scalar<T, NS, P>(p, rows_of(c), b, d0, t0, tid, true);
        }
        __syncthreads();
        if constexpr (!Cfg::kF32) {
            if (vec) {
                bwd_widen<T, NS, P>(stage(c), work, N, tid);
                __syncthreads();
            }
        }
        const float* rows = rows_of(c);
        const float* su = rows + r * FROW;
        const float* sd = rows + (DT + r) * FROW;
        const float* sy = rows + (2 * DT + r) * FROW;
        const float* sB = rows + (3 * DT + g) * FROW;
        const float* sC = rows + (3 * DT + NSP + g) * FROW;

        if (agg) {  // the reverse aggregate: dL/dh carried back from a zero gradient
#pragma unroll 1
            for (int t4 = TC - 4; t4 >= 0; t4 -= 4) {
                float dd[4], dyv[4];
                load4_smem(sd + t4, dd);
                load4_smem(sy + t4, dyv);
#pragma unroll
                for (int k = 0; k < NS; ++k) {
                    float cc[4];
                    load4_smem(sC + k * P * FROW + t4, cc);
#pragma unroll
                    for (int s = 3; s >= 0; --s) G[k] = ex2(dd[s] * Al2[k]) * fmaf(cc[s], dyv[s], G[k]);
                }
            }
            __syncthreads();  // the rows of chunk c are free for the next copy
            continue;
        }

        if constexpr (Cfg::kHReg) {
        // recompute the chunk's states from its boundary state, kept in
        // registers (hr[t][k]: h after step t of the chunk)
        float hs[NS], hr[TC][NS];
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const int n = k * P + g;
            hs[k] = (dval && n < N) ? ck[(long long)c * p.N + n] : 0.f;
            h[k] = hs[k];
        }
#pragma unroll
        for (int t4 = 0; t4 < TC; t4 += 4) {
            float uu[4], dd[4];
            load4_smem(su + t4, uu);
            load4_smem(sd + t4, dd);
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                float bb[4];
                load4_smem(sB + k * P * FROW + t4, bb);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    h[k] = fmaf(ex2(dd[s] * Al2[k]), h[k], (dd[s] * uu[s]) * bb[s]);
                    hr[t4 + s][k] = h[k];
                }
            }
        }

        // reverse sweep, 4 steps at a time.  Per step the sums over the lane's
        // states: sdd = sum g*h_prev*a*A, sgb = sum g*B (ddelta adds u*sgb,
        // du = delta*sgb + D*dy)
#pragma unroll
        for (int t4 = TC - 4; t4 >= 0; t4 -= 4) {
            float uu[4], dd[4], dyv[4], du4[4];
            load4_smem(su + t4, uu);
            load4_smem(sd + t4, dd);
            load4_smem(sy + t4, dyv);
#pragma unroll
            for (int s = 0; s < 4; ++s) du4[s] = dd[s] * uu[s];
            float sgb[4] = {0.f, 0.f, 0.f, 0.f}, sdd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                float bb[4], cc[4];
                load4_smem(sB + k * P * FROW + t4, bb);
                load4_smem(sC + k * P * FROW + t4, cc);
                float pbv[4], pcv[4];
#pragma unroll
                for (int s = 3; s >= 0; --s) {
                    const int t = t4 + s;
                    const float hprev = t > 0 ? hr[t > 0 ? t - 1 : 0][k] : hs[k];
                    const float a = ex2(dd[s] * Al2[k]);
                    const float gt = fmaf(cc[s], dyv[s], G[k]);
                    const float gha = (gt * hprev) * a;
                    dAacc[k] = fmaf(gha, dd[s], dAacc[k]);
                    sdd[s] = fmaf(gha, A[k], sdd[s]);
                    sgb[s] = fmaf(gt, bb[s], sgb[s]);
                    pbv[s] = gt * du4[s];
                    pcv[s] = dyv[s] * hr[t][k];
                    G[k] = a * gt;
                }
                const int n = k * P + g;
                *reinterpret_cast<float4*>(pb + n * RSB + r * FROW + t4) = make_float4(pbv[0], pbv[1], pbv[2], pbv[3]);
                *reinterpret_cast<float4*>(pb + NSP * RSB + n * RSB + r * FROW + t4) =
                    make_float4(pcv[0], pcv[1], pcv[2], pcv[3]);
            }
            float sdu[4];
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                sdd[s] = fmaf(uu[s], sgb[s], sdd[s]);
                sdu[s] = dd[s] * sgb[s];
            }
            if (g == 0) {
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    sdu[s] = fmaf(Dd, dyv[s], sdu[s]);
                    dDacc = fmaf(dyv[s], uu[s], dDacc);
                }
            }
            *reinterpret_cast<float4*>(pu + r * RS + g * FROW + t4) = make_float4(sdu[0], sdu[1], sdu[2], sdu[3]);
            *reinterpret_cast<float4*>(pu + DT * RS + r * RS + g * FROW + t4) =
                make_float4(sdd[0], sdd[1], sdd[2], sdd[3]);
        }
        } else {
        // recompute the chunk's states from its boundary state (lane-private,
        // 4 steps of a state per float4: hb[(t4/4 * NS + k) * NT + tid])
        float hs[NS];
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const int n = k * P + g;
            hs[k] = (dval && n < N) ? ck[(long long)c * p.N + n] : 0.f;
            h[k] = hs[k];
        }
#pragma unroll 2
        for (int t4 = 0; t4 < TC; t4 += 4) {
            float uu[4], dd[4];
            load4_smem(su + t4, uu);
            load4_smem(sd + t4, dd);
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                float bb[4], hv[4];
                load4_smem(sB + k * P * FROW + t4, bb);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    h[k] = fmaf(ex2(dd[s] * Al2[k]), h[k], (dd[s] * uu[s]) * bb[s]);
                    hv[s] = h[k];
                }
                *reinterpret_cast<float4*>(hb + ((t4 / 4) * NS + k) * NT * 4 + tid * 4) =
                    make_float4(hv[0], hv[1], hv[2], hv[3]);
            }
        }

        // reverse sweep, 4 steps at a time.  Per step the sums over the lane's
        // states: sdd = sum g*h_prev*a*A, sgb = sum g*B (ddelta adds u*sgb,
        // du = delta*sgb + D*dy)
#pragma unroll 1
        for (int t4 = TC - 4; t4 >= 0; t4 -= 4) {
            float uu[4], dd[4], dyv[4], du4[4];
            load4_smem(su + t4, uu);
            load4_smem(sd + t4, dd);
            load4_smem(sy + t4, dyv);
#pragma unroll
            for (int s = 0; s < 4; ++s) du4[s] = dd[s] * uu[s];
            float sgb[4] = {0.f, 0.f, 0.f, 0.f}, sdd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                float bb[4], cc[4], hv[4];
                const int o = ((t4 / 4) * NS + k) * NT * 4 + tid * 4;
                load4_smem(sB + k * P * FROW + t4, bb);
                load4_smem(sC + k * P * FROW + t4, cc);
                load4_smem(hb + o, hv);
                float hp;  // h at the step before t4
                if (t4 > 0) hp = hb[o - NS * NT * 4 + 3];
                else hp = hs[k];
                float pbv[4], pcv[4];
#pragma unroll
                for (int s = 3; s >= 0; --s) {
                    const float hprev = s > 0 ? hv[s - 1] : hp;
                    const float a = ex2(dd[s] * Al2[k]);
                    const float gt = fmaf(cc[s], dyv[s], G[k]);
                    const float gha = (gt * hprev) * a;
                    dAacc[k] = fmaf(gha, dd[s], dAacc[k]);
                    sdd[s] = fmaf(gha, A[k], sdd[s]);
                    sgb[s] = fmaf(gt, bb[s], sgb[s]);
                    pbv[s] = gt * du4[s];
                    pcv[s] = dyv[s] * hv[s];
                    G[k] = a * gt;
                }
                const int n = k * P + g;
                *reinterpret_cast<float4*>(pb + n * RSB + r * FROW + t4) = make_float4(pbv[0], pbv[1], pbv[2], pbv[3]);
                *reinterpret_cast<float4*>(pb + NSP * RSB + n * RSB + r * FROW + t4) =
                    make_float4(pcv[0], pcv[1], pcv[2], pcv[3]);
            }
            float sdu[4];
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                sdd[s] = fmaf(uu[s], sgb[s], sdd[s]);
                sdu[s] = dd[s] * sgb[s];
            }
            if (g == 0) {
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    sdu[s] = fmaf(Dd, dyv[s], sdu[s]);
                    dDacc = fmaf(dyv[s], uu[s], dDacc);
                }
            }
            *reinterpret_cast<float4*>(pu + r * RS + g * FROW + t4) = make_float4(sdu[0], sdu[1], sdu[2], sdu[3]);
            *reinterpret_cast<float4*>(pu + DT * RS + r * RS + g * FROW + t4) =
                make_float4(sdd[0], sdd[1], sdd[2], sdd[3]);
        }
        }
        __syncthreads();  // every partial of the chunk is in place

        // epilogue: du, ddelta (sum over the P lanes of a channel)
        T* gdu = static_cast<T*>(p.du);
        T* gdd = static_cast<T*>(p.ddelta);
        for (int q = tid; q < 2 * DT * (TC / 4); q += NT) {
            const int which = q / (DT * (TC / 4));
            const int qq = q % (DT * (TC / 4));
            const int rr = qq % DT, t4 = (qq / DT) * 4;
            const long long dd = d0 + rr, t = t0 + t4;
            if (dd >= p.dim || t >= p.L) continue;
            const float* src = pu + which * DT * RS + rr * RS;
            float v[4];
            load4_smem(src + t4, v);
#pragma unroll
            for (int gg = 1; gg < P; ++gg) {
                float x[4];
                load4_smem(src + gg * FROW + t4, x);
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] += x[e];
            }
            T* o = (which ? gdd : gdu) + (b * p.dim + dd) * p.L + t;
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
                    if (t + e < p.L) o[e] = from_f32<T>(v[e]);
            }
        }
        // epilogue: dB, dC (sum over the CTA's channels, then one atomic add)
        for (int q = tid; q < 2 * NSP * (TC / 4); q += NT) {
            const int which = q / (NSP * (TC / 4));
            const int qq = q % (NSP * (TC / 4));
            const int n = qq % NSP, t4 = (qq / NSP) * 4;
            const long long t = t0 + t4;
            if (n >= N || t >= p.L) continue;
            const float* src = pb + which * NSP * RSB + n * RSB;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            for (int rr = 0; rr < DT; ++rr) {
                if (d0 + rr >= p.dim) break;
                float x[4];
                load4_smem(src + rr * FROW + t4, x);
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] += x[e];
            }
            float* o = (which ? p.dC : p.dB) + (b * p.N + n) * p.L + t;
            if (t + 4 <= p.L && (reinterpret_cast<uintptr_t>(o) & 15u) == 0) {
                red_add_v4(o, v[0], v[1], v[2], v[3]);  // one L2 reduction for the 4 steps
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (t + e < p.L) atomicAdd(o + e, v[e]);
            }
        }
        // the next chunk's copy, partials and recompute start after this barrier
        __syncthreads();
    }
    cp_async_wait<0>();

    if (agg) {
        if (dval) {
#pragma unroll
            for (int k = 0; k < NS; ++k)
                if (k * P + g < N) p.seg_g[(ch * p.S + seg) * p.N + k * P + g] = G[k];
        }
        return;
    }
    if (dval) {
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const int n = k * P + g;
            if (n < N) {
                atomicAdd(p.dA + dch * p.N + n, dAacc[k]);
                if (p.dh0 != nullptr && seg == 0) p.dh0[ch * p.N + n] = G[k];
            }
        }
        if (g == 0 && p.dD != nullptr) atomicAdd(p.dD + dch, dDacc);
    }
}

}  // namespace sscan
