// First-order linear recurrence h_t = a_t h_{t-1} + b_t over rows, on sm_103a.
//
// The pscan(deltaA, BX) primitive of the mamba.py listing ("从矩阵求和到状态更新：
// 图解Blelloch并行扫描如何成为Mamba.py的‘加速引擎’", section 3.2).  A warp owns a
// (row, time segment) and walks it in blocks of 128 steps, 4 per lane:
//   1. each lane folds its 4 pairs (a, b) into one with the associative
//      operator (a1,b1) o (a2,b2) = (a2 a1, a2 b1 + b2) ("并行扫描与硬件感知优化
//      (mhpq.cn/news/1077344)" section 2.2);
//   2. a Hillis-Steele inclusive scan over the 32 lane aggregates with
//      __shfl_up_sync (5 rounds, log-depth; the same page's section 2.3) gives
//      each lane the operator of everything before it in the block;
//   3. applied to the carried state, each lane replays its 4 steps and stores
//      them; lane 31's result is the carry into the next block.
// Blocks are software-pipelined UNROLL deep so that enough loads are in
// flight for HBM.  Rows that are too few to fill the GPU are split into S
// segments: PS_AGG folds each segment (except the last) into one pair, and
// PS_FOLD replays every segment from the fold of the aggregates before it.
#pragma once

#include "device_utils.cuh"

namespace sscan {

enum PscanMode : int { PS_SINGLE = 0, PS_AGG = 1, PS_FOLD = 2 };

struct PscanParams {
    const float* a;
    const float* b;
    float* h;
    const float* h0;
    float* agg_a;  // [rows, S]: product of a over each segment
    float* agg_b;  // [rows, S]: state at the end of each segment started from 0
                   //            (segment 0: started from h0)
    long long rows, len, Tseg;
    int S;
    int mode;
    int seg_count;
};

constexpr int kPscanUnroll = 4;

template <bool VEC>
__device__ __forceinline__ void pscan_load4(const float* row, long long t, long long t_end,
                                            float (&a)[4], float (&b)[4], const float* brow) {
    if (VEC && t + 3 < t_end) {
        const float4 qa = __ldg(reinterpret_cast<const float4*>(row + t));
        const float4 qb = __ldg(reinterpret_cast<const float4*>(brow + t));
        a[0] = qa.x; a[1] = qa.y; a[2] = qa.z; a[3] = qa.w;
        b[0] = qb.x; b[1] = qb.y; b[2] = qb.z; b[3] = qb.w;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool ok = t + j < t_end;
            a[j] = ok ? __ldg(row + t + j) : 1.f;
            b[j] = ok ? __ldg(brow + t + j) : 0.f;
        }
    }
}

template <bool VEC>
__global__ void __launch_bounds__(128) pscan_kernel(const PscanParams p) {
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const long long unit = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    const long long row = unit / p.seg_count;
    const int s = (int)(unit % p.seg_count);
    if (row >= p.rows) return;  // whole warp
    const long long t_begin = (long long)s * p.Tseg;
    const long long t_end = min(p.len, t_begin + p.Tseg);
    const float* arow = p.a + row * p.len;
    const float* brow = p.b + row * p.len;
    float* hrow = p.h + row * p.len;

    float carry;
    if (p.mode == PS_FOLD && s > 0) {
        carry = p.agg_b[row * p.S];
        for (int sp = 1; sp < s; ++sp)
            carry = fmaf(p.agg_a[row * p.S + sp], carry, p.agg_b[row * p.S + sp]);
    } else {
        carry = (s == 0 && p.h0 != nullptr) ? p.h0[row] : 0.f;
    }
    float prod = 1.f;  // product of a over the segment (PS_AGG)
    const bool store = p.mode != PS_AGG;

    for (long long tb = t_begin; tb < t_end; tb += 128LL * kPscanUnroll) {
        float a[kPscanUnroll][4], b[kPscanUnroll][4];
#pragma unroll
        for (int u = 0; u < kPscanUnroll; ++u)
            pscan_load4<VEC>(arow, tb + 128LL * u + 4 * lane, t_end, a[u], b[u], brow);
#pragma unroll
        for (int u = 0; u < kPscanUnroll; ++u) {
            if (tb + 128LL * u >= t_end) break;  // uniform across the warp
            // 1. the lane's own 4 steps as one pair
            float A = a[u][0], Bv = b[u][0];
#pragma unroll
            for (int j = 1; j < 4; ++j) {
                Bv = fmaf(a[u][j], Bv, b[u][j]);
                A *= a[u][j];
            }
            // 2. inclusive Hillis-Steele scan over lanes
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float Ao = __shfl_up_sync(FULL, A, off);
                const float Bo = __shfl_up_sync(FULL, Bv, off);
                if (lane >= off) {
                    Bv = fmaf(A, Bo, Bv);
                    A *= Ao;
                }
            }
            // 3. state entering this lane's first step, then its 4 steps
            float Ae = __shfl_up_sync(FULL, A, 1);
            float Be = __shfl_up_sync(FULL, Bv, 1);
            if (lane == 0) { Ae = 1.f; Be = 0.f; }
            if (store) {
                float hv = fmaf(Ae, carry, Be);
                float out[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    hv = fmaf(a[u][j], hv, b[u][j]);
                    out[j] = hv;
                }
                const long long t = tb + 128LL * u + 4 * lane;
                if (VEC && t + 3 < t_end) {
                    *reinterpret_cast<float4*>(hrow + t) = make_float4(out[0], out[1], out[2], out[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (t + j < t_end) hrow[t + j] = out[j];
                }
            }
            const float A31 = __shfl_sync(FULL, A, 31);
            const float B31 = __shfl_sync(FULL, Bv, 31);
            carry = fmaf(A31, carry, B31);
            prod *= A31;
        }
    }
    if (p.mode == PS_AGG && lane == 0) {
        p.agg_a[row * p.S + s] = prod;
        p.agg_b[row * p.S + s] = carry;
    }
}

}  // namespace sscan
