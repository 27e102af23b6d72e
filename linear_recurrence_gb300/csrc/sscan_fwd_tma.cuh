// Selective-scan forward kernel fed by the Tensor Memory Accelerator, for
// rows that satisfy the tensor-map rules (16-byte aligned rows, sizes below
// 2^31).  It computes exactly what sscan_fwd_chunked computes (the recurrence
// of "Mamba 状态空间模型：从理论到生产级推理的 CUDA 内核优化实战" section 2.3
// with the initial/final state of its section 7.1), fp32 and bf16, the plain
// scan and the options (delta bias and softplus, the output gate, the
// zero-order hold), in the single-segment and local-segment modes and, as its
// CORR instantiation, the carry correction of a time split.
//
// What changes against the cp.async kernel is who waits for whom:
//   * every warp owns its channels end to end.  Its u/delta rows arrive by
//     one TMA box per row set and chunk, issued by its lane 0 into a
//     two-stage ring that only this warp reads, completing on the warp's own
//     mbarrier; the warp sums the P partial outputs of its channels itself
//     (the lanes of a channel sit in one warp), so the chunk epilogue needs
//     __syncwarp only;
//   * the B/C rows of the chunk are shared by the CTA's four warps: one box
//     each, completing on a CTA-wide mbarrier per stage.  A warp done with a
//     stage (its lanes have consumed every value they read, then __syncwarp)
//     counts itself out on a shared-memory counter, and the last of the four
//     refills the stage, so no warp waits for another except for data that
//     has not landed.  A refill only overwrites values already read, so the
//     count needs no fence; the data itself is published by the mbarrier's
//     transaction count and acquired by its wait;
//   * bf16: each warp widens its own u/delta rows into fp32 rows, which
//     frees its raw stage at once (with 16 states per lane and the plain
//     scan the lanes read the raw rows instead, converting as they read); the
//     chunk's B/C rows are widened once per CTA, by warps in turn (chunk c by
//     warp c mod 4, one chunk ahead), into an fp32 ring of WB slots with a
//     full mbarrier (the widening warp's lanes arrive) and an empty one (every
//     warp arrives when it is done with the slot); only the widening warp
//     reads the raw B/C stage, so it refills that stage itself;
//   * the shuffle kernels (SH): the lanes of a channel sum its partial outputs
//     by warp shuffles and store them (no partial-output buffer, no epilogue);
//     their fp32 carry correction, one channel per lane, stages the C rows per
//     warp with the warp's local outputs and delta, so its warps run on their
//     own (no CTA-shared ring, no CTA-wide votes).
// fp32 boxes (and the raw bf16 u/delta boxes read in place) are TC + 16 bytes
// wide: the extra columns (the next chunk's first steps, or zeros past the
// end) pad every shared-memory row exactly as the cp.async ring does, so the
// reads of different rows at one step fall in different banks; the other bf16
// boxes are TC wide (their rows are only widened).  Every mbarrier wait is
// bounded (about a second); a wait that gives up records SSCAN_ERR_TIMEOUT in
// the status word, waits (again bounded) for the copies still in flight, and
// ends the warp's work.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "../../include/sscan.h"
#include "sscan_dispatch.cuh"
#include "sscan_fwd_kernel.cuh"

namespace sscan {

// Tensor maps of one launch, 3-D with the innermost dimension first:
// u, delta (and z) {L, dim, batch} with box {RROW, CPW, 1}; B and C
// {L, N, batch} with box {RROW, NSP, 1}.  The box height past dim (or N)
// reads zeros.
struct TmaMaps {
    CUtensorMap u;
    CUtensorMap delta;
    CUtensorMap B;
    CUtensorMap C;
    CUtensorMap z;  // the output gate (options variant with a gate only)
};

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Register ceiling of the 16-state-lane kernel without the zero-order hold
// (two CTAs per SM fit in any case; left unbounded, the allocation drifted with
// unrelated code changes from 167 to 215 registers and wide64 from 452 to 469
// us; 176 is the lowest that spills nothing).
#ifndef SSCAN_WIDE_MAXNREG
#define SSCAN_WIDE_MAXNREG 176
#endif

// Steps per chunk of the shuffle kernels, and the most resident CTAs per SM
// their register allocation is asked for (8 states per lane).
#ifndef SSCAN_SHFL_CHUNK
#define SSCAN_SHFL_CHUNK 32
#endif
#ifndef SSCAN_SHFL_MAX_BLOCKS
#define SSCAN_SHFL_MAX_BLOCKS 4
#endif

// Depth of the u/delta and B/C rings.  Two stages measured faster than three
// on GB300: the smaller footprint fits one more CTA per SM, and a chunk of
// compute (over a microsecond per warp) covers the TMA latency.
#ifndef SSCAN_TMA_STAGES
#define SSCAN_TMA_STAGES 2
#endif
constexpr int kTmaStages = SSCAN_TMA_STAGES;

template <typename T, int NS, int P, int CPL, int OPT_ = 0, bool SH_ = false>
struct TmaCfg {
    using Base = FwdCfg<T, NS, P, CPL, 0>;
    static constexpr int OPT = OPT_;  // 0 plain; 1 options; 2 options + zero-order hold
    // SH: the lanes sum a channel's P partial outputs by warp shuffles and
    // store the outputs themselves (no partial-output buffer, no epilogue)
    static constexpr bool SH = SH_;
    // the shuffle kernels' fp32 carry correction (one channel per lane) stages
    // the C rows per warp, with the warp's local outputs and delta: every warp
    // runs on its own, without a CTA-shared ring or CTA-wide votes
    static constexpr bool kWarpC = SH_ && CPL == 1 && std::is_same<T, float>::value;
    // row sets of a warp's slot: u (or the local outputs), delta (, z, or C)
    static constexpr int NUR = OPT > 0 || kWarpC ? 3 : 2;
    static constexpr int kWarps = 4;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int GPW = Base::GPW, CPW = Base::CPW, NSP = Base::NSP;
    // steps per chunk: the shuffle kernels may take shorter chunks (a smaller
    // ring, more resident CTAs)
    static constexpr int TC = SH ? SSCAN_SHFL_CHUNK : Base::TC;
    static constexpr int VECE = 16 / (int)sizeof(T);  // elements per 16 bytes
    static constexpr int DT = kWarps * CPW;  // channels per CTA
    // raw row: fp32 rows are read in place, so they keep the TC + 16 bytes
    // of the bank-spreading pad; bf16 rows are only widened (whole 16-byte
    // pieces of consecutive rows) and take no pad, which keeps the wide-state
    // CTA within half an SM's shared memory
    static constexpr int RROW = Base::kF32 ? TC + VECE : TC;
    // bf16 with 64 state slots (plain scan): the lanes read their u/delta
    // rows straight from the raw stage (converting 4 values per read), which
    // saves the per-warp fp32 copy and buys a third widened B/C slot; those
    // raw rows keep the 16-byte pad, so that the 8 channel rows a warp reads
    // at one step fall in distinct banks
    static constexpr bool kRawU = !Base::kF32 && NS > 4 && OPT_ == 0;
    static constexpr int RROW_U = kRawU ? TC + VECE : RROW;  // raw u/delta (z) row
    static constexpr int FROW = TC + 4;  // fp32 row
    static constexpr bool kF32 = Base::kF32;
    static constexpr int STAGES = kTmaStages;
    static constexpr int ESZ = (int)sizeof(T);
    static constexpr int U_BOX = CPW * RROW_U * ESZ;  // bytes of one u (delta, z) box
    static constexpr int BC_BOX = NSP * RROW * ESZ;  // bytes of one B (or C) box
    static constexpr int U_SLOT = align_up(U_BOX, 128);
    static constexpr int BC_SLOT = align_up(BC_BOX, 128);
    // the epilogue runs per half chunk: partial outputs of a warp [CPW][RS]
    // over TS steps, row (channel) stride RS = P*HROW rounded up so that
    // RS/4 = 4 (mod 8): the partial vectors a quarter-warp stores (P lanes of
    // a channel, 8/P channels) and the ones it reads back (two channel rows)
    // fall in distinct bank groups
    static constexpr int TS = TC / 2;
    static constexpr int HROW = TS + 4;
    static constexpr int RS = align_up(P * HROW - 16, 32) + 16;
    // bf16: a warp's widened fp32 rows [u CPW][delta CPW] (, [z CPW]); the
    // chunk's B/C rows are widened once per CTA into a ring of WB slots
    // [B NSP][C NSP]
    static constexpr int WORK_ROWS = NUR * CPW;
    static constexpr int WB = NS > 4 && !kRawU ? 2 : 3;  // two slots where shared memory is short
    static constexpr int BCW_BYTES = kF32 ? 0 : 2 * NSP * FROW * 4;
    // items of the warp epilogue per half chunk: (channel row, 4 steps); per lane
    static constexpr int IPH = CPW * (TS / 4) / 32;
    // resident CTAs per SM the register allocation is asked to allow: for the
    // narrow shapes the number their shared memory allows (without it the
    // compiler kept to 96 registers; measured on GB300: dim512 47.0 -> 46.1
    // us, bf16_2k 131.6 -> 129.8, long64k 506.5 -> 501.2); wide lanes take
    // no such request (sscan_fwd_tma_wide)
    static constexpr int MIN_BLOCKS = NS > 4 ? 1 : P == 4 ? 3 : 4;
    // shared-memory map (bytes from a 128-byte aligned base)
    // mbarriers [kWarps + 1][STAGES], counters [STAGES], then (bf16) the
    // widened ring's full [WB] and empty [WB] mbarriers
    static constexpr int OFF_BAR = 0;
    static constexpr int OFF_U = 1024;  // [STAGES][kWarps][u, delta (, z)] slots
    static constexpr int OFF_BC = OFF_U + STAGES * kWarps * NUR * U_SLOT;  // [STAGES][B, C] slots
    static constexpr int OFF_BCW = OFF_BC + (kWarpC ? 0 : STAGES * 2 * BC_SLOT);
    static constexpr int OFF_WORK = OFF_BCW + WB * BCW_BYTES;
    static constexpr int WORK_BYTES = kF32 || kRawU ? 0 : WORK_ROWS * FROW * 4;  // per warp
    static constexpr int OFF_YP = OFF_WORK + kWarps * WORK_BYTES;
    static constexpr int YP_BYTES = SH ? 0 : CPW * RS * 4;  // per warp
    static constexpr int SMEM_BYTES = OFF_YP + kWarps * YP_BYTES + 128;  // + base alignment
    // shuffle kernels: the register allocation is asked for the resident CTAs
    // that shared memory allows (228 KB per SM, 1 KB reserved per CTA), at most
    // 4, and at most 2 for 16 states per lane, whose registers would spill at 3
    static constexpr int SH_FIT = (228 * 1024) / (SMEM_BYTES + 1024);
    static constexpr int SH_CAP = NS >= 16 ? 2 : SSCAN_SHFL_MAX_BLOCKS;
    static constexpr int SH_MIN_BLOCKS = SH_FIT < 1 ? 1 : SH_FIT > SH_CAP ? SH_CAP : SH_FIT;
    static_assert(SH || TC == 32, "epilogue items assume 8 four-step blocks per chunk");
    static_assert(CPW % 8 == 0, "a warp's epilogue items must fill its lanes");
    static_assert(RS >= P * HROW && (RS / 4) % 8 == 4, "partial row stride");
    // after the mbarriers: the B/C release counters [STAGES] and, per stage,
    // the last chunk whose B/C copy was issued into it
    static constexpr int OFF_BCW_BAR = align_up((kWarps + 1) * STAGES * 8 + 2 * STAGES * 4, 8);
    static_assert(OFF_BCW_BAR + 2 * WB * 8 <= 1024, "barrier area");
    static_assert(RROW * ESZ % 16 == 0 && RROW_U * ESZ % 16 == 0 && FROW % 4 == 0, "16-byte rows");
    static_assert(CPW <= 256 && NSP <= 256 && RROW <= 256 && RROW_U <= 256, "tensor-map box limits");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(!kWarpC || BC_BOX <= U_SLOT, "a warp's C box fits a row-set slot");
};

// Steps [T0, T0 + TS) of a chunk of the recurrence for the calling lane, from
// fp32 rows in shared memory with row stride FROW: u rows su[r], delta rows
// sd[r] of the warp's channel rows r = rl[j]; B/C rows of state slot n at
// sB[n], sC[n].  Per 4-step block: the lane's u/delta vectors and the B/C
// vectors of its NS states (read one block ahead, so that the shared-memory
// latency overlaps the previous block's arithmetic), then per element
// x = delta*A', a = 2^x, h = a*h + (delta*u)*B, y += C*h; the 4 partial
// outputs of each channel go to yp[rl[j]][g] (row stride RS, lane stride
// HROW) as one vector.  SCALAR: one decay rate per channel.  ZOH: the
// zero-order-hold B-bar ((exp(delta A) - 1)/A per unit B) replaces delta*B.
template <typename TU, int UROW, int NS, int P, int CPL, int FROW, int RS, int HROW, int TS, bool SCALAR, bool ZOH>
__device__ __forceinline__ void compute_half_narrow(const TU* su, const TU* sd, const float* sB,
                                                 const float* sC, float* yp, const int (&rl)[CPL], int g,
                                                 int T0, const float (&Al2)[CPL][NS], const float (&As)[CPL],
                                                 const float (&invA)[CPL][NS], const float (&invAs)[CPL],
                                                 float (&h)[CPL][NS]) {
    constexpr int NB = TS / 4;
    const float* bB = sB + g * FROW;
    const float* bC = sC + g * FROW;
    float nu[CPL][4], nd[CPL][4], nb[NS][4], nc[NS][4];
    auto load_block = [&](int t4) {
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            load4_smem(su + rl[j] * UROW + t4, nu[j]);
            load4_smem(sd + rl[j] * UROW + t4, nd[j]);
        }
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            load4_smem(bB + k * P * FROW + t4, nb[k]);
            load4_smem(bC + k * P * FROW + t4, nc[k]);
        }
    };
    load_block(T0);
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
        const int t4 = T0 + 4 * blk;
        float dd[CPL][4], du[CPL][4], as[CPL][4], y[CPL][4], bb[NS][4], cc[NS][4];
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                dd[j][s] = nd[j][s];
                du[j][s] = ZOH ? nu[j][s] : nd[j][s] * nu[j][s];
            }
#pragma unroll
        for (int k = 0; k < NS; ++k)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                bb[k][s] = nb[k][s];
                cc[k][s] = nc[k][s];
            }
        if (blk + 1 < NB) load_block(t4 + 4);
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const float ys = dd[j][s] * As[j];
                as[j][s] = SCALAR ? ex2(ys) : 0.f;
                // zero-order hold with one rate: B-bar/B per (channel, step)
                if (ZOH && SCALAR) du[j][s] *= zoh_coef(dd[j][s], ys, as[j][s], invAs[j]);
                y[j][s] = 0.f;
            }
#pragma unroll
        for (int s = 0; s < 4; ++s)
#pragma unroll
            for (int j = 0; j < CPL; ++j)
#pragma unroll
                for (int k = 0; k < NS; ++k) {
                    const float yk = dd[j][s] * Al2[j][k];
                    const float a = SCALAR ? as[j][s] : ex2(yk);
                    if (ZOH && !SCALAR)
                        h[j][k] = fmaf(a, h[j][k], (zoh_coef(dd[j][s], yk, a, invA[j][k]) * du[j][s]) * bb[k][s]);
                    else
                        h[j][k] = fmaf(a, h[j][k], du[j][s] * bb[k][s]);
                    y[j][s] = fmaf(cc[k][s], h[j][k], y[j][s]);
                }
#pragma unroll
        for (int j = 0; j < CPL; ++j)
            *reinterpret_cast<float4*>(yp + rl[j] * RS + g * HROW + (t4 - T0)) =
                make_float4(y[j][0], y[j][1], y[j][2], y[j][3]);
    }
}

// As compute_half_narrow for wide lanes (NS > 4 states): the u/delta vectors
// are read one block ahead; the B/C vectors are read per quad of states inside
// the block (all of them at once would need 8*NS registers).
template <typename TU, int UROW, int NS, int P, int CPL, int FROW, int RS, int HROW, int TS, bool SCALAR, bool ZOH>
__device__ __forceinline__ void compute_half_wide(const TU* su, const TU* sd, const float* sB,
                                                  const float* sC, float* yp, const int (&rl)[CPL], int g,
                                                  int T0, const float (&Al2)[CPL][NS], const float (&As)[CPL],
                                                  const float (&invA)[CPL][NS], const float (&invAs)[CPL],
                                                  float (&h)[CPL][NS]) {
    constexpr int NB = TS / 4;
    constexpr int QS = 4, NQ = NS / QS;
    static_assert(NS % QS == 0, "states come in whole quads");
    const float* bB = sB + g * FROW;
    const float* bC = sC + g * FROW;
    float nu[CPL][4], nd[CPL][4];
    auto load_block = [&](int t4) {
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            load4_smem(su + rl[j] * UROW + t4, nu[j]);
            load4_smem(sd + rl[j] * UROW + t4, nd[j]);
        }
    };
    load_block(T0);
#pragma unroll 2
    for (int blk = 0; blk < NB; ++blk) {
        const int t4 = T0 + 4 * blk;
        float dd[CPL][4], du[CPL][4], as[CPL][4], y[CPL][4];
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                dd[j][s] = nd[j][s];
                du[j][s] = ZOH ? nu[j][s] : nd[j][s] * nu[j][s];
            }
        if (blk + 1 < NB) load_block(t4 + 4);
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const float ys = dd[j][s] * As[j];
                as[j][s] = SCALAR ? ex2(ys) : 0.f;
                if (ZOH && SCALAR) du[j][s] *= zoh_coef(dd[j][s], ys, as[j][s], invAs[j]);
                y[j][s] = 0.f;
            }
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            float bb[QS][4], cc[QS][4];
#pragma unroll
            for (int kk = 0; kk < QS; ++kk) {
                load4_smem(bB + (q * QS + kk) * P * FROW + t4, bb[kk]);
                load4_smem(bC + (q * QS + kk) * P * FROW + t4, cc[kk]);
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
                        if (ZOH && !SCALAR)
                            h[j][k] = fmaf(a, h[j][k], (zoh_coef(dd[j][s], yk, a, invA[j][k]) * du[j][s]) * bb[kk][s]);
                        else
                            h[j][k] = fmaf(a, h[j][k], du[j][s] * bb[kk][s]);
                        y[j][s] = fmaf(cc[kk][s], h[j][k], y[j][s]);
                    }
        }
#pragma unroll
        for (int j = 0; j < CPL; ++j)
            *reinterpret_cast<float4*>(yp + rl[j] * RS + g * HROW + (t4 - T0)) =
                make_float4(y[j][0], y[j][1], y[j][2], y[j][3]);
    }
}

template <typename TU, int UROW, int NS, int P, int CPL, int FROW, int RS, int HROW, int TS, bool SCALAR, bool ZOH>
__device__ __forceinline__ void compute_half_tma(const TU* su, const TU* sd, const float* sB,
                                                 const float* sC, float* yp, const int (&rl)[CPL], int g,
                                                 int T0, const float (&Al2)[CPL][NS], const float (&As)[CPL],
                                                 const float (&invA)[CPL][NS], const float (&invAs)[CPL],
                                                 float (&h)[CPL][NS]) {
    if constexpr (NS <= 4)
        compute_half_narrow<TU, UROW, NS, P, CPL, FROW, RS, HROW, TS, SCALAR, ZOH>(su, sd, sB, sC, yp, rl, g, T0, Al2, As,
                                                                         invA, invAs, h);
    else
        compute_half_wide<TU, UROW, NS, P, CPL, FROW, RS, HROW, TS, SCALAR, ZOH>(su, sd, sB, sC, yp, rl, g, T0, Al2, As,
                                                                       invA, invAs, h);
}

// SH kernels: one chunk of the recurrence for the calling lane, with its
// outputs finished in registers instead of a shared partial-output buffer.
// Per 4-step block: the lane's u/delta vectors (read one block ahead), the
// B/C vectors of its states per quad, then per element x = delta*A',
// a = 2^x, h = a*h + (delta*u)*B, y += C*h.  The lanes of a channel pair
// hold the pair in opposite register order (rl), so one exchange between
// lanes P/2 apart gives each lane the other's partial sums of the channel it
// keeps (y[0] += partner's y[1]); the remaining P/2 lanes of the channel then
// exchange all four sums (butterfly), after which every lane holds the full
// sums of its kept channel rl[0], and the lanes with (g & (P/2 - 1)) == 0
// store them with D*u added.  A local pass also takes the Kahan sum of the
// kept channel's delta (steps past L hold delta = 0).
template <typename T, typename TU, int UROW, int NS, int P, int FROW, int TC, bool SCALAR>
__device__ __forceinline__ void compute_chunk_shfl(const TU* su, const TU* sd, const float* sB, const float* sC,
                                                   const int (&rl)[2], int g, const float (&Al2)[2][NS],
                                                   const float (&As)[2], float (&h)[2][NS], float Dk, T* orow,
                                                   bool store, int nvalid, bool dsum_on, float& dsum,
                                                   float& dcomp, float& dmin) {
    constexpr int CPL = 2;
    constexpr int NB = TC / 4, QS = 4, NQ = NS / QS;
    constexpr unsigned FULL = 0xffffffffu;
    static_assert(P >= 2 && 32 % P == 0 && NS % QS == 0, "lane pairs and whole quads of states");
    const float* bB = sB + g * FROW;
    const float* bC = sC + g * FROW;
    float nu[CPL][4], nd[CPL][4];
    auto load_block = [&](int t4) {
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            load4_smem(su + rl[j] * UROW + t4, nu[j]);
            load4_smem(sd + rl[j] * UROW + t4, nd[j]);
        }
    };
    load_block(0);
#pragma unroll 2
    for (int blk = 0; blk < NB; ++blk) {
        const int t4 = 4 * blk;
        float dd[CPL][4], du[CPL][4], uk[4], as[CPL][4], y[CPL][4];
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                dd[j][s] = nd[j][s];
                du[j][s] = nd[j][s] * nu[j][s];
            }
#pragma unroll
        for (int s = 0; s < 4; ++s) uk[s] = nu[0][s];
        if (blk + 1 < NB) load_block(t4 + 4);
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                as[j][s] = SCALAR ? ex2(dd[j][s] * As[j]) : 0.f;
                y[j][s] = 0.f;
            }
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            float bb[QS][4], cc[QS][4];
#pragma unroll
            for (int kk = 0; kk < QS; ++kk) {
                load4_smem(bB + (q * QS + kk) * P * FROW + t4, bb[kk]);
                load4_smem(bC + (q * QS + kk) * P * FROW + t4, cc[kk]);
            }
#pragma unroll
            for (int s = 0; s < 4; ++s)
#pragma unroll
                for (int j = 0; j < CPL; ++j)
#pragma unroll
                    for (int kk = 0; kk < QS; ++kk) {
                        const int k = q * QS + kk;
                        const float a = SCALAR ? as[j][s] : ex2(dd[j][s] * Al2[j][k]);
                        h[j][k] = fmaf(a, h[j][k], du[j][s] * bb[kk][s]);
                        y[j][s] = fmaf(cc[kk][s], h[j][k], y[j][s]);
                    }
        }
        // the channel's P partial sums
#pragma unroll
        for (int s = 0; s < 4; ++s) y[0][s] += __shfl_xor_sync(FULL, y[1][s], P / 2);
#pragma unroll
        for (int m = P / 4; m >= 1; m /= 2)
#pragma unroll
            for (int s = 0; s < 4; ++s) y[0][s] += __shfl_xor_sync(FULL, y[0][s], m);
        if (dsum_on) {
            const float yk = ((dd[0][0] + dd[0][1]) + (dd[0][2] + dd[0][3])) - dcomp;
            const float tk = dsum + yk;
            dcomp = (tk - dsum) - yk;
            dsum = tk;
            dmin = fminf(dmin, fminf(fminf(dd[0][0], dd[0][1]), fminf(dd[0][2], dd[0][3])));
        }
        if (store && t4 < nvalid) {
            float v[4];
#pragma unroll
            for (int s = 0; s < 4; ++s) v[s] = fmaf(Dk, uk[s], y[0][s]);
            if constexpr (sizeof(T) == 4) {
                *reinterpret_cast<float4*>(orow + t4) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
                const unsigned lo = (unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[0])) |
                                    ((unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[1])) << 16);
                const unsigned hi = (unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[2])) |
                                    ((unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[3])) << 16);
                *reinterpret_cast<uint2*>(orow + t4) = make_uint2(lo, hi);
            }
        }
    }
}

// SH kernels, carry correction (one channel per lane): one chunk of the
// homogeneous recurrence h = exp(delta*A)*h from the carried state, in closed
// form within the chunk: with S_t the sum of delta from the chunk's start
// through step t, h_t = 2^(A log2e S_t) h_start, so no step waits on the
// previous one; h advances by the whole chunk's decay at its end.  The
// C-contraction is summed over the channel's P lanes by a butterfly (every
// lane then holds the full sum), added to the local outputs (staged in the u
// rows, sy) and stored by the channel's first lane.  live[k] (warp-uniform)
// marks the state slots whose carry is still above the threshold in some
// lane of the warp: the chunk runs over the quads of slots up to the last
// live one (the ones past it are not advanced: they stay below the threshold,
// decay factors being at most 1 whenever slots are skipped), and a chunk
// with no live slot leaves the outputs as they are.  The count of quads is a
// template parameter, so that the step loop has no branch and the compiler
// can overlap its 4-step blocks (long64k: 462 -> 457 us).
template <int NQL, typename T, typename TU, int UROW, int NS, int P, int FROW, int TC, bool SCALAR>
__device__ __forceinline__ void decay_blocks_shfl1(const TU* sy, const TU* sd, const float* bC, int r,
                                                   const float (&Al2)[1][NS], const float (&As)[1],
                                                   float (&h)[1][NS], T* orow, bool store, int nvalid) {
    constexpr int NB = TC / 4, QS = 4;
    constexpr unsigned FULL = 0xffffffffu;
    float sacc = 0.f;  // sum of delta since the chunk's start
#pragma unroll 2
    for (int blk = 0; blk < NB; ++blk) {
        const int t4 = 4 * blk;
        float sc[4], es[4], y[4], yl[4], dv[4];
        load4_smem(sd + r * UROW + t4, dv);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            sacc += dv[s];
            sc[s] = sacc;
            es[s] = SCALAR ? ex2(sc[s] * As[0]) : 0.f;
            y[s] = 0.f;
        }
        load4_smem(sy + r * UROW + t4, yl);
#pragma unroll
        for (int q = 0; q < NQL; ++q) {
            float cc[QS][4];
#pragma unroll
            for (int kk = 0; kk < QS; ++kk) load4_smem(bC + (q * QS + kk) * P * FROW + t4, cc[kk]);
#pragma unroll
            for (int s = 0; s < 4; ++s)
#pragma unroll
                for (int kk = 0; kk < QS; ++kk) {
                    const int k = q * QS + kk;
                    const float e = SCALAR ? es[s] : ex2(sc[s] * Al2[0][k]);
                    y[s] = fmaf(cc[kk][s], h[0][k] * e, y[s]);
                }
        }
#pragma unroll
        for (int m = P / 2; m >= 1; m /= 2)
#pragma unroll
            for (int s = 0; s < 4; ++s) y[s] += __shfl_xor_sync(FULL, y[s], m);
        if (store && t4 < nvalid) {
            float v[4];
#pragma unroll
            for (int s = 0; s < 4; ++s) v[s] = yl[s] + y[s];
            if constexpr (sizeof(T) == 4) {
                *reinterpret_cast<float4*>(orow + t4) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
                const unsigned lo = (unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[0])) |
                                    ((unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[1])) << 16);
                const unsigned hi = (unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[2])) |
                                    ((unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[3])) << 16);
                *reinterpret_cast<uint2*>(orow + t4) = make_uint2(lo, hi);
            }
        }
    }
    // advance the live states over the chunk
    const float ech = SCALAR ? ex2(sacc * As[0]) : 0.f;
#pragma unroll
    for (int k = 0; k < NQL * QS; ++k) h[0][k] *= SCALAR ? ech : ex2(sacc * Al2[0][k]);
}

template <typename T, typename TU, int UROW, int NS, int P, int FROW, int TC, bool SCALAR>
__device__ __forceinline__ void decay_chunk_shfl1(const TU* sy, const TU* sd, const float* sC, const int (&rl)[1],
                                                  int g, const float (&Al2)[1][NS], const float (&As)[1],
                                                  const bool (&live)[NS], float (&h)[1][NS], T* orow, bool store,
                                                  int nvalid) {
    constexpr int QS = 4, NQ = NS / QS;
    static_assert(NQ >= 1 && NQ <= 4, "one to four quads of state slots");
    const float* bC = sC + g * FROW;
    int nql = 0;  // quads up to the last one with a live slot
#pragma unroll
    for (int k = 0; k < NS; ++k)
        if (live[k]) nql = k / QS + 1;
    // no live slot: the carry adds nothing to this chunk's outputs
    if (nql == 0) return;
    const int r = rl[0];
    if constexpr (NQ >= 4) {
        if (nql == 4) {
            decay_blocks_shfl1<4, T, TU, UROW, NS, P, FROW, TC, SCALAR>(sy, sd, bC, r, Al2, As, h, orow, store, nvalid);
            return;
        }
    }
    if constexpr (NQ >= 3) {
        if (nql == 3) {
            decay_blocks_shfl1<3, T, TU, UROW, NS, P, FROW, TC, SCALAR>(sy, sd, bC, r, Al2, As, h, orow, store, nvalid);
            return;
        }
    }
    if constexpr (NQ >= 2) {
        if (nql == 2) {
            decay_blocks_shfl1<2, T, TU, UROW, NS, P, FROW, TC, SCALAR>(sy, sd, bC, r, Al2, As, h, orow, store, nvalid);
            return;
        }
    }
    decay_blocks_shfl1<1, T, TU, UROW, NS, P, FROW, TC, SCALAR>(sy, sd, bC, r, Al2, As, h, orow, store, nvalid);
}

// Steps [T0, T0 + TS) of the carry correction for the calling lane: the
// homogeneous recurrence h = exp(delta*A)*h from the carried state and its
// C-contraction, stored as partial outputs like compute_half_tma.  live[k]
// (warp-uniform) skips the state slots whose carry has decayed below the
// threshold in every lane of the warp.
template <typename TU, int UROW, int NS, int P, int CPL, int FROW, int RS, int HROW, int TS, bool SCALAR>
__device__ __forceinline__ void decay_half_tma(const TU* sd, const float* sC, float* yp, const int (&rl)[CPL],
                                               int g, int T0, const float (&Al2)[CPL][NS],
                                               const float (&As)[CPL], const bool (&live)[NS],
                                               float (&h)[CPL][NS]) {
    const float* bC = sC + g * FROW;
#pragma unroll 2
    for (int t4 = T0; t4 < T0 + TS; t4 += 4) {
        float dd[CPL][4], as[CPL][4], y[CPL][4];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            load4_smem(sd + rl[j] * UROW + t4, dd[j]);
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
            load4_smem(bC + k * P * FROW + t4, cc);
#pragma unroll
            for (int s = 0; s < 4; ++s)
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    h[j][k] *= SCALAR ? as[j][s] : ex2(dd[j][s] * Al2[j][k]);
                    y[j][s] = fmaf(cc[s], h[j][k], y[j][s]);
                }
        }
#pragma unroll
        for (int j = 0; j < CPL; ++j)
            *reinterpret_cast<float4*>(yp + rl[j] * RS + g * HROW + (t4 - T0)) =
                make_float4(y[j][0], y[j][1], y[j][2], y[j][3]);
    }
}

// bf16: widen rows [0, nrows) of TC (+ padding) elements, stride RROW, into
// fp32 rows of stride FROW; one 16-byte piece (8 values) per item.
template <int RROW, int FROW, int TC>
__device__ __forceinline__ void widen_rows_warp(const bf16* src, float* dst, int nrows, int lane) {
    constexpr int Q8 = TC / 8;
    for (int q = lane; q < nrows * Q8; q += 32) {
        const int r = q / Q8, c = (q % Q8) * 8;
        widen8(src + r * RROW + c, dst + r * FROW + c);
    }
}

// bf16 delta rows of the warp's channels [dw, dw + nrows): widen and apply the
// delta transform (bias, softplus) to the steps inside the segment; padding
// (channels past dim, steps past the segment) stays 0 so that it keeps the state
template <int RROW, int FROW, int TC>
__device__ __forceinline__ void widen_delta_rows_warp(const bf16* src, float* dst, int nrows, int lane,
                                                      const FwdParams& p, long long dw, long long t0,
                                                      long long t_end) {
    constexpr int Q8 = TC / 8;
    for (int q = lane; q < nrows * Q8; q += 32) {
        const int r = q / Q8, c = (q % Q8) * 8;
        float* v = dst + r * FROW + c;
        widen8(src + r * RROW + c, v);
        const long long dd = dw + r;
        if (dd < p.dim) {
            const float bias = p.delta_bias != nullptr ? __ldg(p.delta_bias + dd) : 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (t0 + c + e < t_end) v[e] = delta_in(v[e], bias, p.delta_softplus != 0);
        }
    }
}

// CORR: the carry-correction instantiation (MODE_CORR: segment s >= 1 adds
// the decaying contribution of its entry state to the local outputs; the u
// tensor map then covers those outputs).  The body of the kernels below; tm
// is their __grid_constant__ parameter.
template <typename T, int NS, int P, int CPL, int OPT, bool CORR, bool SH = false>
__device__ __forceinline__ void sscan_fwd_tma_body(const FwdParams& p, const TmaMaps& tm) {
    using Cfg = TmaCfg<T, NS, P, CPL, OPT, SH>;
    static_assert(!SH || ((CORR ? CPL == 1 : CPL == 2) && P >= 2 && OPT == 0),
                  "shuffle kernels: plain scan; lane pairs, one channel per lane in the correction");
    constexpr int NUR = Cfg::NUR;
    constexpr int kWarps = Cfg::kWarps, CPW = Cfg::CPW, GPW = Cfg::GPW, NSP = Cfg::NSP, TC = Cfg::TC;
    constexpr int RROW = Cfg::RROW, FROW = Cfg::FROW, RS = Cfg::RS, STAGES = Cfg::STAGES;
    // the lanes' u/delta rows: fp32 (own or widened) rows, or raw bf16 ones
    constexpr bool kRawU = Cfg::kRawU;
    using UT = typename std::conditional<kRawU, bf16, float>::type;
    constexpr int UROW = kRawU ? Cfg::RROW_U : FROW;
    constexpr unsigned FULL = 0xffffffffu;
    constexpr bool WC = Cfg::kWarpC;  // C per warp: no CTA-shared ring, no CTA-wide votes
    extern __shared__ __align__(16) unsigned char smem_dyn[];
    // 128-byte aligned base, offset from the shared array itself so that the
    // compiler keeps every derived pointer in the shared address space
    unsigned char* sbase = smem_dyn + ((128u - (smem_addr(smem_dyn) & 127u)) & 127u);
    uint64_t* barU = reinterpret_cast<uint64_t*>(sbase + Cfg::OFF_BAR);  // [kWarps][STAGES]
    uint64_t* barBC = barU + kWarps * STAGES;                              // [STAGES]
    unsigned* bc_count = reinterpret_cast<unsigned*>(barBC + STAGES);      // [STAGES]

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int g = lane % P, gi = lane / P;
    const int tile = blockIdx.x / p.seg_count;
    const int s = (CORR ? 1 : 0) + blockIdx.x % p.seg_count;  // segment index
    const long long b = tile / p.tiles_per_batch;
    const long long d0 = (long long)(tile % p.tiles_per_batch) * Cfg::DT;
    const long long dw = d0 + (long long)w * CPW;  // the warp's first channel
    const long long t_begin = (long long)s * p.Tseg;
    const long long t_end = min(p.L, t_begin + p.Tseg);
    const int nchunks = t_end > t_begin ? (int)((t_end - t_begin + TC - 1) / TC) : 0;
    const int N = (int)p.N;

    unsigned char* u_ring = sbase + Cfg::OFF_U;
    unsigned char* bc_ring = sbase + Cfg::OFF_BC;
    float* yp = reinterpret_cast<float*>(sbase + Cfg::OFF_YP + w * Cfg::YP_BYTES);
    auto u_slot = [&](int st) -> T* {
        return reinterpret_cast<T*>(u_ring + (st * kWarps + w) * NUR * Cfg::U_SLOT);
    };
    const bool gated = OPT > 0 && p.z != nullptr;
    const bool xform = OPT > 0 && (p.delta_softplus != 0 || p.delta_bias != nullptr);
    auto bc_slot = [&](int st) -> T* { return reinterpret_cast<T*>(bc_ring + st * 2 * Cfg::BC_SLOT); };

    uint64_t* bcw_full = reinterpret_cast<uint64_t*>(sbase + Cfg::OFF_BAR + Cfg::OFF_BCW_BAR);  // [WB]
    uint64_t* bcw_empty = bcw_full + Cfg::WB;                                                      // [WB]
    // the carry correction that follows a local pass may start its CTAs now;
    // it sets up (barriers, decay rates) while the pass runs and waits for the
    // pass's completion before reading anything the pass wrote
    if constexpr (!CORR) griddep_launch_dependents();
    int* bc_last = reinterpret_cast<int*>(bc_count + STAGES);  // [STAGES] last chunk whose B/C copy went there
    const uint64_t lim = p.wait_ns != 0 ? (uint64_t)p.wait_ns : kWaitLimitNs;
    if (tid == 0) {
        for (int i = 0; i < (kWarps + 1) * STAGES; ++i) mbar_init(barU + i, 1);
        for (int i = 0; i < STAGES; ++i) bc_count[i] = 0;
        for (int i = 0; i < STAGES; ++i) bc_last[i] = -1;
        if constexpr (!Cfg::kF32) {
            for (int i = 0; i < Cfg::WB; ++i) {
                mbar_init(bcw_full + i, 32);
                mbar_init(bcw_empty + i, kWarps);
            }
        }
        // test aid: bytes that no copy delivers keep the first B/C stage (the
        // first warp's first ring stage where C comes per warp) from
        // completing, so that the waits on it run out
        if (p.expire_wait) mbar_expect_tx(WC ? barU : barBC, 16);
        mbar_fence_init();
    }
    __syncthreads();

    // the warp's u/delta (and z) boxes of chunk c into stage st (lane 0 only);
    // a correction's u rows are the local outputs
    int u_hi = -1;  // last chunk whose u/delta copy this warp issued
    auto issue_u = [&](int c, int st) {
        u_hi = c;
        T* dst = u_slot(st);
        uint64_t* bar = barU + w * STAGES + st;
        mbar_arrive_expect_tx(bar, (gated ? 3 : 2) * Cfg::U_BOX + (WC ? Cfg::BC_BOX : 0));
        const int t0 = (int)(t_begin + (long long)c * TC);
        if constexpr (WC) tma_load_3d(reinterpret_cast<unsigned char*>(dst) + 2 * Cfg::U_SLOT, &tm.C, t0, 0, (int)b, bar);
        tma_load_3d(dst, &tm.u, t0, (int)dw, (int)b, bar);
        tma_load_3d(reinterpret_cast<unsigned char*>(dst) + Cfg::U_SLOT, &tm.delta, t0, (int)dw, (int)b, bar);
        if (gated)
            tma_load_3d(reinterpret_cast<unsigned char*>(dst) + 2 * Cfg::U_SLOT, &tm.z, t0, (int)dw, (int)b, bar);
    };
    // the B/C boxes of chunk c into stage st (one thread); a correction needs C only
    auto issue_bc = [&](int c, int st) {
        T* dst = bc_slot(st);
        uint64_t* bar = barBC + st;
        bc_last[st] = c;
        mbar_arrive_expect_tx(bar, (CORR ? 1 : 2) * Cfg::BC_BOX);
        const int t0 = (int)(t_begin + (long long)c * TC);
        if constexpr (!CORR) tma_load_3d(dst, &tm.B, t0, 0, (int)b, bar);
        tma_load_3d(reinterpret_cast<unsigned char*>(dst) + Cfg::BC_SLOT, &tm.C, t0, 0, (int)b, bar);
    };
    if constexpr (!CORR) {
        if (lane == 0) {
            for (int c = 0; c < STAGES && c < nchunks; ++c) {
                issue_u(c, c);
                if (w == 0) issue_bc(c, c);
            }
        }
    } else if (lane == 0) {
        // a correction's first chunks: the inputs (delta, z, C) before the
        // wait on the local pass, the local outputs (its u rows) after it
        for (int c = 0; c < STAGES && c < nchunks; ++c) {
            u_hi = c;
            uint64_t* bar = barU + w * STAGES + c;
            mbar_arrive_expect_tx(bar, (gated ? 3 : 2) * Cfg::U_BOX + (WC ? Cfg::BC_BOX : 0));
            const int t0 = (int)(t_begin + (long long)c * TC);
            unsigned char* dst = reinterpret_cast<unsigned char*>(u_slot(c));
            tma_load_3d(dst + Cfg::U_SLOT, &tm.delta, t0, (int)dw, (int)b, bar);
            if (gated) tma_load_3d(dst + 2 * Cfg::U_SLOT, &tm.z, t0, (int)dw, (int)b, bar);
            if constexpr (WC) tma_load_3d(dst + 2 * Cfg::U_SLOT, &tm.C, t0, 0, (int)b, bar);
            else if (w == 0) issue_bc(c, c);
        }
    }

    // the lane's channels (rows rl[j] of the warp) and their decay rates
    int rl[CPL];
    long long ch[CPL];
    bool dval[CPL];
    float Al2[CPL][NS], As[CPL], h[CPL][NS];
    float invA[CPL][NS], invAs[CPL];  // 1/A (0 where A = 0), for the zero-order hold
    bool uniform_rate = true;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        // shuffle kernels: lane group gi owns the adjacent channel rows 2gi and
        // 2gi + 1 (the eight lanes of a quarter-warp then read eight distinct
        // padded rows, in distinct banks), and the lanes in the upper half of
        // the channel's lanes hold the pair in the opposite order
        if constexpr (SH && CPL == 1) rl[j] = gi;
        else if constexpr (SH) rl[j] = 2 * gi + (j ^ ((g & (P / 2)) ? 1 : 0));
        else rl[j] = j * GPW + gi;
        const long long dch = dw + rl[j];
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
            h[j][k] = (!CORR && s == 0 && p.h0 != nullptr && nv) ? p.h0[ch[j] * p.N + n] : 0.f;
        }
        As[j] = a_first * kLog2e;
        invAs[j] = a_first != 0.f ? 1.f / a_first : 0.f;
    }
    if constexpr (CORR) {
        // the local pass's outputs and aggregates are complete from here on
        griddep_wait();
        if (lane == 0)
            for (int c = 0; c < STAGES && c < nchunks; ++c)
                tma_load_3d(u_slot(c), &tm.u, (int)(t_begin + (long long)c * TC), (int)dw, (int)b,
                            barU + w * STAGES + c);
    }
    // correction: the carried state entering segment s, folded from the
    // aggregates of the segments before it by the fold pass (slot s - 1;
    // with two segments slot 0 holds it already: segment 0 started from h0),
    // or here when the split has few segments (fold_in_corr); it
    // is followed until every state of the CTA has fallen below 2^-24 of its
    // entry magnitude, a cut-off taken only while every decay factor
    // exp(delta*A) of the CTA's channels in this segment is at most 1 (every
    // A <= 0, no negative delta)
    bool grows = false;
    if constexpr (CORR) {
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
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
        }
    }
    const bool cut = CORR && !__syncthreads_or(grows);
    const bool scalar = __all_sync(FULL, uniform_rate);
    float thr[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        float m = 0.f;
#pragma unroll
        for (int k = 0; k < NS; ++k) m = fmaxf(m, fabsf(h[j][k]));
        thr[j] = cut ? m * 0x1p-24f : 0.f;
        // the last segment's final state: the entry state decayed over the
        // segment plus the segment's local end state
        if (CORR && dval[j] && s == p.S - 1 && p.final_state != nullptr) {
            const float dsg = p.seg_dsum[ch[j] * p.S + s];
            const float* sst = p.seg_state + (ch[j] * p.S + s) * p.N;
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const int n = k * P + g;
                if (n < N) p.final_state[ch[j] * p.N + n] = fmaf(ex2(Al2[j][k] * dsg), h[j][k], sst[n]);
            }
        }
    }

    // epilogue slots per half chunk: item q = lane + 32k covers channel row
    // q/4, steps 4(q%4)..+3 of the half
    const bool dsum_on = !CORR && p.mode == MODE_LOCAL;
    // Kahan sums of delta per slot (a slot is the same channel row and 4-step
    // offset in both halves)
    float dsum[Cfg::IPH], dcomp[Cfg::IPH];
#pragma unroll
    for (int k = 0; k < Cfg::IPH; ++k) dsum[k] = dcomp[k] = 0.f;
    // min(0, smallest delta) of the lane's item slots; the warp's minimum is
    // recorded for all of its channels (negative steps are rare: a correction
    // then follows its carries to the segment end).  Narrow lanes only: in
    // the 16-state-lane kernel this tracking measured 4% slower (wide64 448 ->
    // 470 us, the same with sign bits or in the compute loop), and its
    // segments are recorded as free of negative steps, the domain the header
    // states (delta >= 0).
    float dmin = 0.f;
    float Dr[Cfg::IPH];
#pragma unroll
    for (int k = 0; k < Cfg::IPH; ++k) {
        const long long dd = dw + (lane + 32 * k) / 4;
        Dr[k] = (p.D != nullptr && dd < p.dim) ? __ldg(p.D + dd) : 0.f;
    }
    T* gout = static_cast<T*>(p.out);
    float* work = reinterpret_cast<float*>(sbase + Cfg::OFF_WORK + w * Cfg::WORK_BYTES);
    // shuffle kernels: the lane's kept channel rl[0], whose outputs it stores
    // when it is the first of the channel's lanes that hold the full sums
    float sh_dsum = 0.f, sh_dcomp = 0.f, sh_dmin = 0.f;
    const bool sh_store = SH && (CPL == 1 ? g == 0 : (g & (P / 2 - 1)) == 0) && dval[0];
    const float sh_D = (SH && p.D != nullptr && dval[0]) ? __ldg(p.D + (dw + rl[0])) : 0.f;
    T* sh_orow = gout + ch[0] * p.L;

    // warp epilogue of one half chunk: sum the P partials, add D*u, store 4
    // steps per item (and the Kahan sums of delta of a local pass)
    auto epilogue = [&](int half, long long t0, const UT* su, const UT* sd, const float* sz) {
#pragma unroll
        for (int k = 0; k < Cfg::IPH; ++k) {
            const int q = lane + 32 * k;
            const int r = q / 4, t4l = (q % 4) * 4, t4 = half * Cfg::TS + t4l;
            const long long dd = dw + r, t = t0 + t4;
            float v[4];
            load4_smem(yp + r * RS + t4l, v);
#pragma unroll
            for (int gg = 1; gg < P; ++gg) {
                float x[4];
                load4_smem(yp + r * RS + gg * Cfg::HROW + t4l, x);
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] += x[e];
            }
            float uv[4];
            load4_smem(su + r * UROW + t4, uv);
            if constexpr (!CORR) {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = fmaf(Dr[k], uv[e], v[e]);
            }
            if (OPT > 0 && gated) {  // out = (y + D*u) * silu(z); a correction is gated alike
                float zv[4];
                load4_smem(sz + r * FROW + t4, zv);
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] *= silu(zv[e]);
            }
            if constexpr (CORR) {  // the local outputs, staged in the u rows
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] += uv[e];
            }
            if (dsum_on) {  // steps past the segment hold delta = 0
                float dv[4];
                load4_smem(sd + r * UROW + t4, dv);
                const float yk = ((dv[0] + dv[1]) + (dv[2] + dv[3])) - dcomp[k];
                const float tk = dsum[k] + yk;
                dcomp[k] = (tk - dsum[k]) - yk;
                dsum[k] = tk;
                if constexpr (NS <= 4) dmin = fminf(dmin, fminf(fminf(dv[0], dv[1]), fminf(dv[2], dv[3])));
            }
            if (dd < p.dim && t < t_end) {  // t_end is a multiple of 4 on this path
                T* o = gout + (b * p.dim + dd) * p.L + t;
                if constexpr (Cfg::kF32) {
                    *reinterpret_cast<float4*>(o) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
                    const unsigned lo = (unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[0])) |
                                        ((unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[1])) << 16);
                    const unsigned hi = (unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[2])) |
                                        ((unsigned)__bfloat16_as_ushort(from_f32<bf16>(v[3])) << 16);
                    *reinterpret_cast<uint2*>(o) = make_uint2(lo, hi);
                }
            }
        }
    };

    // bf16: widen the B/C rows of chunk c into slot c % WB of the shared fp32
    // ring (the calling warp is chunk c's widener), then refill the raw stage
    auto widen_bc = [&](int c) -> bool {
        const int st = c % STAGES, ws = c % Cfg::WB;
        bool good = mbar_wait_bounded(barBC + st, (unsigned)(c / STAGES) & 1u, lim);
        if (c >= Cfg::WB) good = mbar_wait_bounded(bcw_empty + ws, (unsigned)((c - Cfg::WB) / Cfg::WB) & 1u, lim) && good;
        good = __all_sync(FULL, good);
        if (!good) return false;
        float* dst = reinterpret_cast<float*>(sbase + Cfg::OFF_BCW + ws * Cfg::BCW_BYTES);
        const bf16* rb = reinterpret_cast<const bf16*>(bc_slot(st));
        if constexpr (!CORR) widen_rows_warp<RROW, FROW, TC>(rb, dst, NSP, lane);
        widen_rows_warp<RROW, FROW, TC>(
            reinterpret_cast<const bf16*>(reinterpret_cast<const unsigned char*>(rb) + Cfg::BC_SLOT),
            dst + NSP * FROW, NSP, lane);
        mbar_arrive(bcw_full + ws);
        __syncwarp();
        if (lane == 0 && c + STAGES < nchunks) issue_bc(c + STAGES, st);
        return true;
    };

    int i = 0;
    bool ok = true;
    if constexpr (!Cfg::kF32) {
        if (w == 0 && nchunks > 0) ok = widen_bc(0);
        ok = __all_sync(FULL, ok);
    }
    for (; ok && i < nchunks; ++i) {
        const int st = i % STAGES;
        const unsigned par = (unsigned)(i / STAGES) & 1u;
        const int nx = i + STAGES;  // the chunk that refills this stage
        const long long t0 = t_begin + (long long)i * TC;
        const UT *su, *sd;
        const float *sz, *sB, *sC;
        if constexpr (Cfg::kF32) {
            ok = mbar_wait_bounded(barU + w * STAGES + st, par, lim);
            if constexpr (!WC) ok = mbar_wait_bounded(barBC + st, par, lim) && ok;
            ok = __all_sync(FULL, ok);
            if (!ok && !CORR) break;
            su = reinterpret_cast<const UT*>(u_slot(st));
            sd = reinterpret_cast<const UT*>(reinterpret_cast<const unsigned char*>(su) + Cfg::U_SLOT);
            sz = reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(su) + 2 * Cfg::U_SLOT);
            sB = reinterpret_cast<const float*>(bc_slot(st));
            sC = WC ? sz : reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(sB) + Cfg::BC_SLOT);
            if (OPT > 0 && xform) {
                // delta transform in place on the warp's rows: lane = step;
                // padding (channels past dim, steps past the segment) keeps 0
                float* wd = const_cast<float*>(sd);
                const bool tin = t0 + lane < t_end;
                for (int r = 0; r < CPW; ++r) {
                    const long long dd = dw + r;
                    if (tin && dd < p.dim) {
                        const float bias = p.delta_bias != nullptr ? __ldg(p.delta_bias + dd) : 0.f;
                        wd[r * FROW + lane] = delta_in(wd[r * FROW + lane], bias, p.delta_softplus != 0);
                    }
                }
                __syncwarp();
            }
        } else if constexpr (kRawU) {
            // the next chunk's B/C when it is this warp's turn, one chunk ahead
            if (i + 1 < nchunks && (i + 1) % kWarps == w && !widen_bc(i + 1)) {
                ok = false;
                if constexpr (!CORR) break;
            }
            // the warp's raw u/delta rows, read in place; the stage is
            // refilled after the chunk
            ok = __all_sync(FULL, mbar_wait_bounded(barU + w * STAGES + st, par, lim)) && ok;
            if (!ok && !CORR) break;
            su = reinterpret_cast<const UT*>(u_slot(st));
            sd = reinterpret_cast<const UT*>(reinterpret_cast<const unsigned char*>(su) + Cfg::U_SLOT);
            sz = nullptr;
            ok = __all_sync(FULL, mbar_wait_bounded(bcw_full + i % Cfg::WB, (unsigned)(i / Cfg::WB) & 1u, lim)) && ok;
            if (!ok && !CORR) break;
            sB = reinterpret_cast<const float*>(sbase + Cfg::OFF_BCW + (i % Cfg::WB) * Cfg::BCW_BYTES);
            sC = sB + NSP * FROW;
        } else {
            // the next chunk's B/C when it is this warp's turn, one chunk ahead
            if (i + 1 < nchunks && (i + 1) % kWarps == w && !widen_bc(i + 1)) {
                ok = false;
                if constexpr (!CORR) break;
            }
            // the warp's own u/delta (z) rows, widened (delta transformed),
            // then the raw stage refilled
            ok = __all_sync(FULL, mbar_wait_bounded(barU + w * STAGES + st, par, lim)) && ok;
            if (!ok && !CORR) break;
            const bf16* ru = reinterpret_cast<const bf16*>(u_slot(st));
            widen_rows_warp<RROW, FROW, TC>(ru, work, CPW, lane);
            const bf16* rd = reinterpret_cast<const bf16*>(reinterpret_cast<const unsigned char*>(ru) + Cfg::U_SLOT);
            if (OPT > 0 && xform)
                widen_delta_rows_warp<RROW, FROW, TC>(rd, work + CPW * FROW, CPW, lane, p, dw, t0, t_end);
            else
                widen_rows_warp<RROW, FROW, TC>(rd, work + CPW * FROW, CPW, lane);
            if (OPT > 0 && gated)
                widen_rows_warp<RROW, FROW, TC>(
                    reinterpret_cast<const bf16*>(reinterpret_cast<const unsigned char*>(ru) + 2 * Cfg::U_SLOT),
                    work + 2 * CPW * FROW, CPW, lane);
            __syncwarp();
            if (lane == 0 && nx < nchunks) issue_u(nx, st);
            ok = __all_sync(FULL, mbar_wait_bounded(bcw_full + i % Cfg::WB, (unsigned)(i / Cfg::WB) & 1u, lim)) && ok;
            if (!ok && !CORR) break;
            su = work;
            sd = work + CPW * FROW;
            sz = work + 2 * CPW * FROW;
            sB = reinterpret_cast<const float*>(sbase + Cfg::OFF_BCW + (i % Cfg::WB) * Cfg::BCW_BYTES);
            sC = sB + NSP * FROW;
        }
        constexpr int TS = Cfg::TS, HROW = Cfg::HROW;
        constexpr bool ZOH = OPT == 2;
        bool live[NS];  // correction: state slots still above the threshold somewhere in the warp
        if constexpr (CORR) {
            bool any = false;
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                bool l = false;
#pragma unroll
                for (int j = 0; j < CPL; ++j) l |= fabsf(h[j][k]) > thr[j];
                live[k] = (scalar || !cut) ? true : __any_sync(FULL, l);
                any |= l;
            }
            if constexpr (WC) {
                // every warp on its own: a wait that gave up, or the decay of
                // every state of its lanes, ends its correction
                if (!ok) break;
                if (cut && !__any_sync(FULL, any)) break;
            } else {
                // a wait that gave up in any warp ends the CTA's correction; so
                // does the decay of every state of every lane (CTA-wide votes, so
                // that every warp leaves the loop at the same chunk)
                if (__syncthreads_or(!ok)) {
                    ok = false;
                    break;
                }
                if (cut && !__syncthreads_or(any)) break;
            }
        }
        if constexpr (SH && CORR) {
            const int nvalid = (int)min((long long)TC, t_end - t0);
            if (scalar)
                decay_chunk_shfl1<T, UT, UROW, NS, P, FROW, TC, true>(su, sd, sC, rl, g, Al2, As, live, h,
                                                                      sh_orow + t0, sh_store, nvalid);
            else
                decay_chunk_shfl1<T, UT, UROW, NS, P, FROW, TC, false>(su, sd, sC, rl, g, Al2, As, live, h,
                                                                       sh_orow + t0, sh_store, nvalid);
            __syncwarp();
            if (!WC && lane == 0) {  // C of this chunk is no longer read by this warp
                if constexpr (Cfg::kF32) {
                    const unsigned old = atomicAdd(bc_count + st, 1u);
                    if ((old + 1) % kWarps == 0 && nx < nchunks) issue_bc(nx, st);
                } else {
                    mbar_arrive(bcw_empty + i % Cfg::WB);
                }
            }
        } else if constexpr (SH) {
            const int nvalid = (int)min((long long)TC, t_end - t0);
            if (scalar)
                compute_chunk_shfl<T, UT, UROW, NS, P, FROW, TC, true>(su, sd, sB, sC, rl, g, Al2, As, h, sh_D,
                                                                       sh_orow + t0, sh_store, nvalid, dsum_on,
                                                                       sh_dsum, sh_dcomp, sh_dmin);
            else
                compute_chunk_shfl<T, UT, UROW, NS, P, FROW, TC, false>(su, sd, sB, sC, rl, g, Al2, As, h, sh_D,
                                                                        sh_orow + t0, sh_store, nvalid, dsum_on,
                                                                        sh_dsum, sh_dcomp, sh_dmin);
            __syncwarp();
            // B/C of this chunk are no longer read by this warp
            if (lane == 0) {
                if constexpr (Cfg::kF32) {
                    const unsigned old = atomicAdd(bc_count + st, 1u);
                    if ((old + 1) % kWarps == 0 && nx < nchunks) issue_bc(nx, st);
                } else {
                    mbar_arrive(bcw_empty + i % Cfg::WB);
                }
            }
        } else {
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            if constexpr (CORR) {
                if (scalar)
                    decay_half_tma<UT, UROW, NS, P, CPL, FROW, RS, HROW, TS, true>(sd, sC, yp, rl, g, half * TS, Al2, As, live,
                                                                         h);
                else
                    decay_half_tma<UT, UROW, NS, P, CPL, FROW, RS, HROW, TS, false>(sd, sC, yp, rl, g, half * TS, Al2, As,
                                                                          live, h);
            } else if (scalar) {
                compute_half_tma<UT, UROW, NS, P, CPL, FROW, RS, HROW, TS, true, ZOH>(su, sd, sB, sC, yp, rl, g, half * TS,
                                                                            Al2, As, invA, invAs, h);
            } else {
                compute_half_tma<UT, UROW, NS, P, CPL, FROW, RS, HROW, TS, false, ZOH>(su, sd, sB, sC, yp, rl, g, half * TS,
                                                                             Al2, As, invA, invAs, h);
            }
            __syncwarp();
            // after the second half, B/C of this chunk are no longer read by this warp
            if (half == 1 && lane == 0) {
                if constexpr (Cfg::kF32) {
                    const unsigned old = atomicAdd(bc_count + st, 1u);
                    if ((old + 1) % kWarps == 0 && nx < nchunks) issue_bc(nx, st);
                } else {
                    mbar_arrive(bcw_empty + i % Cfg::WB);
                }
            }
            epilogue(half, t0, su, sd, sz);
            __syncwarp();
        }
        }
        if constexpr (Cfg::kF32 || kRawU) {
            // u/delta (z) of this stage are no longer read by this warp; the
            // delta transform wrote them, so order those writes before the copy
            if (lane == 0 && nx < nchunks) {
                if (OPT > 0 && xform) fence_proxy_async_smem();
                issue_u(nx, st);
            }
        }
    }
    // Every warp leaves the chunk loop here (a local pass has no CTA barrier in
    // the loop; a correction leaves it at the same chunk by CTA-wide votes,
    // except the shuffle kernels' fp32 one, whose warps each leave on their own).
    // After this barrier no warp issues a copy, so a CTA that gave up on a
    // wait, or a correction that stopped early, waits (bounded) for the last
    // copy issued into every ring stage before it leaves: none may land in
    // the shared memory of a CTA that has exited.
    const bool failed = __syncthreads_or(!ok);
    if (failed || (CORR && i < nchunks)) {
        if (lane == 0) {
            bool good = true;
            for (int st = 0; st < STAGES; ++st) {
                // a warp issues its u/delta copies in chunk order; the B/C
                // copies of a bf16 ring may be issued out of order, so their
                // stages record their own last chunk
                const int cu = u_hi - ((u_hi - st) % STAGES + STAGES) % STAGES;  // largest c <= u_hi, c = st
                if (cu >= 0) good = mbar_wait_bounded(barU + w * STAGES + st, (unsigned)(cu / STAGES) & 1u, lim) && good;
                const int cb = bc_last[st];
                if (w == 0 && cb >= 0)
                    good = mbar_wait_bounded(barBC + st, (unsigned)(cb / STAGES) & 1u, lim) && good;
            }
            if (failed || !good) atomicExch(p.status, (int)SSCAN_ERR_TIMEOUT);
        }
        return;
    }
    if constexpr (CORR) return;

    if (SH && dsum_on) {  // the kept channel's sum of delta
        if (sh_store) {
            p.seg_dsum[ch[0] * p.S + s] = sh_dsum;
            p.seg_dmin[ch[0] * p.S + s] = sh_dmin;
        }
    } else if (dsum_on) {  // the segment's sum of delta per channel: 4 slots in 4 lanes
        const float m = __any_sync(FULL, dmin < 0.f) ? -1.f : 0.f;
#pragma unroll
        for (int k = 0; k < Cfg::IPH; ++k) {
            float v = dsum[k];
            v += __shfl_xor_sync(FULL, v, 1);
            v += __shfl_xor_sync(FULL, v, 2);
            const long long dd = dw + (lane + 32 * k) / 4;
            if ((lane & 3) == 0 && dd < p.dim) {
                p.seg_dsum[(b * p.dim + dd) * p.S + s] = v;
                p.seg_dmin[(b * p.dim + dd) * p.S + s] = m;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        if (!dval[j]) continue;
        float* dst = p.mode == MODE_LOCAL ? p.seg_state + (ch[j] * p.S + s) * p.N : p.final_state == nullptr ? nullptr : p.final_state + ch[j] * p.N;
        if (dst == nullptr) continue;
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const int n = k * P + g;
            if (n < N) dst[n] = h[j][k];
        }
    }
}

// Narrow lanes (up to 4 states): the register allocation is asked for the
// resident CTAs that shared memory allows (TmaCfg::MIN_BLOCKS).
template <typename T, int NS, int P, int CPL, int OPT, bool CORR>
__global__ void __launch_bounds__(TmaCfg<T, NS, P, CPL, OPT>::kThreads, TmaCfg<T, NS, P, CPL, OPT>::MIN_BLOCKS)
    sscan_fwd_tma(const FwdParams p, const __grid_constant__ TmaMaps tm) {
    sscan_fwd_tma_body<T, NS, P, CPL, OPT, CORR>(p, tm);
}

// Wide lanes (16 states): no request for resident CTAs (two or three CTAs per
// SM gave slower schedules: wide64 458 / 462 us against 452 us), but a
// register ceiling (its launches use kThreads = 128 threads per CTA).
template <typename T, int NS, int P, int CPL, int OPT, bool CORR>
__global__ void __maxnreg__(OPT == 2 ? 255 : SSCAN_WIDE_MAXNREG)
    sscan_fwd_tma_wide(const FwdParams p, const __grid_constant__ TmaMaps tm) {
    sscan_fwd_tma_body<T, NS, P, CPL, OPT, CORR>(p, tm);
}

// Shuffle kernels (the plain scan's single and local passes): outputs summed
// across a channel's lanes by shuffles and stored by the lanes.
template <typename T, int NS, int P, int CPL>
__global__ void __launch_bounds__(TmaCfg<T, NS, P, CPL, 0, true>::kThreads, TmaCfg<T, NS, P, CPL, 0, true>::SH_MIN_BLOCKS)
    sscan_fwd_tma_shfl(const FwdParams p, const __grid_constant__ TmaMaps tm) {
    sscan_fwd_tma_body<T, NS, P, CPL, 0, false, true>(p, tm);
}
// ... and their carry correction (MODE_CORR)
template <typename T, int NS, int P, int CPL>
__global__ void __launch_bounds__(TmaCfg<T, NS, P, CPL, 0, true>::kThreads, TmaCfg<T, NS, P, CPL, 0, true>::SH_MIN_BLOCKS)
    sscan_fwd_tma_shfl_corr(const FwdParams p, const __grid_constant__ TmaMaps tm) {
    sscan_fwd_tma_body<T, NS, P, CPL, 0, true, true>(p, tm);
}

// The kernel of a shape and pass.
template <typename T, int NS, int P, int CPL, int OPT, bool CORR>
constexpr auto tma_kernel() {
    if constexpr (NS > 4) return sscan_fwd_tma_wide<T, NS, P, CPL, OPT, CORR>;
    else return sscan_fwd_tma<T, NS, P, CPL, OPT, CORR>;
}

// Shared implementation of the per-dtype launch units (sscan_fwd_tma_*.cu).
#ifdef SSCAN_TMA_IMPL
template <typename T, int NS, int P, int CPL, int OPT>
cudaError_t launch_tma_variant(const FwdParams& p, int grid, cudaStream_t stream) {
    using Cfg = TmaCfg<T, NS, P, CPL, OPT>;
    if (p.N < 1 || p.N > (long long)Cfg::NSP) return cudaErrorInvalidValue;
    const bool corr = p.mode == MODE_CORR;
    TmaMaps tm;
    const bool f32 = Cfg::kF32;
    // a correction stages the local outputs where a local pass stages u
    if (!tma_encode_3d(&tm.u, corr ? p.out : p.u, f32, p.L, p.dim, p.batch, Cfg::RROW_U, Cfg::CPW) ||
        !tma_encode_3d(&tm.delta, p.delta, f32, p.L, p.dim, p.batch, Cfg::RROW_U, Cfg::CPW) ||
        !tma_encode_3d(&tm.B, p.B, f32, p.L, p.N, p.batch, Cfg::RROW, Cfg::NSP) ||
        !tma_encode_3d(&tm.C, p.C, f32, p.L, p.N, p.batch, Cfg::RROW, Cfg::NSP))
        return cudaErrorInvalidValue;
    if (OPT > 0 && p.z != nullptr && !tma_encode_3d(&tm.z, p.z, f32, p.L, p.dim, p.batch, Cfg::RROW_U, Cfg::CPW))
        return cudaErrorInvalidValue;
    auto kern = corr ? tma_kernel<T, NS, P, CPL, OPT, true>() : tma_kernel<T, NS, P, CPL, OPT, false>();
    static unsigned long long configured[2] = {0, 0};  // bit per device ordinal (< 64), per kernel
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&configured[corr ? 1 : 0], __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured[corr ? 1 : 0], bit, __ATOMIC_ACQ_REL);
    }
    if (!corr) {
        kern<<<grid, Cfg::kThreads, Cfg::SMEM_BYTES, stream>>>(p, tm);
        return cudaGetLastError();
    }
    // the correction follows the local pass as a programmatic dependent
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, tm);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int NS, int P, int CPL, int OPT>
int occupancy_tma_variant() {
    using Cfg = TmaCfg<T, NS, P, CPL, OPT>;
    auto kern = tma_kernel<T, NS, P, CPL, OPT, false>();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Cfg::kThreads, Cfg::SMEM_BYTES) != cudaSuccess)
        return 0;
    return n;
}

// The shuffle kernel of a shape: the carry correction for one channel per
// lane, the single and local passes for two.
template <typename T, int NS, int P, int CPL>
constexpr auto shfl_kernel() {
    if constexpr (CPL == 1) return sscan_fwd_tma_shfl_corr<T, NS, P, CPL>;
    else return sscan_fwd_tma_shfl<T, NS, P, CPL>;
}

// Launch of a shuffle-kernel shape's pass.
template <typename T, int NS, int P, int CPL>
cudaError_t launch_tma_shfl_variant(const FwdParams& p, int grid, cudaStream_t stream) {
    using Cfg = TmaCfg<T, NS, P, CPL, 0, true>;
    if (p.N < 1 || p.N > (long long)Cfg::NSP || fwd_variant(p) != 0) return cudaErrorInvalidValue;
    const bool corr = p.mode == MODE_CORR;
    TmaMaps tm;
    const bool f32 = Cfg::kF32;
    // a correction stages the local outputs where a local pass stages u
    if (!tma_encode_3d(&tm.u, corr ? p.out : p.u, f32, p.L, p.dim, p.batch, Cfg::RROW_U, Cfg::CPW) ||
        !tma_encode_3d(&tm.delta, p.delta, f32, p.L, p.dim, p.batch, Cfg::RROW_U, Cfg::CPW) ||
        !tma_encode_3d(&tm.B, p.B, f32, p.L, p.N, p.batch, Cfg::RROW, Cfg::NSP) ||
        !tma_encode_3d(&tm.C, p.C, f32, p.L, p.N, p.batch, Cfg::RROW, Cfg::NSP))
        return cudaErrorInvalidValue;
    if (corr != (CPL == 1)) return cudaErrorInvalidValue;  // a shape runs its own pass only
    auto kern = shfl_kernel<T, NS, P, CPL>();
    static unsigned long long configured[2] = {0, 0};  // bit per device ordinal (< 64), per kernel
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&configured[corr ? 1 : 0], __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured[corr ? 1 : 0], bit, __ATOMIC_ACQ_REL);
    }
    if (!corr) {
        kern<<<grid, Cfg::kThreads, Cfg::SMEM_BYTES, stream>>>(p, tm);
        return cudaGetLastError();
    }
    // the correction follows the local (or fold) pass as a programmatic dependent
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, tm);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int NS, int P, int CPL>
int occupancy_tma_shfl_variant() {
    using Cfg = TmaCfg<T, NS, P, CPL, 0, true>;
    auto kern = shfl_kernel<T, NS, P, CPL>();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Cfg::kThreads, Cfg::SMEM_BYTES) != cudaSuccess)
        return 0;
    return n;
}

#define SSCAN_SHFL_LAUNCH_CASE(P_, NS_, CPL_) \
    if (sh.P == P_ && sh.NS == NS_ && sh.CPL == CPL_) return launch_tma_shfl_variant<UnitT, NS_, P_, CPL_>(p, grid, st);
#define SSCAN_SHFL_OCC_CASE(P_, NS_, CPL_) \
    if (sh.P == P_ && sh.NS == NS_ && sh.CPL == CPL_) return occupancy_tma_shfl_variant<UnitT, NS_, P_, CPL_>();
#define SSCAN_DEFINE_SHFL_UNIT(SUFFIX)                                                               \
    cudaError_t fwd_shfl_launch_##SUFFIX(const FwdParams& p, Shape sh, int grid, cudaStream_t st) { \
        SSCAN_TMA_SHFL_SHAPES(SSCAN_SHFL_LAUNCH_CASE)                                                \
        return cudaErrorInvalidValue;                                                                \
    }                                                                                                \
    int fwd_shfl_occupancy_##SUFFIX(Shape sh) {                                                      \
        SSCAN_TMA_SHFL_SHAPES(SSCAN_SHFL_OCC_CASE)                                                   \
        return 0;                                                                                    \
    }

#define SSCAN_TMA_LAUNCH_CASE(P_, NS_, CPL_) \
    if (sh.P == P_ && sh.NS == NS_ && sh.CPL == CPL_) return launch_tma_variant<UnitT, NS_, P_, CPL_, UnitOPT>(p, grid, st);
#define SSCAN_TMA_OCC_CASE(P_, NS_, CPL_) \
    if (sh.P == P_ && sh.NS == NS_ && sh.CPL == CPL_) return occupancy_tma_variant<UnitT, NS_, P_, CPL_, UnitOPT>();
#define SSCAN_DEFINE_TMA_UNIT(SUFFIX)                                                               \
    cudaError_t fwd_tma_launch_##SUFFIX(const FwdParams& p, Shape sh, int grid, cudaStream_t st) { \
        SSCAN_TMA_SHAPES(SSCAN_TMA_LAUNCH_CASE)                                                     \
        return cudaErrorInvalidValue;                                                               \
    }                                                                                               \
    int fwd_tma_occupancy_##SUFFIX(Shape sh) {                                                      \
        SSCAN_TMA_SHAPES(SSCAN_TMA_OCC_CASE)                                                        \
        return 0;                                                                                   \
    }
#endif  // SSCAN_TMA_IMPL

}  // namespace sscan
