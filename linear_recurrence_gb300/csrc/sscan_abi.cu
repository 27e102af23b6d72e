// C ABI of libsscan.so (declared in include/sscan.h): argument validation,
// launch planning and stream-ordered scratch for the selective-scan and pscan
// kernels.  Nothing here computes on the host; every step of the scan runs in
// the kernels it launches.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/sscan.h"
#include "pscan_kernel.cuh"
#include "sscan_dispatch.cuh"

namespace {

using sscan::FwdParams;
using sscan::Shape;

struct CallRecord {
    int launches = 0;
    cudaStream_t stream = nullptr;
    int pending_error = SSCAN_OK;
    char plan[256] = "none";
};
thread_local CallRecord g_rec;
// sscan_debug_expire_next_wait: the bound (microseconds) of the waits of this
// thread's next forward call, whose first B/C stage is made to never complete
// (0: not armed)
thread_local unsigned g_expire_wait_us = 0;
// sscan_debug_expire_next_correction_wait: the same for the carry correction
// of this thread's next forward call (0: not armed)
thread_local unsigned g_expire_corr_us = 0;

int sm_count() {
    static std::atomic<int> cached[64] = {};  // per device ordinal; host threads may race
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::atomic<int>& c = cached[dev & 63];
    int v = c.load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        c.store(v, std::memory_order_relaxed);
    }
    return v;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

int fail_cuda(cudaError_t e) {
    g_rec.pending_error = SSCAN_ERR_CUDA;
    snprintf(g_rec.plan, sizeof(g_rec.plan), "cuda error: %s", cudaGetErrorString(e));
    return SSCAN_ERR_CUDA;
}

cudaError_t launch_fwd(bool f32, const FwdParams& p, Shape sh, long long grid, cudaStream_t st) {
    if (grid <= 0) return cudaSuccess;
    ++g_rec.launches;
    return sscan::fwd_launch(f32, p, sh, (int)grid, st);
}
cudaError_t launch_fwd_tma(bool f32, const FwdParams& p, Shape sh, long long grid, cudaStream_t st) {
    if (grid <= 0) return cudaSuccess;
    ++g_rec.launches;
    return sscan::fwd_tma_launch(f32, p, sh, (int)grid, st);
}
cudaError_t launch_fwd_shfl(bool f32, const FwdParams& p, Shape sh, long long grid, cudaStream_t st) {
    if (grid <= 0) return cudaSuccess;
    ++g_rec.launches;
    return sscan::fwd_shfl_launch(f32, p, sh, (int)grid, st);
}
cudaError_t launch_fold(const FwdParams& p, cudaStream_t st) {
    ++g_rec.launches;
    return sscan::fwd_fold_launch(p, st);
}

// Device status word of the kernels' bounded waits (SSCAN_OK or
// SSCAN_ERR_TIMEOUT), one per device; read and cleared by sscan_get_last_error.
__device__ int g_device_status = 0;

// Its device address on the current device (looked up once per device; the
// lookup may load the module, so a first call should precede stream capture).
int* device_status_ptr() {
    static std::atomic<int*> cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    int* v = cached[dev].load(std::memory_order_acquire);
    if (v == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return nullptr;
        v = static_cast<int*>(ptr);
        cached[dev].store(v, std::memory_order_release);
    }
    return v;
}

}  // namespace

namespace sscan {

// The default stream-ordered pool returns its memory to the driver whenever
// the host synchronises, and the next allocation maps it again (measured on
// GB300: 80-125 us added to the first call after a synchronisation); this
// pool keeps what it holds up to kScratchRetainBytes.
cudaError_t scratch_alloc(void** ptr, size_t bytes, cudaStream_t stream) {
    static std::mutex mu;
    static cudaMemPool_t pools[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaMemPool_t pool = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (pools[dev & 63] == nullptr) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            cudaMemPool_t created = nullptr;
            e = cudaMemPoolCreate(&created, &props);
            if (e != cudaSuccess) return e;
            unsigned long long keep = kScratchRetainBytes;
            e = cudaMemPoolSetAttribute(created, cudaMemPoolAttrReleaseThreshold, &keep);
            if (e != cudaSuccess) {
                cudaMemPoolDestroy(created);
                return e;
            }
            pools[dev & 63] = created;
        }
        pool = pools[dev & 63];
    }
    return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

// Call record of an entry point defined in another translation unit.
void record_call(int launches, cudaStream_t stream, const char* plan) {
    g_rec.launches = launches;
    g_rec.stream = stream;
    snprintf(g_rec.plan, sizeof(g_rec.plan), "%s", plan);
}
void record_error(cudaError_t e) { fail_cuda(e); }
// The device status word of the current device (nullptr if it cannot be
// found); looking it up allocates nothing.
int* device_status_word() { return device_status_ptr(); }

// Warps per SM the automatic plan aims for when it splits time: about three
// per scheduler, enough to cover the FMA/MUFU and shared-memory latencies of
// the scan loop.
#ifndef SSCAN_TARGET_WARPS
#define SSCAN_TARGET_WARPS 12
#endif
constexpr long long kTargetWarpsPerSm = SSCAN_TARGET_WARPS;
// Shortest automatic segment, in chunks (cp.async kernel, TMA kernel).
constexpr long long kMinSegmentChunks = 8;
constexpr long long kMinTmaSegmentChunks = 13;

// Automatic shape per state count, measured on GB300: two or four states per
// lane and one channel per lane keep the most warps in flight, which the
// exponent-bound general case needs; wide states (N > 32) prefer 16 states x 2
// channels per lane (B/C reuse across channels) when that still gives 3 warps
// per SM.
struct ShapePref {
    long long max_n;
    Shape sh;
    long long min_warps_per_sm;
};
constexpr ShapePref kPrefs[] = {
    {4, {1, 4, 1}, 0},  {8, {2, 4, 1}, 0},  {16, {8, 2, 1}, 0},
    {32, {8, 4, 1}, 0}, {64, {4, 16, 2}, 3}, {64, {8, 8, 1}, 0},
};

// Resident CTAs per SM of a shape, queried once per device.
int cached_occupancy(bool f32, Shape sh) {
    constexpr int kNumShapes = (int)(sizeof(kShapes) / sizeof(kShapes[0]));
    static std::atomic<int> cache[64][2][kNumShapes] = {};  // host threads may race
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int idx = 0;
    while (idx < kNumShapes &&
           !(kShapes[idx].P == sh.P && kShapes[idx].NS == sh.NS && kShapes[idx].CPL == sh.CPL))
        ++idx;
    if (idx == kNumShapes) return 0;
    std::atomic<int>& c = cache[dev & 63][f32 ? 0 : 1][idx];
    int v = c.load(std::memory_order_relaxed);
    if (v == 0) {
        v = fwd_occupancy(f32, sh);
        c.store(v, std::memory_order_relaxed);
    }
    return v;
}

int plan_fwd(bool f32, long long batch, long long dim, long long seqlen, long long N, int segments,
             int lanes, long long max_segments, FwdPlan* out) {
    const int nsm = std::max(sm_count(), 1);
    Shape chosen{0, 0, 0};
    if (lanes == 0) {
        for (const ShapePref& pr : kPrefs) {
            if (N > pr.max_n) continue;
            const long long warps = batch * ceil_div(dim, shape_channels(pr.sh)) * shape_warps(pr.sh);
            if (warps >= pr.min_warps_per_sm * nsm) {
                chosen = pr.sh;
                break;
            }
        }
    } else {
        // the compiled shape with P = lanes and the fewest state slots >= N
        for (const Shape& c : kShapes)
            if (c.P == lanes && (long long)c.NS * c.P >= N &&
                (chosen.P == 0 || c.NS * c.P < chosen.NS * chosen.P))
                chosen = c;
    }
    auto warps_of = [&](Shape c) { return batch * ceil_div(dim, shape_channels(c)) * shape_warps(c); };
    auto target_of = [&](Shape c) {
        return std::min((long long)nsm * std::max(cached_occupancy(f32, c), 1) * shape_warps(c),
                        (long long)nsm * kTargetWarpsPerSm);
    };
    // When so few channels that the sequence must be cut into many segments
    // (12 or more), two channels per lane halve the shared-memory traffic per
    // element for B and C; the extra segments they need cost less (measured on
    // 512 channels x 8192 steps).
    if (lanes == 0 && chosen.P != 0 && chosen.CPL == 1 && segments == 0) {
        const long long w1 = warps_of(chosen), t1 = target_of(chosen);
        if (w1 < t1 && ceil_div(t1, std::max(w1, 1LL)) >= 12) {
            for (const Shape& c : kShapes)
                if (c.P == chosen.P && c.NS == chosen.NS && c.CPL == 2) {
                    chosen = c;
                    break;
                }
        }
    }
    const long long chosen_warps = chosen.P == 0 ? 0 : warps_of(chosen);
    const long long target = chosen.P == 0 ? 0 : target_of(chosen);
    if (chosen.P == 0) return SSCAN_ERR_INVALID;
    const long long DT = shape_channels(chosen);
    const long long TC = kChunkSteps;
    FwdPlan pl;
    pl.sh = chosen;
    pl.tiles_per_batch = ceil_div(dim, DT);
    pl.tiles = batch * pl.tiles_per_batch;
    if (pl.tiles > (1LL << 30)) return SSCAN_ERR_INVALID;
    long long S = segments;
    if (S == 0) {
        // a grid within a quarter of the target runs unsplit: a second wave
        // or a carry correction costs more than the missing warps (bf16
        // 8192 channels x 4096 steps x 64 states: 605 us unsplit, 653 us in
        // two segments)
        S = 4 * chosen_warps >= 3 * target ? 1 : ceil_div(target, std::max(chosen_warps, 1LL));
        S = std::min(S, std::max(1LL, seqlen / (kMinSegmentChunks * TC)));
        S = std::min(S, std::max(1LL, max_segments));
    }
    S = std::max(1LL, std::min(S, ceil_div(seqlen, TC)));
    pl.Tseg = ceil_div(ceil_div(seqlen, S), TC) * TC;
    pl.S = ceil_div(seqlen, pl.Tseg);
    if (pl.tiles * pl.S > (1LL << 30)) return SSCAN_ERR_INVALID;
    pl.tma = false;
    pl.shfl = false;
    pl.corr_sh = pl.sh;
    pl.corr_tma = false;
    pl.corr_shfl = false;
    pl.corr_tiles_per_batch = pl.tiles_per_batch;
    pl.corr_tiles = pl.tiles;
    *out = pl;
    return SSCAN_OK;
}

void choose_correction(FwdPlan& best, bool wide, long long batch, long long dim);

// Resident CTAs per SM of a TMA-kernel shape, queried once per device.
int cached_tma_occupancy(bool f32, Shape sh, int variant) {
    static std::atomic<int> cache[64][2][3][3] = {};  // device, dtype, (8,2,2) / (4,4,2) / (4,16,2), variant
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::atomic<int>& c = cache[dev & 63][f32 ? 0 : 1][sh.P == 8 ? 0 : sh.NS == 4 ? 1 : 2][variant % 3];
    int v = c.load(std::memory_order_relaxed);
    if (v == 0) {
        v = fwd_tma_occupancy(f32, sh, variant);
        c.store(v, std::memory_order_relaxed);
    }
    return v;
}

// Plan of the TMA-fed kernel for 8 < N <= 16 (shapes of 16 state slots) or
// 32 < N <= 64 (shape (4,16,2), 64 slots), or SSCAN_ERR_INVALID when it does
// not apply.  A time split fills at most one wave of the GPU's resident CTA
// slots and keeps segments of about 14 chunks or more: every segment beyond
// the first adds a carry correction over the decay horizon of its entry state
// (a few chunks for typical step sizes), so shorter segments cost more in
// corrections than they gain in local-pass parallelism (measured on GB300 with
// 512 channels x 8192 steps: 16, 19, 21 and 23 segments 48.8, 46.1, 52.8 and
// 56.4 us; 1536 x 65536: 16, 19, 22 and 25 segments 576, 501, 731 and 615
// us).  A problem wide enough to give (4,4,2), else (8,2,2), 6 warps per SM
// runs unsplit on that shape (8192 fp32 channels x 2048 steps:
// (8,2,2) unsplit 123 us, (4,4,2) in 2 or 3 segments 130 / 148 us; 16384
// channels: (4,4,2) unsplit 187 us, (8,2,2) 207 us).
// Otherwise the shape is the one with the most channels per lane whose
// segments stay at least 16 chunks long ((4,4,2)), else (8,2,2).  The
// carry correction's shape is chosen below.
int plan_fwd_tma(bool f32, int variant, long long batch, long long dim, long long seqlen, long long N,
                 int segments, int lanes, FwdPlan* out) {
    if (N <= 8 || N > 64 || (N > 16 && N <= 32)) return SSCAN_ERR_INVALID;
    const bool wide = N > 32;  // 64 state slots: shape (4,16,2)
    const int nsm = std::max(sm_count(), 1);
    const long long TC = kChunkSteps;
    const Shape cands[] = {wide ? Shape{4, 16, 2} : Shape{4, 4, 2}, {8, 2, 2}};
    const long long min_chunks[] = {wide ? 0 : 16, 0};
    // warps per SM that an unsplit launch must give to be taken as it is
    const long long min_warps[] = {6, 6};
    // without a pinned plan, the first candidate whose unsplit grid is wide
    // enough runs unsplit (a split adds carry corrections whose horizon grows
    // with slow decays)
    int unsplit = -1;
    if (segments == 0)
        for (int i = 0; i < (wide ? 1 : 2) && unsplit < 0; ++i) {
            const Shape sh = cands[i];
            if (lanes != 0 && lanes != sh.P) continue;
            if (batch * ceil_div(dim, tma_channels(sh)) * 4 >= min_warps[i] * nsm) unsplit = i;
        }
    FwdPlan best{};
    bool found = false;
    for (int i = 0; i < (wide ? 1 : 2) && !found; ++i) {
        const Shape sh = cands[i];
        if (!tma_has_shape(sh) || (lanes != 0 && lanes != sh.P)) continue;
        if (unsplit >= 0 && i != unsplit) continue;
        FwdPlan pl{};
        pl.sh = sh;
        pl.tma = true;
        pl.tiles_per_batch = ceil_div(dim, tma_channels(sh));
        pl.tiles = batch * pl.tiles_per_batch;
        if (pl.tiles > (1LL << 30)) return SSCAN_ERR_INVALID;
        const long long slots = (long long)nsm * std::max(cached_tma_occupancy(f32, sh, variant), 1);
        long long S = segments;
        if (S == 0 && unsplit >= 0) {
            S = 1;
        } else if (S == 0) {
            S = pl.tiles >= slots ? 1 : slots / pl.tiles;
            S = std::min(S, std::max(1LL, seqlen / (kMinTmaSegmentChunks * TC)));
        }
        S = std::max(1LL, std::min(S, ceil_div(seqlen, TC)));
        pl.Tseg = ceil_div(ceil_div(seqlen, S), TC) * TC;
        pl.S = ceil_div(seqlen, pl.Tseg);
        if (pl.tiles * pl.S > (1LL << 30)) return SSCAN_ERR_INVALID;
        const bool last = i == (wide ? 0 : 1) || lanes != 0 || segments != 0;
        if (pl.S == 1 || pl.Tseg >= min_chunks[i] * TC || last) {
            best = pl;
            found = true;
        }
    }
    if (!found) return SSCAN_ERR_INVALID;
    best.shfl = false;
    choose_correction(best, wide, batch, dim);
    if (best.corr_tiles * best.S > (1LL << 30)) return SSCAN_ERR_INVALID;
    *out = best;
    return SSCAN_OK;
}

// The carry correction of a TMA-fed plan: for long segments (long sequences,
// where long memories make long decay horizons) on the TMA-fed kernel, shape
// (4,4,2); for short ones, and for 64 state slots, on the cp.async kernel,
// shapes (8,2,1) and (8,8,1), whose smaller CTAs start and stop sooner.
void choose_correction(FwdPlan& best, bool wide, long long batch, long long dim) {
    const long long TC = kChunkSteps;
    // measured on GB300: 512 channels x 8192 steps in 19 segments 47.1 / 49.2 /
    // 53.2 us with (8,2,1) / TMA (8,2,2) / TMA (4,4,2), and 46.9 / 49.0 / 51.0 us
    // with (8,2,1) / (4,4,1) / (2,8,1), whose fewer lanes per channel let
    // decayed states drop out sooner but give fewer warps; 1536 x 65536 in 19
    // segments 554 / 548 / 509 us with the first three, 531 / 557 us with
    // (4,4,1) / (2,8,1).  64 state slots (8 x 1024 channels x 4096 steps in 2
    // segments): 449 us with TMA (4,16,2), whose 128 CTAs leave a sixth of
    // the SMs idle, 427 / 426 us with cp.async (8,8,1) / (16,4,1)
    best.corr_tma = best.S > 1 && !wide && best.Tseg >= 32 * TC;
    best.corr_sh = wide ? Shape{8, 8, 1} : best.corr_tma ? Shape{4, 4, 2} : Shape{8, 2, 1};
    best.corr_tiles_per_batch = ceil_div(dim, best.corr_tma ? tma_channels(best.corr_sh) : shape_channels(best.corr_sh));
    best.corr_tiles = batch * best.corr_tiles_per_batch;
    best.corr_shfl = false;
}

// Resident CTAs per SM of a shuffle-kernel shape, queried once per device.
int cached_shfl_occupancy(bool f32, Shape sh) {
    static std::atomic<int> cache[64][2] = {};  // device, dtype
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::atomic<int>& c = cache[dev & 63][f32 ? 0 : 1];
    int v = c.load(std::memory_order_relaxed);
    if (v == 0) {
        v = fwd_shfl_occupancy(f32, sh);
        c.store(v, std::memory_order_relaxed);
    }
    return v;
}

// Shortest segment of an automatic plan that takes the shuffle kernel in a
// time split (measured on GB300: 1536 channels x 65536 steps in 25 segments of
// 2624 steps 467 us against 510 us on (4,4,2); 512 channels x 8192 steps in
// 64 segments of 128 steps 55 us against 46 us on (8,2,2)).
constexpr long long kShflMinAutoSegmentSteps = 1024;

// Shortest automatic segment of a shuffle plan, in chunks.
#ifndef SSCAN_MIN_SHFL_SEGMENT_CHUNKS
#define SSCAN_MIN_SHFL_SEGMENT_CHUNKS 2
#endif
constexpr long long kMinShflSegmentChunks = SSCAN_MIN_SHFL_SEGMENT_CHUNKS;

// Plan of the shuffle variant of the TMA-fed kernel (plain scan).  Its lanes
// hold two channels of 8 states each, so a problem has a quarter of the lanes
// of the (8,2,2) shape: a time split fills one wave of the GPU's resident CTA
// slots (each segment beyond the first adds a carry correction over the decay
// horizon of its entry state).
int plan_fwd_shfl(bool f32, long long batch, long long dim, long long seqlen, long long N, int segments,
                  int lanes, long long max_segments, FwdPlan* out) {
    if (N <= 8 || N > 16) return SSCAN_ERR_INVALID;
    const Shape sh{2, 8, 2};
    if (!shfl_has_shape(sh) || (lanes != 0 && lanes != sh.P)) return SSCAN_ERR_INVALID;
    const int nsm = std::max(sm_count(), 1);
    const long long TC = kChunkSteps;
    FwdPlan pl{};
    pl.sh = sh;
    pl.tma = true;
    pl.shfl = true;
    pl.tiles_per_batch = ceil_div(dim, tma_channels(sh));
    pl.tiles = batch * pl.tiles_per_batch;
    if (pl.tiles > (1LL << 30)) return SSCAN_ERR_INVALID;
    const long long slots = (long long)nsm * std::max(cached_shfl_occupancy(f32, sh), 1);
    long long S = segments;
    if (S == 0) {
        S = pl.tiles >= slots ? 1 : slots / pl.tiles;
        S = std::min(S, std::max(1LL, seqlen / (kMinShflSegmentChunks * TC)));
        S = std::min(S, std::max(1LL, max_segments));
    }
    S = std::max(1LL, std::min(S, ceil_div(seqlen, TC)));
    pl.Tseg = ceil_div(ceil_div(seqlen, S), TC) * TC;
    pl.S = ceil_div(seqlen, pl.Tseg);
    if (pl.tiles * pl.S > (1LL << 30)) return SSCAN_ERR_INVALID;
    // the correction runs on the same kernel's correction instantiation, with
    // one channel per lane: twice the warps of the local pass's shape, so that
    // its latency-bound chunks overlap more (1536 channels x 65536 steps in 25
    // segments: correction 105.6 -> 99 us)
    pl.corr_tma = pl.S > 1;
    pl.corr_shfl = pl.S > 1;
    pl.corr_sh = Shape{2, 8, 1};
    pl.corr_tiles_per_batch = ceil_div(dim, tma_channels(pl.corr_sh));
    pl.corr_tiles = batch * pl.corr_tiles_per_batch;
    *out = pl;
    return SSCAN_OK;
}
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

void sscan_debug_expire_next_wait(unsigned int wait_limit_us) { g_expire_wait_us = wait_limit_us; }
void sscan_debug_expire_next_correction_wait(unsigned int wait_limit_us) { g_expire_corr_us = wait_limit_us; }

int sscan_last_launch_count(void) { return g_rec.launches; }

const char* sscan_last_plan(void) { return g_rec.plan; }

int sscan_get_last_error(void) {
    int status = g_rec.pending_error;
    cudaError_t e = cudaStreamSynchronize(g_rec.stream);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) {  // a bounded wait that gave up on this device
        int dev_status = SSCAN_OK;
        e = cudaMemcpyFromSymbol(&dev_status, g_device_status, sizeof(int));
        if (e == cudaSuccess && dev_status != SSCAN_OK) {
            const int zero = SSCAN_OK;
            e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
            if (status == SSCAN_OK) status = dev_status;
        }
    }
    if (e != cudaSuccess && status == SSCAN_OK) status = SSCAN_ERR_CUDA;
    g_rec.pending_error = SSCAN_OK;
    return status;
}

int sscan_fwd_fused(const void* u, const void* delta, const float* A, const void* B, const void* C,
                    const float* D, const void* z, const float* delta_bias, const float* h0, void* out,
                    float* final_state, int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                    int dtype, int flags, int segments, int lanes, void* stream) {
    g_rec.launches = 0;
    snprintf(g_rec.plan, sizeof(g_rec.plan), "rejected");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    g_rec.stream = st;
    if (dtype != SSCAN_F32 && dtype != SSCAN_BF16) return SSCAN_ERR_INVALID;
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1 || dstate > sscan::kMaxDstate)
        return SSCAN_ERR_INVALID;
    if (segments < 0 || lanes < 0) return SSCAN_ERR_INVALID;
    if (flags & ~(SSCAN_DELTA_SOFTPLUS | SSCAN_ZOH)) return SSCAN_ERR_INVALID;
    // every element index of every array must fit comfortably in int64 and
    // every grid in a 32-bit grid dimension
    const long long big = (long long)1 << 46;
    if (batch > big || dim > big || seqlen > big || (batch && dim > big / batch) ||
        (batch * dim && seqlen > big / (batch * dim)))
        return SSCAN_ERR_INVALID;
    // empty problems: arrays with no elements may be NULL
    if (batch == 0 || dim == 0) {
        snprintf(g_rec.plan, sizeof(g_rec.plan), "empty");
        return SSCAN_OK;
    }
    if (lanes != 0 && lanes != 1 && lanes != 2 && lanes != 4 && lanes != 8 && lanes != 16)
        return SSCAN_ERR_INVALID;
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

    const bool f32 = dtype == SSCAN_F32;
    const int esz = f32 ? 4 : 2;
    const int vece = 16 / esz;
    const bool vec = (seqlen % vece) == 0 && aligned16(u) && aligned16(delta) && aligned16(B) &&
                     aligned16(C) && aligned16(out) && (z == nullptr || aligned16(z));
    // the TMA-fed kernel takes the pass when the tensor-map rules hold
    // (16-byte aligned rows, coordinates below 2^31) and it has a shape for N
    const int variant = (flags & SSCAN_ZOH) ? 2 : (z != nullptr || delta_bias != nullptr || flags != 0) ? 1 : 0;
    const long long lim = (1LL << 31) - 256;
    sscan::FwdPlan pl;
    const bool tma_ok = vec && seqlen < lim && dim < lim && batch < lim;
    // the plain scan on the shuffle variant where it has a shape, else the
    // TMA-fed kernel's other shapes, else the cp.async kernel
    // (automatic plans: when it runs unsplit or in segments long enough that
    // the carry corrections stay a small part of the work; pinned plans: lanes
    // 2, or a pinned split with lanes 0)
    bool use_shfl = false;
    if (tma_ok && variant == 0 && (lanes == 0 || lanes == 2) &&
        sscan::plan_fwd_shfl(f32, batch, dim, seqlen, dstate, segments, lanes, 1LL << 40, &pl) == SSCAN_OK)
        use_shfl = lanes == 2 || segments != 0 || pl.S == 1 || pl.Tseg >= sscan::kShflMinAutoSegmentSteps;
    const bool use_tma = use_shfl || (tma_ok && sscan::plan_fwd_tma(f32, variant, batch, dim, seqlen, dstate,
                                                                    segments, lanes, &pl) == SSCAN_OK);
    if (!use_tma) {
        const int prc = sscan::plan_fwd(f32, batch, dim, seqlen, dstate, segments, lanes, 1LL << 40, &pl);
        if (prc != SSCAN_OK) return prc;
    }
    const Shape sh = pl.sh;
    const long long S = pl.S, tiles = pl.tiles;
    int* status = device_status_ptr();
    if (status == nullptr) return fail_cuda(cudaErrorInvalidDevicePointer);

    FwdParams p{};
    p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.h0 = h0;
    p.out = out; p.final_state = final_state;
    p.batch = batch; p.dim = dim; p.L = seqlen; p.N = dstate;
    p.Tseg = pl.Tseg; p.S = (int)S; p.tiles_per_batch = (int)pl.tiles_per_batch;
    p.vec = vec ? 1 : 0;
    p.z = z;
    p.delta_bias = delta_bias;
    p.delta_softplus = (flags & SSCAN_DELTA_SOFTPLUS) ? 1 : 0;
    p.zoh = (flags & SSCAN_ZOH) ? 1 : 0;
    p.status = status;
    // the test aids apply to the first pass, or to the carry correction, of
    // this call only
    const unsigned expire_us = g_expire_wait_us;
    g_expire_wait_us = 0;
    const unsigned expire_corr_us = g_expire_corr_us;
    g_expire_corr_us = 0;
    p.wait_ns = (unsigned long long)expire_us * 1000ull;
    p.expire_wait = expire_us != 0 ? 1 : 0;

    snprintf(g_rec.plan, sizeof(g_rec.plan),
             "sscan %s P=%d NS=%d CPL=%d vec=%d tiles=%lld S=%lld Tseg=%lld %s%s%s%s%s%s%s",
             f32 ? "f32" : "bf16", sh.P, sh.NS, sh.CPL, (int)vec, tiles, S, pl.Tseg,
             use_shfl ? "tma shfl " : use_tma ? "tma " : "",
             S == 1 ? "single" : S <= sscan::kFoldInCorrectionMaxSegments ? "local+correct" : "local+fold+correct",
             delta_bias ? " bias" : "",
             p.delta_softplus ? " softplus" : "", p.zoh ? " zoh" : "", z ? " gate" : "",
             S == 1 ? "" : pl.corr_shfl ? " corr=tma shfl" : pl.corr_tma ? " corr=tma" : " corr=cp.async");
    if (S > 1) {  // the correction's shape
        const size_t n = strlen(g_rec.plan);
        snprintf(g_rec.plan + n, sizeof(g_rec.plan) - n, "(%d,%d,%d)", pl.corr_sh.P, pl.corr_sh.NS,
                 pl.corr_sh.CPL);
    }

    cudaError_t e;
    if (S == 1) {
        p.mode = sscan::MODE_SINGLE;
        p.seg_count = 1;
        e = use_shfl  ? launch_fwd_shfl(f32, p, sh, tiles, st)
            : use_tma ? launch_fwd_tma(f32, p, sh, tiles, st)
                      : launch_fwd(f32, p, sh, tiles, st);
        if (e != cudaSuccess) return fail_cuda(e);
        return SSCAN_OK;
    }

    const size_t nseg = (size_t)(batch * dim) * (size_t)S;
    const size_t scratch_bytes = nseg * (size_t)sscan::split_floats_per_segment(dstate) * sizeof(float);
    void* scratch = nullptr;
    e = sscan::scratch_alloc(&scratch, scratch_bytes, st);
    if (e != cudaSuccess) return fail_cuda(e);
    p.seg_state = static_cast<float*>(scratch);
    p.seg_dsum = p.seg_state + nseg * (size_t)dstate;
    p.seg_dmin = p.seg_dsum + nseg;
    // pass 1: every segment from its local start, writing y and its aggregate;
    // pass 2 (more than kFoldInCorrectionMaxSegments segments): fold the
    // aggregates into the state entering each segment; pass 3: add the carried
    // state's decaying contribution (folding the aggregates itself when pass 2
    // did not run) and compose the final state
    // (bf16 outputs are rounded twice, the second time with the carry added)
    p.mode = sscan::MODE_LOCAL;
    p.seg_count = (int)S;
    e = use_shfl  ? launch_fwd_shfl(f32, p, sh, tiles * S, st)
        : use_tma ? launch_fwd_tma(f32, p, sh, tiles * S, st)
                  : launch_fwd(f32, p, sh, tiles * S, st);
    p.wait_ns = 0;
    p.expire_wait = 0;
    p.fold_in_corr = S <= sscan::kFoldInCorrectionMaxSegments ? 1 : 0;
    if (e == cudaSuccess && S > 2 && !p.fold_in_corr) e = launch_fold(p, st);
    if (e == cudaSuccess) {
        p.wait_ns = (unsigned long long)expire_corr_us * 1000ull;
        p.expire_wait = expire_corr_us != 0 ? 1 : 0;
        p.mode = sscan::MODE_CORR;
        p.seg_count = (int)(S - 1);
        p.tiles_per_batch = (int)pl.corr_tiles_per_batch;
        e = pl.corr_shfl  ? launch_fwd_shfl(f32, p, pl.corr_sh, pl.corr_tiles * (S - 1), st)
            : pl.corr_tma ? launch_fwd_tma(f32, p, pl.corr_sh, pl.corr_tiles * (S - 1), st)
                          : launch_fwd(f32, p, pl.corr_sh, pl.corr_tiles * (S - 1), st);
    }
    cudaError_t ef = cudaFreeAsync(scratch, st);
    if (e != cudaSuccess) return fail_cuda(e);
    if (ef != cudaSuccess) return fail_cuda(ef);
    return SSCAN_OK;
}

int sscan_fwd_ex(const void* u, const void* delta, const float* A, const void* B, const void* C,
                 const float* D, const float* h0, void* out, float* final_state, int64_t batch,
                 int64_t dim, int64_t seqlen, int64_t dstate, int dtype, int segments, int lanes,
                 void* stream) {
    return sscan_fwd_fused(u, delta, A, B, C, D, nullptr, nullptr, h0, out, final_state, batch, dim,
                           seqlen, dstate, dtype, 0, segments, lanes, stream);
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
    e = sscan::scratch_alloc(&scratch, (size_t)(rows * S) * 2 * sizeof(float), st);
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
