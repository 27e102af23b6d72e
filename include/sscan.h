/*
 * sscan.h -- C ABI of libsscan.so: the selective-scan forward pass and the
 * first-order linear-recurrence primitive on one GB300 (sm_103a).
 *
 * Every entry point takes plain pointers and sizes; no framework types cross
 * this boundary.  Device pointers are caller-owned (the library keeps none
 * after a call returns).  Calls are asynchronous on the caller's stream; the
 * return code reports argument validation and launch status only.  Kernel
 * faults surface through sscan_get_last_error() or any later synchronisation.
 *
 * Layouts are contiguous and row-major:
 *   u, delta, out        [batch, dim, seqlen]    (the I/O dtype)
 *   B, C                 [batch, dstate, seqlen] (the I/O dtype)
 *   A                    [dim, dstate]           float32
 *   D                    [dim]                   float32, may be NULL
 *   h0, final_state      [batch, dim, dstate]    float32, may be NULL
 */
#ifndef SSCAN_H
#define SSCAN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* I/O dtype of u, delta, B, C and out.  A, D, h0 and final_state are always
 * float32, and the state and every accumulation are float32 for both (the
 * pages keep the decay and state at full precision: "为什么Mamba的“并行扫描”不是真并行 (mhpq.cn/news/1057127)" section 4, pitfall 2; "并行扫描与硬件感知优化 (mhpq.cn/news/1077344)" page section 4.3). */
typedef enum { SSCAN_F32 = 0, SSCAN_BF16 = 1 } sscan_dtype;

/* Status codes.  No entry point aborts or throws. */
enum {
    SSCAN_OK = 0,
    SSCAN_ERR_INVALID = 1, /* a required pointer is NULL, a size is negative or
                              too large, dstate exceeds sscan_max_dstate(), or
                              dtype is unknown; nothing was launched          */
    SSCAN_ERR_CUDA = 2,    /* a CUDA call failed (launch, allocation, or an
                              asynchronous fault seen by sscan_get_last_error) */
    SSCAN_ERR_TIMEOUT = 3  /* a bounded device-side wait gave up; reported by
                              sscan_get_last_error()                          */
};

/*
 * sscan_fwd -- selective-scan forward pass, fused in one pass over HBM.
 *
 * Defined by the selective_scan pseudocode of "Mamba 状态空间模型：从理论到生产级推理的 CUDA 内核优化实战" (section
 * 2.3: discretise with A-bar = exp(delta*A), B-bar = delta*B; h = A-bar*h +
 * B-bar*x; y = C.h; plus D*x) and its PyTorch reference (section 7.1, which
 * also takes an initial state and returns the final state), and by the
 * mamba.py listing of "图解Blelloch并行扫描" (section 3.2).  For every batch b,
 * channel d and step t, with diagonal A:
 *
 *   h_t[n]   = exp(delta[b,d,t]*A[d,n]) * h_{t-1}[n] + delta[b,d,t]*B[b,n,t]*u[b,d,t]
 *   out[b,d,t] = sum_n C[b,n,t]*h_t[n] + D[d]*u[b,d,t]
 *
 * h_{-1} = h0[b,d,:] (zeros when h0 is NULL); final_state[b,d,:] = h after
 * the last step (not written when NULL).  delta is used as given (no
 * softplus is applied).  D == NULL means no skip term.
 *
 * u, delta, B, C, A: required device pointers.  out: required device pointer
 * (it must not alias any input).  batch, dim, seqlen >= 0 and
 * 1 <= dstate <= sscan_max_dstate(); a zero-sized problem returns SSCAN_OK
 * without launching (final_state, when given, then receives h0 or zeros if
 * seqlen == 0).  dtype: sscan_dtype.  stream: a cudaStream_t (NULL = legacy
 * default stream).
 *
 * Scratch: long sequences with few channels are split in time; the split
 * needs batch*dim*segments*(dstate+2) floats of scratch, taken stream-ordered
 * from the library's memory pool on the current device (which keeps up to
 * 1 GiB mapped while idle) and returned on the same stream.
 *
 * Time splits and the domain of delta: each segment after the first adds the
 * decaying contribution of its entry state to the outputs, and stops once
 * every carried state has decayed below 2^-24 of its entry magnitude.  That
 * cut-off is exact (to float32 rounding) while every decay factor
 * exp(delta*A) is at most 1, i.e. delta >= 0 (a step size, as softplus
 * produces) and A <= 0.  Rates A > 0 are always detected and the carries are
 * then followed to each segment's end; negative delta values lie outside the
 * stated domain (delta >= 0), but are detected the same way by every pass
 * except the 16-state-lane TMA-fed one (dstate > 32).
 */
int sscan_fwd(const void *u, const void *delta, const float *A, const void *B,
              const void *C, const float *D, const float *h0, void *out,
              float *final_state, int64_t batch, int64_t dim, int64_t seqlen,
              int64_t dstate, int dtype, void *stream);

/*
 * sscan_fwd_ex -- sscan_fwd with the launch plan pinned, for testing and
 * tuning.  segments: number of time segments per channel (0 = automatic; 1 =
 * no time split); lanes: lanes per channel sharing the state vector (0 =
 * automatic; 1, 2, 4, 8 or 16, subject to dstate <= 16*lanes; with 16-byte
 * aligned rows and 8 < dstate <= 16, lanes = 2 selects the kernel whose lanes
 * sum their partial outputs by shuffles).  Results are the same computation
 * under any plan (up to float32 rounding order).
 */
int sscan_fwd_ex(const void *u, const void *delta, const float *A, const void *B,
                 const void *C, const float *D, const float *h0, void *out,
                 float *final_state, int64_t batch, int64_t dim, int64_t seqlen,
                 int64_t dstate, int dtype, int segments, int lanes, void *stream);

/*
 * pscan -- first-order linear recurrence over rows, the pscan(a, b) primitive
 * that the mamba.py listing of "图解Blelloch并行扫描" (section 3.2) calls on
 * (deltaA, BX); with a = 1 it is the prefix sum of that page's section 1.1.
 *
 *   h[r,t] = a[r,t]*h[r,t-1] + b[r,t],   h[r,-1] = h0[r] (0 when h0 is NULL)
 *
 * a, b, h: device float32 [rows, len], required (h must not alias a or b);
 * h0: device float32 [rows] or NULL.  rows, len >= 0.  The result is the
 * same recurrence under any bracketing of the associative operator
 * (a1,b1) o (a2,b2) = (a2*a1, a2*b1 + b2) ("并行扫描与硬件感知优化 (mhpq.cn/news/1077344)" page, section
 * 2.2), up to float32 rounding order.
 */
int pscan(const float *a, const float *b, float *h, const float *h0,
          int64_t rows, int64_t len, void *stream);

/* Option bits of sscan_fwd_fused. */
#define SSCAN_DELTA_SOFTPLUS 1 /* delta <- softplus(delta (+ delta_bias)) inside the op */
#define SSCAN_ZOH 2            /* zero-order-hold B-bar instead of delta*B               */

/*
 * sscan_fwd_fused -- sscan_fwd with the options the pages attach to the scan,
 * each applied inside the same kernels (no extra pass over memory):
 *
 *   delta_bias [dim] float32 or NULL: delta <- delta + delta_bias[d];
 *   SSCAN_DELTA_SOFTPLUS: then delta <- softplus(delta) = log(1 + e^delta)
 *       (the F.softplus(delta) of the reference in "Mamba 状态空间模型：从理论到
 *       生产级推理的 CUDA 内核优化实战" section 7.1; delta = softplus(Linear(x))
 *       of its section 2.2);
 *   SSCAN_ZOH: B-bar = (delta*A)^-1 (exp(delta*A) - 1) delta*B, i.e. per state
 *       expm1(delta*A[d,n]) / A[d,n] * B (delta*B where A = 0): the
 *       zero-order-hold discretisation of that page's section 1.2;
 *   z [batch, dim, L] in the I/O dtype or NULL: out = (y + D*u) * silu(z),
 *       silu(z) = z / (1 + e^-z), the output gate (the sigmoid gate activation
 *       fused into the scan kernel on the "为什么Mamba的“并行扫描”不是真并行"
 *       page, section 2, taken as Mamba's SiLU gate).
 *
 * The final state is that of the scan (the gate does not touch it).  segments
 * and lanes pin the plan as in sscan_fwd_ex (0 = automatic).  Other arguments,
 * layouts, ownership and errors are those of sscan_fwd; unknown flag bits are
 * SSCAN_ERR_INVALID.
 */
int sscan_fwd_fused(const void *u, const void *delta, const float *A, const void *B,
                    const void *C, const float *D, const void *z, const float *delta_bias,
                    const float *h0, void *out, float *final_state, int64_t batch, int64_t dim,
                    int64_t seqlen, int64_t dstate, int dtype, int flags, int segments, int lanes,
                    void *stream);

/*
 * sscan_bwd -- gradients of sscan_fwd (no options), the backward pass with the
 * chunk-boundary recompute of "并行扫描与硬件感知优化 (mhpq.cn/news/1077344)"
 * section 3.3: the state at every 16-step boundary is kept in library scratch
 * (batch*dim*ceil(L/16)*N floats, stream-ordered), and each chunk's states are
 * recomputed from it during the reverse sweep.  For upstream gradients
 * dy = dL/dy and dfinal_state = dL/d(final state) (a_t = exp(delta_t*A[d,n])):
 *
 *   g_t      = C_t*dy_t + a_{t+1}*g_{t+1},  g_{L-1} = C*dy + dfinal_state
 *   ddelta_t = sum_n g_t*(h_{t-1}*a_t*A + u_t*B_t)
 *   du_t     = sum_n g_t*delta_t*B_t + D*dy_t
 *   dB[b,n,t] = sum_d g_t*delta_t*u_t,  dC[b,n,t] = sum_d dy_t*h_t
 *   dA[d,n]   = sum_{b,t} g_t*h_{t-1}*a_t*delta_t,  dD[d] = sum_{b,t} dy_t*u_t
 *   dh0       = a_0*g_0
 *
 * Inputs are those of sscan_fwd plus dy [batch, dim, L] (I/O dtype) and
 * dfinal_state [batch, dim, N] float32 or NULL (zero).  Outputs (device,
 * caller-owned, overwritten): du, ddelta [batch, dim, L] in the I/O dtype;
 * dA [dim, N], dB and dC [batch, N, L] float32; dD [dim] float32 (ignored when
 * D is NULL; may be NULL); dh0 [batch, dim, N] float32 or NULL.  dA, dB, dC and
 * dD are sums over channels or batches accumulated with float atomics, so
 * their rounding order is not fixed.  Errors as sscan_fwd.
 */
int sscan_bwd(const void *u, const void *delta, const float *A, const void *B, const void *C,
              const float *D, const float *h0, const void *dy, const float *dfinal_state,
              void *du, void *ddelta, float *dA, float *dB, float *dC, float *dD, float *dh0,
              int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int dtype, void *stream);

/*
 * sscan_step -- one autoregressive decode step: advance the cached state of
 * every (batch, channel) by one token and read it out (the recurrent
 * inference step whose state cache "Mamba 状态空间模型：从理论到生产级推理的
 * CUDA 内核优化实战" describes in section 5.1):
 *
 *   state[b,d,n] <- exp(delta[b,d]*A[d,n])*state[b,d,n] + delta[b,d]*B[b,n]*u[b,d]
 *   out[b,d]      = sum_n C[b,n]*state[b,d,n] + D[d]*u[b,d]    (the updated state)
 *
 * It equals sscan_fwd with seqlen = 1, h0 = state and final_state = state.
 * u, delta, out: [batch, dim] in the I/O dtype; A [dim, N] float32; B, C
 * [batch, N] in the I/O dtype; D [dim] float32 or NULL; state [batch, dim, N]
 * float32, updated in place.  All are device pointers; state must not alias
 * any other argument.  Returns SSCAN_OK, SSCAN_ERR_INVALID (missing pointer,
 * bad size or dtype, N > sscan_max_dstate()) or SSCAN_ERR_CUDA (launch).
 */
int sscan_step(const void *u, const void *delta, const float *A, const void *B,
               const void *C, const float *D, float *state, void *out, int64_t batch,
               int64_t dim, int64_t dstate, int dtype, void *stream);

/* Bytes of device memory that sscan_fwd_noalloc keeps, per GPU, for the
 * carry of time-split launches (a fixed array, held until the process exits). */
#define SSCAN_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * sscan_fwd_noalloc -- sscan_fwd for callers that cannot allocate device
 * memory while they run.  The pages have no counterpart: this is a deployment
 * variant of the same computation.
 *
 * Some callers must never allocate on their execution path -- an inference
 * engine's per-request plugin hook running under a fixed memory budget, a
 * real-time loop in which an allocation could synchronise the device or wait
 * on the allocator, a runtime that hands out all memory up front.  sscan_fwd
 * takes the scratch of a time-split launch from a stream-ordered pool;
 * this entry point keeps that scratch in a fixed device array of
 * SSCAN_NOALLOC_SCRATCH_BYTES instead and calls no allocating routine.  The
 * caller still passes every input and output.
 *
 * Arguments are those of sscan_fwd plus segments: 0 picks the time split
 * automatically, shrunk so that its carry (batch*dim*segments*(dstate+2)
 * floats) fits the array; a positive value pins it, and a pinned split whose
 * carry does not fit is rejected with SSCAN_ERR_INVALID before anything is
 * launched.  The passes run on the library's cp.async-fed kernels (the
 * general path of sscan_fwd, whatever the row alignment), so the results
 * agree with sscan_fwd's up to float32 rounding order, and within the same
 * tolerances against the definition.
 *
 * The first call on each device looks up the array's address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  All calls share the array and each
 * call writes everything it reads from it, so no clearing is needed, but
 * calls whose kernels may overlap on the GPU (unordered streams) race on it.
 * sscan_last_launch_count() and sscan_last_plan() describe these calls too.
 */
int sscan_fwd_noalloc(const void *u, const void *delta, const float *A, const void *B,
                      const void *C, const float *D, const float *h0, void *out,
                      float *final_state, int64_t batch, int64_t dim, int64_t seqlen,
                      int64_t dstate, int dtype, int segments, void *stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char *sscan_status_string(int status);

/* Synchronises the stream of this thread's last call and reports any
 * asynchronous failure since: SSCAN_OK, SSCAN_ERR_CUDA or SSCAN_ERR_TIMEOUT.
 * Clears the recorded error. */
int sscan_get_last_error(void);

/*
 * sscan_debug_expire_next_wait -- a test aid for the timeout path of the
 * error contract above; the pages have no counterpart.  It arms the calling
 * thread's next sscan_fwd / sscan_fwd_ex / sscan_fwd_fused call.  If that
 * call's first pass runs on the TMA-fed kernels (16-byte aligned rows and a
 * dstate they serve), the barrier of the first B/C ring stage of each of its
 * CTAs is made to expect 16 bytes that no copy delivers, and every bounded
 * wait of that pass gives up after wait_limit_us microseconds (instead of
 * about a second).  The waits on that stage then run out as a real stall
 * would: the kernel waits (bounded) for the copies it still has in flight,
 * records SSCAN_ERR_TIMEOUT in the device status word and ends, and
 * sscan_get_last_error() reports SSCAN_ERR_TIMEOUT.  No fault is involved and
 * the context stays usable; the outputs of that call are undefined.  The
 * next call consumes the setting whichever kernel it runs; 0 disarms it.
 */
void sscan_debug_expire_next_wait(unsigned int wait_limit_us);

/*
 * sscan_debug_expire_next_correction_wait -- the same test aid for the carry
 * correction of a time split; the pages have no counterpart.  It arms the
 * calling thread's next sscan_fwd / sscan_fwd_ex / sscan_fwd_fused call: if
 * that call splits time and its correction runs on the TMA-fed kernels, one
 * ring stage of each correction CTA (the first B/C stage, or the first warp's
 * first stage where the warps stage C themselves) is made to expect 16 bytes
 * that no copy delivers, and the correction's bounded waits give up after
 * wait_limit_us microseconds; the outcome is as above (SSCAN_ERR_TIMEOUT,
 * outputs undefined, context usable).  The next call consumes the setting
 * whichever plan it runs; 0 disarms it.
 */
void sscan_debug_expire_next_correction_wait(unsigned int wait_limit_us);

/*
 * sscan_probe_ex2 -- a measurement aid for the roofline of the scan; the
 * pages have no counterpart.  It launches `blocks` CTAs of 256 threads on
 * `stream`, each thread running 16 independent chains of `iters` exponentials
 * 2^x on the MUFU unit -- the operation every element of the scan takes (one
 * per channel and step for a channel with a single rate).  Timing the launch
 * with CUDA events and dividing sscan_probe_ex2_count(blocks, iters) by the
 * time gives the unit's throughput on this GPU.  sink: device float32
 * [blocks*256], required (it keeps the work alive and is not written in
 * practice).  Returns SSCAN_OK, SSCAN_ERR_INVALID (sink NULL, blocks or iters
 * < 1) or SSCAN_ERR_CUDA (launch failure).
 */
int sscan_probe_ex2(float *sink, int blocks, int iters, void *stream);
/* Exponentials one sscan_probe_ex2 launch computes. */
long long sscan_probe_ex2_count(int blocks, int iters);

/*
 * sscan_probe_element -- a measurement aid for the roofline of the scan; the
 * pages have no counterpart.  It launches `blocks` CTAs of 256 threads on
 * `stream` (two resident per SM); each thread runs 16 independent state
 * chains (32 when shared_rate != 0) for `iters` steps of the element
 * arithmetic of "Mamba 状态空间模型：从理论到生产级推理的 CUDA 内核优化实战"
 * section 2.3: a = 2^(delta*A*log2 e), h = a*h + (delta*u)*B, y += C*h --
 * one exponent per element, or one per step shared by all chains when
 * shared_rate != 0 (a channel with a single decay rate).  Timing the launch
 * with CUDA events and dividing sscan_probe_element_count(blocks, iters,
 * shared_rate) by the time gives the peak element rate of the arithmetic on
 * this GPU: the exponent and the FP32 operations share the SMs' issue slots,
 * so it lies below both units' separate peaks.  sink: device float32
 * [blocks*256], required (not written in practice).  Returns SSCAN_OK,
 * SSCAN_ERR_INVALID (sink NULL, blocks or iters < 1) or SSCAN_ERR_CUDA.
 */
int sscan_probe_element(float *sink, int blocks, int iters, int shared_rate, void *stream);
/* Elements one sscan_probe_element launch computes. */
long long sscan_probe_element_count(int blocks, int iters, int shared_rate);

/* Largest dstate that sscan_fwd accepts. */
int sscan_max_dstate(void);

/* Number of kernels the calling thread's last sscan_fwd / pscan call
 * launched (0 for zero-sized problems or rejected calls). */
int sscan_last_launch_count(void);

/* Text description of the calling thread's last launch plan (kernel
 * variant, grid, segments, lanes); static per-thread storage. */
const char *sscan_last_plan(void);

#ifdef __cplusplus
}
#endif

#endif /* SSCAN_H */
