/*
 * evoattn.h -- C ABI of the GB300 (sm_103a) EvoAttention library.
 *
 * EvoAttention is the memory-efficient 3D attention over the 2D pair
 * representation that MegaFold calls EvoFlash-3D (MegaFold: Efficient
 * Training of Next-Generation 3D Attention Protein Models on Cross-Platform
 * GPUs; technical summary, "Methodik" section 1 "EvoFlash-3D": the logits are
 * produced tile by tile in on-chip memory with an online, numerically stable
 * softmax in both the forward and the backward pass, never materialising the
 * O(N^3) attention map in HBM, and carry an additively broadcast pair-bias
 * term).  Successive layers alternate the attention axis, row-wise then
 * column-wise (same page, "Methodik" section 2 "EvoSP-3D", Kommunikation);
 * the column-wise (ending-node) layer is expressed here as strides, not as a
 * copy.
 *
 * For every batch b, row s in [0,S) and head h, with query row j and key k in
 * [0,N) and feature d in [0,D):
 *
 *   x[j,k]   = sum_d q[b,s,h,j,d] k[b,s,h,k,d] / sqrt(D)
 *              + pair_bias[b,h,j,k] + (mask[b,s,k] ? 0 : -1e9)
 *   lse[j]   = log sum_k exp(x[j,k])                        (natural log)
 *   O[j,d]   = sum_k exp(x[j,k] - lse[j]) v[b,s,h,k,d]
 *   out      = sigmoid(gate) * O     (elementwise; out = O when gate is NULL)
 *
 * The pair bias is shared by all S rows (triangle attention around the
 * starting or ending node: S = N; MSA-row attention with pair bias: S = MSA
 * depth).  The backward returns dq, dk, dv, dgate and
 *
 *   dbias[b,h,j,k] = sum_s dlogits[b,s,h,j,k]
 *
 * CONVENTIONS (all entry points)
 *  - Ownership: the caller owns every buffer.  Device pointers point to
 *    device memory of the current CUDA device.  The library never allocates
 *    device memory at run time; what it holds is static: two 4-byte status
 *    words per device (see evoattn_get_device_status), the
 *    EVOATTN_NOALLOC_SCRATCH_BYTES array that only evoattn_bwd_noalloc uses
 *    (held on every device that loads the library until the process exits,
 *    shared by all calls of that entry point, which must be serialised), the
 *    cached driver entry point used to build tensor maps, and the settings of
 *    evoattn_debug_set_wait.
 *  - Execution: work is enqueued on `stream` (a cudaStream_t; 0 = legacy
 *    default stream) and the call returns without synchronising, except
 *    evoattn_get_device_status.  Calls on different streams may run
 *    concurrently when their outputs and workspaces do not overlap.
 *  - Errors: arguments are validated on the host before anything is
 *    enqueued; a failing call returns a non-zero evoattn_status and enqueues
 *    nothing.  A launch failure returns EVOATTN_ERR_CUDA.  The library never
 *    aborts the process.  Every wait inside a kernel is bounded (2 s by
 *    default); a kernel that gives up a wait stops every CTA of its own
 *    launch, leaves its outputs undefined and sets EVOATTN_ERR_TIMEOUT in the
 *    device status (evoattn_get_device_status).  Other launches, earlier or
 *    later, on any stream, are not affected.
 *  - Shapes: B, S, H, N >= 1.  BF16: D in {16, 32, 64} for the forward,
 *    {16, 32} for the backward (evoattn_bwd, evoattn_bwd_profiled and
 *    evoattn_bwd_noalloc return EVOATTN_ERR_UNSUPPORTED for BF16 D = 64, and
 *    evoattn_bwd_workspace_size returns 0).  F32: D in {16, 32, 64, 128}.
 *  - Strides are in ELEMENTS (not bytes), one per logical axis, for the
 *    logical shapes:  q/k/v/gate/out/dout/dq/dk/dv/dgate  [B,S,H,N,D]  as
 *    {b, s, h, n, d};  pair_bias [B,H,N,N] as {b, h, j, k};  mask [B,S,N] as
 *    {b, s, k}.  Any non-negative strides are accepted for F32.  For BF16 the
 *    d stride must be 1, every other stride of a [B,S,H,N,D] tensor a
 *    multiple of 8 elements (16 bytes), the base address 16-byte aligned;
 *    the pair bias needs a unit stride along k or along j and its other
 *    strides multiples of 8 elements.  Otherwise EVOATTN_ERR_ALIGNMENT.
 *  - mask is uint8, nonzero = keep; NULL means every key is kept.  A row
 *    whose keys are all masked yields a uniform softmax over its keys (every
 *    logit saturates at -1e9 in fp32).
 *  - The forward writes lse as fp32 [B,S,H,N] contiguous; the backward reads
 *    it in the same layout.
 *  - BF16 inputs produce BF16 out/dq/dk/dv/dgate; dbias and lse are always
 *    fp32.  F32 inputs produce F32 outputs.
 */
#ifndef EVOATTN_H
#define EVOATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EVOATTN_OK = 0,
    EVOATTN_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad flag */
    EVOATTN_ERR_UNSUPPORTED = 2,   /* D or dtype outside the supported set */
    EVOATTN_ERR_ALIGNMENT = 3,     /* stride / address rule of the BF16 path broken */
    EVOATTN_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than required */
    EVOATTN_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
    EVOATTN_ERR_TIMEOUT = 6        /* a kernel gave up a bounded wait (device status) */
} evoattn_status;

typedef enum { EVOATTN_BF16 = 0, EVOATTN_F32 = 1 } evoattn_dtype;

/* evoattn_bwd flags */
#define EVOATTN_DBIAS_DETERMINISTIC 0u  /* fixed s-slots + ordered sum: bit-identical */
#define EVOATTN_DBIAS_ATOMIC 1u         /* s-slot partials added with fp32 atomics */
#define EVOATTN_DQ_DETERMINISTIC 2u     /* per-key-tile dQ slices + ordered sum */
#define EVOATTN_DBIAS_FUSED 4u          /* dbias summed in the dK/dV pass (fp32 atomics) */

/*
 * Forward (MegaFold technical summary, "Methodik" section 1 "EvoFlash-3D",
 * Mechanismus and Optimierung).
 *
 *  q, k, v, gate : [B,S,H,N,D] device, dtype `dtype`; gate may be NULL.
 *  pair_bias     : [B,H,N,N] device, dtype `dtype` (indexed [b,h,j,k]).
 *  mask          : [B,S,N] device uint8 or NULL (then mask_strides is ignored).
 *  out           : [B,S,H,N,D] device, written.
 *  lse           : [B,S,H,N] device fp32 contiguous, written (natural log of
 *                  the softmax normaliser of each query row, as in x above).
 *  *_strides     : host arrays, element strides as in CONVENTIONS.
 * Returns EVOATTN_OK once the kernels are enqueued.
 */
evoattn_status evoattn_fwd(const void* q, const int64_t q_strides[5],
                           const void* k, const int64_t k_strides[5],
                           const void* v, const int64_t v_strides[5],
                           const void* pair_bias, const int64_t bias_strides[4],
                           const uint8_t* mask, const int64_t mask_strides[3],
                           const void* gate, const int64_t gate_strides[5],
                           void* out, const int64_t out_strides[5],
                           float* lse,
                           int B, int S, int H, int N, int D,
                           evoattn_dtype dtype, cudaStream_t stream);

/*
 * Bytes of device workspace evoattn_bwd needs for this problem (0 on invalid
 * sizes or flags).  Linear in B*S*H*N*D plus O(B*H*N*N) for the dbias
 * partial sums; never proportional to B*S*H*N*N -- except with
 * EVOATTN_DQ_DETERMINISTIC on the BF16 path, which adds ceil(N/128) - 1
 * further fp32 copies of dq (4 * B*S*H*N*D bytes each): the price of a fixed
 * summation order without giving up the load balance of the dK/dV kernel.
 */
size_t evoattn_bwd_workspace_size(int B, int S, int H, int N, int D,
                                  evoattn_dtype dtype, unsigned flags);

/*
 * Backward (same section: the logits are recomputed tile by tile in the
 * backward pass as well).
 *
 *  q..gate, pair_bias, mask : as passed to evoattn_fwd.
 *  out, lse                 : the forward's outputs for these inputs.
 *  dout                     : [B,S,H,N,D] device, gradient of the loss w.r.t. out.
 *  dq, dk, dv               : [B,S,H,N,D] device, written.
 *  dbias                    : [B,H,N,N] device fp32 contiguous, written (the
 *                             sum over s of the logit gradients).
 *  dgate                    : [B,S,H,N,D] device, written; must be NULL
 *                             exactly when gate is NULL.
 *  flags                    : EVOATTN_DBIAS_DETERMINISTIC (bit-identical
 *                             dbias from run to run and box to box) or
 *                             EVOATTN_DBIAS_ATOMIC (same partials combined
 *                             with atomics; order-dependent rounding), OR-ed
 *                             with EVOATTN_DQ_DETERMINISTIC to make dq
 *                             bit-identical too: by default the BF16 path
 *                             adds the dQ partial of every key tile into an
 *                             fp32 buffer with atomics (rounding depends on
 *                             their order); with the flag each key tile
 *                             stores its partial into a slice of its own
 *                             and the slices are summed in key-tile order
 *                             (workspace: ceil(N/128) fp32 copies of dq
 *                             instead of one).  EVOATTN_DBIAS_FUSED (BF16;
 *                             it overrides the two dbias modes above) adds
 *                             every logit gradient into dbias with fp32
 *                             atomics from the pass that computes dK and dV,
 *                             so the logits are recomputed once instead of
 *                             twice; order-dependent rounding, no slot
 *                             partials in the workspace.  dk, dv and dgate
 *                             are bit-identical in every mode; the F32 path
 *                             is deterministic whatever the flags.  Other
 *                             bits set: EVOATTN_ERR_INVALID_ARG.
 *  workspace                : device, 256-byte aligned, at least
 *                             evoattn_bwd_workspace_size(...) bytes; the
 *                             library overwrites it; it must not be used by
 *                             another call that runs concurrently.
 */
evoattn_status evoattn_bwd(const void* q, const int64_t q_strides[5],
                           const void* k, const int64_t k_strides[5],
                           const void* v, const int64_t v_strides[5],
                           const void* pair_bias, const int64_t bias_strides[4],
                           const uint8_t* mask, const int64_t mask_strides[3],
                           const void* gate, const int64_t gate_strides[5],
                           const void* out, const int64_t out_strides[5],
                           const float* lse,
                           const void* dout, const int64_t dout_strides[5],
                           void* dq, const int64_t dq_strides[5],
                           void* dk, const int64_t dk_strides[5],
                           void* dv, const int64_t dv_strides[5],
                           float* dbias,
                           void* dgate, const int64_t dgate_strides[5],
                           int B, int S, int H, int N, int D,
                           evoattn_dtype dtype, unsigned flags,
                           void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/*
 * Same as evoattn_bwd, and additionally records stage_events[0..4] on
 * `stream` around its kernels: [0] before the first kernel, [1] after the
 * per-row preprocessing (delta, dgate, gated output gradient), [2] after the
 * dK/dV kernel (which also accumulates dQ), [3] after the dbias kernel, [4]
 * after the final reductions (ordered dbias sum, dQ conversion).  The events
 * are created and owned by the caller (cudaEventCreate); elapsed times
 * between consecutive events are the stage durations.  stage_events may not
 * be NULL.  For profiling; the work done is identical to evoattn_bwd.
 */
evoattn_status evoattn_bwd_profiled(const void* q, const int64_t q_strides[5],
                                    const void* k, const int64_t k_strides[5],
                                    const void* v, const int64_t v_strides[5],
                                    const void* pair_bias, const int64_t bias_strides[4],
                                    const uint8_t* mask, const int64_t mask_strides[3],
                                    const void* gate, const int64_t gate_strides[5],
                                    const void* out, const int64_t out_strides[5],
                                    const float* lse,
                                    const void* dout, const int64_t dout_strides[5],
                                    void* dq, const int64_t dq_strides[5],
                                    void* dk, const int64_t dk_strides[5],
                                    void* dv, const int64_t dv_strides[5],
                                    float* dbias,
                                    void* dgate, const int64_t dgate_strides[5],
                                    int B, int S, int H, int N, int D,
                                    evoattn_dtype dtype, unsigned flags,
                                    void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream, cudaEvent_t stage_events[5]);

/*
 * Capacity in bytes of the library-owned scratch that evoattn_bwd_noalloc
 * uses in place of a caller workspace.
 */
#define EVOATTN_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * Backward for callers that cannot allocate device memory.  There is no
 * counterpart in the MegaFold paper; it is a deployment convenience.
 *
 * Some callers cannot hand the library a workspace: a plugin that runs inside
 * a host framework which owns every device allocation and gives its plugins no
 * allocator, or a latency-critical caller that must not call cudaMalloc
 * (which can synchronise the device) on its hot path.  This entry point does
 * the same work as evoattn_bwd with the same arguments, minus the workspace:
 * its scratch lives in one statically sized device array inside the library,
 * EVOATTN_NOALLOC_SCRATCH_BYTES large, which every GPU that loads the library
 * holds until the process exits.  It never calls cudaMalloc, cudaFree or any
 * allocating routine.
 *
 *  - Problems whose scratch need (evoattn_bwd_workspace_size for the same
 *    arguments) exceeds EVOATTN_NOALLOC_SCRATCH_BYTES are rejected with
 *    EVOATTN_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on a device looks up the device address of the scratch
 *    array (with that device current); make that first call before any stream
 *    capture begins.
 *  - Every call on a device shares the one array and leaves its contents
 *    behind; the kernels overwrite every scratch byte they later read, so
 *    nothing needs clearing between calls.  Calls whose work overlaps on the
 *    GPU (different streams, or different host threads without ordering)
 *    race on the array and give undefined results: serialise them.
 */
evoattn_status evoattn_bwd_noalloc(const void* q, const int64_t q_strides[5],
                                   const void* k, const int64_t k_strides[5],
                                   const void* v, const int64_t v_strides[5],
                                   const void* pair_bias, const int64_t bias_strides[4],
                                   const uint8_t* mask, const int64_t mask_strides[3],
                                   const void* gate, const int64_t gate_strides[5],
                                   const void* out, const int64_t out_strides[5],
                                   const float* lse,
                                   const void* dout, const int64_t dout_strides[5],
                                   void* dq, const int64_t dq_strides[5],
                                   void* dk, const int64_t dk_strides[5],
                                   void* dv, const int64_t dv_strides[5],
                                   float* dbias,
                                   void* dgate, const int64_t dgate_strides[5],
                                   int B, int S, int H, int N, int D,
                                   evoattn_dtype dtype, unsigned flags,
                                   cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the calling device's status
 * word.  *device_status receives EVOATTN_OK, or EVOATTN_ERR_TIMEOUT when a
 * kernel enqueued since the last read gave up a bounded wait (its outputs are
 * then undefined).  Returns EVOATTN_ERR_CUDA if synchronising or the copy
 * fails, EVOATTN_ERR_INVALID_ARG if device_status is NULL.
 */
evoattn_status evoattn_get_device_status(cudaStream_t stream, int* device_status);

/*
 * LayerNorm of the pair representation fused with the bias-free linear
 * projection that produces the queries, keys, values, gate and pair bias of
 * triangle attention (MegaFold technical summary, "Methodik" section 3
 * "EvoFusion", Umfang and Mechanismus: the normalised N x N x C tensor is not
 * written to HBM between normalisation and projection).  For every row
 * r = (b, i, j):
 *
 *   y[r, c]   = (z[r, c] - mean_c z[r, :]) / sqrt(var_c z[r, :] + eps)
 *               * gamma[c] + beta[c]      (var: mean squared deviation)
 *   out[r, o] = sum_c y[r, c] w[o, c]     (y rounded to bf16, fp32 sums)
 *   q[b, i, j, h, d] = out[r, h*D + d],          k: + H*D,  v: + 2*H*D,
 *   g[b, i, j, h, d] = out[r, 3*H*D + h*D + d],  pair_bias[b, h, i, j] = out[r, 4*H*D + h]
 *
 *  z          : [B, N, N, C] device bf16, dense (C contiguous), 16-byte aligned.
 *  gamma, beta: [C] device fp32.
 *  w          : [4*H*D + H, C] device bf16, dense row-major, 16-byte aligned.
 *  eps        : > 0, added to the variance.
 *  q, k, v, g : [B, N, N, H, D] device bf16, dense, 16-byte aligned, written
 *               (the pair projections in the layout the attention reads as
 *               starting- or ending-node views).
 *  pair_bias  : [B, H, N, N] device bf16, dense, written.
 * Supported: C = 128, H * D = 128, H <= 8, B * N * N < 2^31 - 128 (otherwise
 * EVOATTN_ERR_UNSUPPORTED).  g is the gate's pre-activation: the attention
 * applies the sigmoid.  Returns EVOATTN_OK once the kernel is enqueued.
 */
evoattn_status evoattn_ln_proj(const void* z, const float* gamma, const float* beta,
                               const void* w, float eps,
                               void* q, void* k, void* v, void* g, void* pair_bias,
                               int B, int N, int C, int H, int D, cudaStream_t stream);

/*
 * The operators that follow the gated attention in a pair-stack block, as one
 * fused operator (MegaFold technical summary, "Methodik" section 3
 * "EvoFusion", Umfang: layer normalisation, linear projections and SwiGLU
 * activations; Mechanismus: no intermediate N x N tensor is written to HBM
 * between them): the attention's output projection with its residual add
 * (when o is given), then the SwiGLU transition with its residual add.  For
 * every row r = (b, i, j), with F hidden units:
 *
 *   z1[r, c]  = z[r, c] + sum_e o[r, e] w_o[c, e]        (fp32; z1 = z without o)
 *   y[r, c]   = bf16((z1[r, c] - mean_c z1[r, :]) / sqrt(var_c z1[r, :] + eps)
 *                    * gamma[c] + beta[c])          (var: mean squared deviation)
 *   a[r, f]   = sum_c y[r, c] w1[f, c],   b[r, f] = sum_c y[r, c] w1[F + f, c]
 *   h[r, f]   = bf16(silu(a[r, f]) * b[r, f]),   silu(x) = x / (1 + exp(-x))
 *   out[r, c] = bf16(z1[r, c] + sum_f h[r, f] w2[c, f])    (fp32 sums)
 *
 *  z          : [B, N, N, C] device bf16, dense (C contiguous), 16-byte aligned.
 *  o          : [B, N, N, HD] device bf16, dense, 16-byte aligned: the gated
 *               attention output of the same rows (evoattn_fwd's out, stored
 *               with (b, i, j) outermost); NULL for the transition alone.
 *  w_o        : [C, HD] device bf16, dense row-major, 16-byte aligned; NULL
 *               exactly when o is NULL.
 *  gamma, beta: [C] device fp32.
 *  w1         : [2F, C] device bf16, dense row-major, 16-byte aligned (rows
 *               0..F-1 the SiLU branch, F..2F-1 the linear branch).
 *  w2         : [C, F] device bf16, dense row-major, 16-byte aligned.
 *  eps        : > 0, added to the variance.
 *  out        : [B, N, N, C] device bf16, dense, 16-byte aligned, written; it
 *               may not overlap z or o.
 * Supported: C = 128, HD = 128 (with o), F = 4C, B * N * N < 2^31 - 128
 * (otherwise EVOATTN_ERR_UNSUPPORTED).  Returns EVOATTN_OK once the kernel is
 * enqueued.
 */
evoattn_status evoattn_transition(const void* z, const void* o, const void* w_o,
                                  const float* gamma, const float* beta,
                                  const void* w1, const void* w2, float eps, void* out,
                                  int B, int N, int C, int HD, int F, cudaStream_t stream);

/*
 * Testing hook for the bounded-wait failure path; not needed in normal use.
 * Applies to every tcgen05 kernel enqueued after the call, on any device, by
 * any thread of the process.
 *
 *  limit_ns : limit of each pipeline wait inside the kernels (0 restores the
 *             default, 2 s).  The waits of a kernel's wind-down after a
 *             give-up (for its own copies and MMAs already in flight) keep
 *             the default limit.
 *  stall    : nonzero makes the compute warps' first wait in each such
 *             kernel wait for an event that nothing ever signals, so every
 *             CTA gives up after limit_ns, winds down and reports
 *             EVOATTN_ERR_TIMEOUT through evoattn_get_device_status; the
 *             outputs of those launches are undefined.  0 restores normal
 *             operation.
 * Always returns EVOATTN_OK.  Not synchronised with launches already
 * enqueued by other host threads.
 */
evoattn_status evoattn_debug_set_wait(unsigned long long limit_ns, int stall);

/* Static, NUL-terminated English description of a status code. */
const char* evoattn_status_string(evoattn_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int evoattn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* EVOATTN_H */
