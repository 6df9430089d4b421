/*
 * ssm.h -- C ABI of the B300 selective state space (S6) library (libssm.so).
 *
 * Five operations, from the Mamba paper (arXiv 2312.00752) and its Mamba-2
 * successor as restated on the pages this library follows:
 *
 *   ssm_scan_fwd      the selective-scan forward pass.  For every batch b,
 *                     channel d and state n:
 *                       Delta_t   = softplus(delta[b,d,t] + delta_bias[d])
 *                       Abar_t[n] = exp(Delta_t * A[d,n])
 *                       h_t[n]    = Abar_t[n] h_{t-1}[n] + Delta_t B[b,n,t] u[b,d,t]
 *                                   (or the exact zero-order-hold input term, SSM_DISC_ZOH)
 *                       y[b,d,t]  = (sum_n C[b,n,t] h_t[n] + Dskip[d] u[b,d,t]) * silu(z[b,d,t])
 *                     ("Mamba paper translation", gitcode.csdn.net: section 2
 *                     "State Space Models" for the recurrence and the
 *                     per-channel diagonal A, section 3.2 for the selection
 *                     of Delta, B, C and softplus, section 3.3.2 for the
 *                     fused scan that never writes h to HBM, section 3.6 for
 *                     the Delta bias; "Mamba and state space models",
 *                     docs.ifdog.com: section "Discretisation" for
 *                     Abar = exp(Delta A), the numpy selective-SSM listing for
 *                     the Euler input term Delta B u, section "Mamba
 *                     architecture" for the silu gate.)
 *   ssm_state_update  one recurrent (decode) step of the same recurrence
 *                     against a persistent fp32 state ("gitcode", section 1
 *                     and section 2: constant time per generated token).
 *   ssm_scan_bwd      the gradients of the scan for training, with the
 *                     forward states recomputed rather than stored
 *                     ("gitcode", section 3.3.2).
 *   ssm_causal_conv1d_fwd
 *                     the causal depthwise convolution along time, with an
 *                     optional SiLU, that produces the SSM branch's input
 *                     ("docs.ifdog.com", section "Mamba architecture", step
 *                     3a; step 3b feeds its output to the projections that
 *                     make Delta, B and C and to the scan as u).
 *   ssm_ssd_fwd       the Mamba-2 state-space-dual layer (scalar A per head,
 *                     chunked on the tensor cores; see ssm_ssd_args_t).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers unless stated otherwise; the
 *     caller owns every buffer, including the optional workspace.  The
 *     library never allocates, frees or synchronises, and keeps no state
 *     between calls other than the device status word (below).
 *   - Strides are in ELEMENTS.  The time (last) stride of every sequence
 *     tensor must be 1.  Other strides must be >= 0; a batch stride of 0
 *     broadcasts a tensor across the batch.  Output tensors (y, h_last,
 *     state) must not overlap each other or any input.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous: SSM_OK means "validated and enqueued".  Errors in a
 *     kernel that has already been enqueued surface at the caller's next
 *     synchronisation, or through ssm_get_device_status().
 *   - Argument errors are detected on the host before anything is enqueued;
 *     nothing is written in that case.  No C++ exception crosses the ABI.
 *   - Calls on different streams may run concurrently; the library is
 *     re-entrant.
 */
#ifndef SSM_B300_H
#define SSM_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,   /* null pointer, bad size or stride, overlapping outputs */
    SSM_ERR_UNSUPPORTED = 2,   /* well-formed but outside what the kernels implement */
    SSM_ERR_CUDA = 3,          /* a CUDA call failed while enqueueing (error is cleared) */
    SSM_ERR_TIMEOUT = 4,       /* a bounded device-side wait gave up (device status only) */
    SSM_ERR_WORKSPACE = 5      /* workspace missing or smaller than ssm_scan_workspace_size() */
} ssm_status_t;

typedef enum {
    SSM_F32 = 0,               /* IEEE binary32 */
    SSM_BF16 = 1               /* bfloat16; the state and all arithmetic stay fp32 */
} ssm_dtype_t;

/* discretisation of the input term ("docs.ifdog.com", section "Discretisation"):
 * Euler Bbar x = Delta B u (the default), or the exact zero-order hold
 * Bbar x = (exp(Delta A) - 1) / A * B u (Delta B u where A = 0).  Abar = exp(Delta A)
 * in both. */
#define SSM_DISC_EULER 0
#define SSM_DISC_ZOH   1

/* flags for ssm_scan_args_t.flags (testing and tuning; 0 = automatic) */
#define SSM_SCAN_FORCE_GENERIC 0x1   /* use the stride-general kernel */
#define SSM_SCAN_FORCE_TILED   0x2   /* use the tiled single-pass kernel (error if impossible) */
#define SSM_SCAN_FORCE_CHUNKED 0x4   /* use the three-pass chunked kernel (error if impossible) */
/* use the warp-shuffle associative scan: lanes over 32 consecutive steps,
 * five combine rounds per tile, one warp per channel (Euler input term, real
 * A, dstate <= 16, any strides; SSM_ERR_UNSUPPORTED otherwise).  Never chosen
 * automatically: it does several times the arithmetic per state update. */
#define SSM_SCAN_FORCE_WARPSCAN 0x8

/*
 * Arguments of ssm_scan_fwd.  Shapes (with strides in elements, time stride 1):
 *   u, delta, z, y : (batch, dim, seqlen)     io_dtype
 *   Bm, Cm         : (batch, dstate, seqlen)  io_dtype  (batch stride may be 0)
 *   A              : (dim, dstate)            fp32, real (normally negative)
 *   Dskip          : (dim,)                   fp32, contiguous, nullable (no skip term)
 *   delta_bias     : (dim,)                   fp32, contiguous, nullable (bias 0)
 *   h0, h_last     : (batch, dim, dstate)     fp32, nullable (zero initial state /
 *                                             final state not returned)
 *   z              : nullable (no gate)
 * Limits: 1 <= dstate <= 64; batch, dim, seqlen >= 0 (an empty problem is a no-op).
 *
 * Complex A ("gitcode", section 3.6: complex states, the S4D-Lin initialisation
 * A[d,n] = -1/2 + n i): when A_imag is set, A + i A_imag is a complex diagonal
 * (both fp32 with the strides stride_A), the state h is complex, Abar =
 * exp(Delta A) is the complex exponential, the input term Delta B u is real
 * and enters the state as it is, and the output reads the real part of the C
 * contraction: y = (Re(sum_n C h) + Dskip u) * silu(z).  h0 and h_last then
 * hold complex numbers as (re, im) fp32 pairs: element (b, d, n) has its real
 * part at [b*s0 + d*s1 + n*s2] and its imaginary part one float after it
 * (a dense (batch, dim, dstate, 2) array has strides (2*dim*dstate,
 * 2*dstate, 2)).  Complex A takes the Euler input term, the single-pass or
 * stride-general kernels (never the chunked path) and is not supported by
 * ssm_scan_bwd, ssm_scan_fwd_noalloc or ssm_state_update
 * (SSM_ERR_UNSUPPORTED).
 */
typedef struct ssm_scan_args {
    int64_t batch, dim, seqlen, dstate;        /* B, D, L, N */
    ssm_dtype_t io_dtype;
    int32_t delta_softplus;                    /* 1: Delta = softplus(delta + bias); 0: delta + bias */
    const void *u, *delta, *z, *Bm, *Cm;
    const float *A, *Dskip, *delta_bias;
    const float *h0;
    float *h_last;
    void *y;
    int64_t stride_u[3], stride_delta[3], stride_z[3], stride_y[3];   /* (b, d, t) */
    int64_t stride_B[3], stride_C[3];                                 /* (b, n, t) */
    int64_t stride_A[2];                                              /* (d, n)    */
    int64_t stride_h0[3], stride_h_last[3];                           /* (b, d, n) */
    int32_t flags;                             /* SSM_SCAN_FORCE_*; 0 = automatic */
    int32_t discretization;                    /* SSM_DISC_EULER (0) or SSM_DISC_ZOH */
    int64_t chunk_len;                         /* chunked path: timesteps per chunk; 0 = automatic */
    void *workspace;                           /* device scratch, caller-owned, nullable if 0 bytes needed */
    size_t workspace_bytes;
    const float *A_imag;                       /* nullable: imaginary part of a complex A (see below) */
} ssm_scan_args_t;

/*
 * Arguments of ssm_state_update (one decode step, the state updated in place).
 *   state          : (batch, dim, dstate)  fp32, read then overwritten
 *   u, delta, z, y : (batch, dim)          io_dtype; z nullable
 *   Bm, Cm         : (batch, dstate)       io_dtype (batch stride may be 0)
 *   A              : (dim, dstate) fp32;  Dskip, delta_bias : (dim,) fp32 contiguous, nullable
 * Limits: 1 <= dstate <= 64.
 */
typedef struct ssm_step_args {
    int64_t batch, dim, dstate;
    ssm_dtype_t io_dtype;
    int32_t delta_softplus;
    float *state;
    const void *u, *delta, *z, *Bm, *Cm;
    const float *A, *Dskip, *delta_bias;
    void *y;
    int64_t stride_state[3];                   /* (b, d, n) */
    int64_t stride_u[2], stride_delta[2], stride_z[2], stride_y[2];   /* (b, d) */
    int64_t stride_B[2], stride_C[2];          /* (b, n) */
    int64_t stride_A[2];                       /* (d, n) */
    int32_t discretization;                    /* SSM_DISC_EULER (0) or SSM_DISC_ZOH */
    int32_t reserved0;
} ssm_step_args_t;

/*
 * Arguments of ssm_scan_bwd: the gradients of ssm_scan_fwd (training).  With
 * L the scalar being differentiated, dy = dL/dy and dh_last = dL/dh_last,
 * it writes dL/d(every input) of the forward call described by `fwd`, by the
 * chain rule through the recurrence run backwards in time (the adjoint
 * lambda_t = dL/dh_t = dy_t silu(z_t) C_t + Abar_{t+1} lambda_{t+1}).  The
 * forward states are not stored by ssm_scan_fwd: this call recomputes them
 * ("gitcode", section 3.3.2, recomputation), keeping one state checkpoint
 * every SSM_BWD_SEGMENT steps in the caller's workspace.
 *   fwd           : the forward call's inputs; its y, h_last, flags and chunk_len
 *                   are ignored, its workspace fields are used for the checkpoints
 *   dy            : (batch, dim, seqlen)   io_dtype
 *   dh_last       : (batch, dim, dstate)   fp32, nullable (zero)
 *   du, ddelta    : (batch, dim, seqlen)   io_dtype
 *   dz            : (batch, dim, seqlen)   io_dtype, required exactly when fwd.z is set
 *   dA            : (dim, dstate)          fp32
 *   dB, dC        : (batch, dstate, seqlen) fp32; batch stride 0 (a single row) when
 *                   fwd's B / C are shared across the batch (their batch stride is 0)
 *   dDskip        : (dim,) fp32 contiguous, required exactly when fwd.Dskip is set
 *   ddelta_bias   : (dim,) fp32 contiguous, nullable
 *   dh0           : (batch, dim, dstate)   fp32, nullable
 * dA, dB, dC, dDskip and ddelta_bias are sums over the batch (and time, and
 * for dB/dC over the channels): the call overwrites them (zeroes, then adds
 * with atomics, so the order of the fp32 sums is not fixed).  Both input
 * terms of fwd.discretization are differentiated: Euler (g = Delta) and the
 * exact zero-order hold (g = (exp(Delta A) - 1) / A, whose derivatives are
 * dg/dDelta = exp(Delta A) and dg/dA = Delta^2 psi(Delta A) with
 * psi(x) = (x e^x - (e^x - 1)) / x^2).  Limits: 1 <= dstate <= 64; a real A
 * (fwd.A_imag NULL); the gradient outputs must not overlap each other or any
 * input.
 */
#define SSM_BWD_SEGMENT 8
typedef struct ssm_scan_bwd_args {
    ssm_scan_args_t fwd;
    const void *dy;
    const float *dh_last;
    void *du, *ddelta, *dz;
    float *dA, *dB, *dC, *dDskip, *ddelta_bias, *dh0;
    int64_t stride_dy[3], stride_du[3], stride_ddelta[3], stride_dz[3];   /* (b, d, t) */
    int64_t stride_dB[3], stride_dC[3];                                  /* (b, n, t) */
    int64_t stride_dh_last[3], stride_dh0[3];                            /* (b, d, n) */
} ssm_scan_bwd_args_t;

/* Bytes of device workspace ssm_scan_bwd needs (the state checkpoints:
 * batch * dim * ceil(seqlen / SSM_BWD_SEGMENT) * NP floats, NP = 16, 32 or 64
 * for dstate up to 16, 32 or 64).  Host-only. */
ssm_status_t ssm_scan_bwd_workspace_size(const ssm_scan_bwd_args_t *args, size_t *bytes);

/* Gradients of the selective scan (see ssm_scan_bwd_args_t). */
ssm_status_t ssm_scan_bwd(const ssm_scan_bwd_args_t *args, void *stream);

/*
 * Arguments of ssm_causal_conv1d_fwd.  Per batch b, channel d and step t:
 *   out[b,d,t] = act(bias[d] + sum_{k=0}^{width-1} weight[d,k] * x[b,d,t-(width-1)+k])
 * Tap width-1 multiplies the current step (the tap order of a framework
 * Conv1d with width-1 steps of left padding).  Inputs before t = 0 are
 * x_hist[b,d,0..width-2], oldest first, or zero when x_hist is NULL, so a
 * sequence split at any step continues exactly when the next call gets the
 * last width-1 inputs of the previous one.  act is SiLU, v * sigmoid(v), when
 * silu != 0, else the identity.
 *   x, out  : (batch, dim, seqlen)   io_dtype, time stride 1
 *   weight  : (dim, width)           fp32
 *   bias    : (dim,)                 fp32, contiguous, nullable (no bias)
 *   x_hist  : (batch, dim, width-1)  io_dtype, nullable
 * Limits: 1 <= width <= 16; batch, dim, seqlen >= 0 (empty is a no-op).
 * out must not overlap x, weight, bias or x_hist.  Arithmetic is fp32; a
 * bf16 out is rounded to nearest even.
 */
typedef struct ssm_conv_args {
    int64_t batch, dim, seqlen;                /* B, D, L */
    int32_t width;                             /* taps, W */
    ssm_dtype_t io_dtype;                      /* x, x_hist, out */
    int32_t silu;                              /* 1: SiLU after the bias */
    int32_t reserved0;
    const void *x;
    const float *weight, *bias;
    const void *x_hist;
    void *out;
    int64_t stride_x[3], stride_out[3];        /* (b, d, t) */
    int64_t stride_weight[2];                  /* (d, k) */
    int64_t stride_x_hist[3];                  /* (b, d, k) */
} ssm_conv_args_t;

/* Causal depthwise convolution (+ SiLU) along time (see ssm_conv_args_t). */
ssm_status_t ssm_causal_conv1d_fwd(const ssm_conv_args_t *args, void *stream);

/*
 * Arguments of ssm_ssd_fwd: the Mamba-2 state-space-dual (SSD) layer ("Mamba
 * close reading", alishangtian.com, section on SSD and Mamba-2: A is a scalar
 * times the identity per head, heads as in multi-head attention, larger
 * states; "Mamba and state space models", docs.ifdog.com, section "Mamba-2
 * and structured duality": the layer is multiplication by a semiseparable
 * matrix (L o C B^T) with a data-dependent decay mask L).  With H heads of P
 * channels each (channel d = h P + p), per batch b, state n and step t:
 *   Delta_t  = softplus(delta[b,h,t] + delta_bias[h])   (or the plain sum)
 *   h_t[p,n] = exp(Delta_t A[h]) h_{t-1}[p,n] + Delta_t B[b,t,n] x[b,d,t]
 *   y[b,d,t] = (sum_n C[b,t,n] h_t[p,n] + Dskip[h] x[b,d,t]) * silu(z[b,d,t])
 * B and C are shared by all heads.  Shapes (strides in elements):
 *   x, z, y      : (batch, nheads * headdim, seqlen)  io_dtype, time stride 1; z nullable
 *   delta        : (batch, nheads, seqlen)            io_dtype, time stride 1
 *   Bm, Cm       : (batch, seqlen, dstate)            io_dtype (state index contiguous in the
 *                                                     fast kernel; any strides otherwise)
 *   A, Dskip, delta_bias : (nheads,) fp32 contiguous; Dskip and delta_bias nullable
 *   h0, h_last   : (batch, nheads, headdim, dstate)   fp32, nullable
 * Limits: 1 <= dstate <= 256.  bf16 I/O with headdim 64, dstate 128, dense
 * x (rows of seqlen, seqlen a multiple of 8) and dense B / C rows of 128 runs
 * the chunked tensor-core kernel (tcgen05.mma on 128-step chunks); every other
 * case runs the recurrence on the CUDA cores.  Outputs must not overlap inputs.
 */
#define SSM_SSD_FORCE_GENERIC 0x1   /* flags: run the CUDA-core recurrence */
typedef struct ssm_ssd_args {
    int64_t batch, nheads, headdim, seqlen, dstate;   /* B, H, P, L, N */
    ssm_dtype_t io_dtype;
    int32_t delta_softplus;
    const void *x, *delta, *z, *Bm, *Cm;
    const float *A, *Dskip, *delta_bias;
    const float *h0;
    float *h_last;
    void *y;
    int64_t stride_x[3], stride_z[3], stride_y[3];    /* (b, d, t) */
    int64_t stride_delta[3];                          /* (b, h, t) */
    int64_t stride_B[3], stride_C[3];                 /* (b, t, n) */
    int64_t stride_h0[4], stride_h_last[4];           /* (b, h, p, n) */
    int32_t flags;                                    /* SSM_SSD_FORCE_GENERIC or 0 */
    int32_t reserved0;
} ssm_ssd_args_t;

/* The Mamba-2 SSD layer (see ssm_ssd_args_t).  Asynchronous on `stream`. */
ssm_status_t ssm_ssd_fwd(const ssm_ssd_args_t *args, void *stream);

/* 1 if ssm_ssd_fwd takes the tensor-core kernel for these arguments, 0 if
 * the CUDA-core recurrence, -1 if the arguments are invalid.  Host-only. */
int ssm_ssd_plan_path(const ssm_ssd_args_t *args);

/* Bytes of device workspace ssm_scan_fwd needs for these arguments (0 for
 * the single-pass paths).  Host-only; validates the arguments first.  The
 * plan it reflects depends on the current device's SM count. */
ssm_status_t ssm_scan_workspace_size(const ssm_scan_args_t *args, size_t *bytes);

/* The selective-scan forward pass (see the header comment). */
ssm_status_t ssm_scan_fwd(const ssm_scan_args_t *args, void *stream);

/* One decode step against a persistent fp32 state. */
ssm_status_t ssm_state_update(const ssm_step_args_t *args, void *stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *ssm_status_string(ssm_status_t status);

/* Details of the last host-side error on the calling thread (static
 * thread-local buffer, empty string if none). */
const char *ssm_last_error_detail(void);

/* Reads (and, if clear != 0, resets) the current device's status word, which
 * kernels set when a bounded wait gives up (SSM_ERR_TIMEOUT).  Synchronises
 * `stream`.  *code receives SSM_OK or the first error recorded. */
ssm_status_t ssm_get_device_status(void *stream, int clear, int *code);

/*
 * ssm_scan_fwd_noalloc -- the chunked (three-pass) scan for callers that
 * cannot allocate device memory.  No counterpart in the paper: it is a
 * packaging of ssm_scan_fwd's chunked path for a deployment constraint.
 *
 * Some callers have no way to hand the library a workspace: a plugin inside
 * an engine that owns every byte of device memory, a host that only holds
 * the raw input and output pointers, or code that must not take the implicit
 * device synchronisation of cudaMalloc/cudaFree.  This entry point takes the
 * same arguments as ssm_scan_fwd, except that args->workspace and
 * args->workspace_bytes are ignored and args->flags must be 0 or
 * SSM_SCAN_FORCE_CHUNKED (any other bit is SSM_ERR_INVALID_ARG): it always
 * runs the chunked path.  The chunk records live in a scratch array that the
 * library reserves statically on every GPU it is loaded on, for the life of
 * the process: SSM_NOALLOC_SCRATCH_BYTES bytes.  It calls no allocator.
 *
 *   - The problem must fit: ssm_scan_workspace_size() with
 *     flags = SSM_SCAN_FORCE_CHUNKED must report at most
 *     SSM_NOALLOC_SCRATCH_BYTES, else SSM_ERR_WORKSPACE is returned and
 *     nothing is enqueued.  The 1 x 1536-channel, 2^20-step bf16 scan with
 *     automatic chunking needs about 2.6 MB.  Layouts the chunked path cannot
 *     take return SSM_ERR_UNSUPPORTED.
 *   - Every call looks up the scratch array's address in the current
 *     device's context (cudaGetSymbolAddress, a host-side query).
 *   - Every call on a device shares the one scratch array and leaves its
 *     records there.  No record needs to start at zero (each call writes
 *     every record before reading it), but calls whose kernels overlap on
 *     the GPU (different streams, no ordering between them) race on the
 *     array and corrupt each other's results: order them on one stream.
 */
#define SSM_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
ssm_status_t ssm_scan_fwd_noalloc(const ssm_scan_args_t *args, void *stream);

/* Measurement helper, not part of the method: enqueues blocks x 256 threads,
 * each issuing iters x 8 independent SFU operations (op 0: ex2.approx.f32, the
 * scan's exponential; op 1: rcp.approx.f32, the reciprocal in silu), and writes
 * one float per thread to sink (device, blocks * 256 floats).  Timing the
 * launch with events on `stream` gives the special-function-unit rate that
 * bounds the scan's arithmetic (its second roofline).  Returns
 * SSM_ERR_INVALID_ARG for a bad op, size or NULL sink. */
ssm_status_t ssm_probe_sfu(int op, int blocks, int iters, float *sink, void *stream);

/* Kernel path ssm_scan_fwd would take for these arguments:
 * 0 = generic, 1 = tiled single pass, 2 = chunked three-pass, 3 = warp-shuffle
 * scan (SSM_SCAN_FORCE_WARPSCAN), 4 = tiled single pass split over two launches
 * (bf16 grids of more than 4 and at most 5 32-channel blocks per SM: 4 per SM
 * on two-warp CTAs, the rest on four-warp CTAs that run beside them); -1 on
 * error. */
int ssm_scan_plan_path(const ssm_scan_args_t *args);

/* Library ABI version: (major << 16) | minor. */
int ssm_version(void);

/* sizeof of the argument structs as compiled into the library, so that a
 * binding can check its mirror of them: which = 0 -> ssm_scan_args_t,
 * 1 -> ssm_step_args_t, 2 -> ssm_conv_args_t, 3 -> ssm_scan_bwd_args_t,
 * 4 -> ssm_ssd_args_t; 0 for any other value. */
size_t ssm_abi_sizeof(int which);

#ifdef __cplusplus
}
#endif

#endif /* SSM_B300_H */
