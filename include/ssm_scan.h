/*
 * ssm_scan.h -- C ABI of libssmscan.so, the Mamba S6 selective scan on one
 * GB300 (sm_103a).
 *
 * The operation (rustytorch commit log, "MambaBlock" S6 forward commit:
 * "delta=softplus(dt.dt_proj+dt_bias) -> A=-exp(A_log) -> sequential scan
 * h=dA.h+dBu, y=sum C.h + D.u -> gate by SiLU(z)"):
 *
 *   Delta[b,t,d] = softplus(dt[b,t,d] + dt_bias[d])     (dt + dt_bias if delta_softplus == 0)
 *   h[b,d,n]    <- exp(Delta*A[d,n]) * h[b,d,n] + Delta*x[b,t,d]*Bm[b,t,n]
 *   y[b,t,d]     = (sum_n Cm[b,t,n]*h[b,d,n] + Dskip[d]*x[b,t,d]) * silu(z[b,t,d])
 *
 * with h starting from h0 (zeros when NULL). The caller folds A = -exp(A_log)
 * itself; the gradient of A_log is dA * A (the analytic-VJP commit:
 * "A_log (via A=-exp(A_log) => dA_log = dA.A)").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Memory: every pointer is DEVICE memory of the current CUDA device, owned
 *   by the caller. The library allocates, frees and synchronises nothing on
 *   these calls (ssm_poll_status excepted, which synchronises its stream).
 * - Layout: dense row-major, channel-contiguous ("token-major"):
 *     x, z, dt, y, dy, dx, dz, d_dt      [B, L, D]
 *     Bm, Cm, dB, dC                      [B, L, N]   (per token, shared by all channels)
 *     A, dA                               [D, N]
 *     Dskip, dt_bias, dD, d_dt_bias       [D]
 *     h0, h_last, dh_last, dh0, state     [B, D, N]
 *     ckpt                                [B, ceil(L/8), N/2, D, 2]  (state before tokens 0, 8, 16,
 *                                          ...; state n of channel d at [.., n/2, d, n%2])
 * - Types: x, z, Bm, Cm, y, dy, dx, dz (and the step's x_t, z_t, Bm_t, Cm_t,
 *   y_t) use the I/O dtype (SSM_F32 or SSM_BF16). Everything else is fp32.
 *   All arithmetic and the recurrent state are fp32.
 * - Shapes: N must be 16 (else SSM_ERR_UNSUPPORTED). D must be a multiple of
 *   8 and every pointer 16-byte aligned (else SSM_ERR_ALIGNMENT). B, L or
 *   D may be 0.
 * - Streams: calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 *   legacy default stream). Inputs must stay valid until the work completes.
 * - Errors: argument errors are found on the host before anything is
 *   launched and return a negative code; nothing is written. A failed launch
 *   returns SSM_ERR_CUDA. Non-finite outputs are latched on the device in the
 *   workspace status word and reported by ssm_poll_status.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = -1, /* null required pointer, negative size, bad flag */
    SSM_ERR_UNSUPPORTED = -2, /* N != 16, unknown dtype, B*L > 2^30 */
    SSM_ERR_ALIGNMENT = -3,   /* D % 8 != 0 or a pointer not 16-byte aligned */
    SSM_ERR_WORKSPACE = -4,   /* workspace missing or smaller than ssm_scan_workspace_bytes */
    SSM_ERR_CUDA = -5,        /* a CUDA runtime call or launch failed */
    SSM_ERR_TIMEOUT = -6,     /* (ssm_poll_status) a bounded wait inside a kernel ran out */
    SSM_ERR_NONFINITE = -7,   /* (ssm_poll_status) a kernel produced Inf/NaN */
    SSM_ERR_SCRATCH_LIMIT = -8 /* (ssm_scan_fwd_noalloc) carries exceed the built-in 8 MiB array */
};

/* Forward over a whole sequence.
 * Inputs: x, z (NULL = no gate: y = p), Bm, Cm [I/O dtype]; dt [fp32];
 *   dt_bias, Dskip (NULL = 0), A [fp32]; h0 (NULL = zero state).
 * Outputs: y [I/O dtype]; h_last (nullable) = state after token L-1;
 *   ckpt (nullable) = the state before every 8th token, which
 *   ssm_scan_bwd needs; size ssm_scan_ckpt_elems() floats.
 * workspace: >= ssm_scan_workspace_bytes(B, L, D, N) bytes, 16-byte
 *   aligned, holding the status word and the chunk carries along L.
 * nsplit / groups: launch shape; 0 = automatic. groups = number of
 *   L-segments scanned in parallel, joined by chunk carries (0: chosen from
 *   the device's occupancy). The forward kernel has one lane layout (two
 *   lanes share a pair of channels, 8 states each): nsplit must be 0, 1, 2
 *   or 4 and is otherwise ignored here. Results are the same up to rounding for every
 *   choice; with groups == 1 the forward is bitwise equal to stepping
 *   ssm_step through the sequence. */
typedef struct {
    int64_t B, L, D, N;
    int32_t io_dtype;       /* ssm_dtype */
    int32_t delta_softplus; /* 1: Delta = softplus(dt + dt_bias); 0: Delta = dt + dt_bias */
    const void* x;
    const void* z;
    const void* Bm;
    const void* Cm;
    const float* dt;
    const float* dt_bias;
    const float* A;
    const float* Dskip;
    const float* h0;
    void* y;
    float* h_last;
    float* ckpt;
    void* workspace;
    size_t workspace_bytes;
    int32_t nsplit;
    int32_t groups;
    /* Elements from one token's Bm row to the next token's (the same for
     * Cm); 0 = N, dense [B,L,N]. Bm and Cm may be column slices of the
     * x_proj output [B*L, R + 2N] ("MambaBlock" S6 forward commit: x_proj
     * emits dt_rank + 2*d_state per token), read in place with bc_stride =
     * R + 2N. Must be >= N (else SSM_ERR_INVALID_ARG) and a multiple of 16
     * bytes (else SSM_ERR_ALIGNMENT). dB and dC stay dense [B,L,N]. */
    int64_t bc_stride;
} ssm_fwd_args;

/* Reverse pass for loss = <dy, y> + <dh_last, h_last> (the analytic VJP:
 * "reverse-time recurrence over the cached h trajectory", gradients summed
 * over the batch).
 * f: the forward arguments of the same call (x, z, Bm, Cm, dt, dt_bias, A,
 *   Dskip, h0 are read; f.ckpt must hold what ssm_scan_fwd wrote; f.y and
 *   f.h_last are not touched). f.groups sets this pass's L-groups (0:
 *   chosen from the device's occupancy); the backward kernels have one lane
 *   layout (two lanes share a pair of channels, each taking 8 of the 16
 *   states), so f.nsplit is validated and otherwise ignored here.
 * dy [I/O dtype]; dh_last [fp32, nullable = 0].
 * Outputs, written for every element:
 *   dx, dz [I/O dtype] (dz required iff f.z != NULL); d_dt [fp32] = dLoss/d(dt);
 *   dA [D,N], dD [D], d_dt_bias [D], dB, dC [B,L,N] fp32, OVERWRITTEN
 *   (zeroed on the stream first; summed over batch and tokens / channels);
 *   dh0 [B,D,N] fp32 (nullable).
 * In place: dx may alias dy, dz may alias z, d_dt may alias dt. */
typedef struct {
    ssm_fwd_args f;
    const void* dy;
    const float* dh_last;
    void* dx;
    void* dz;
    float* d_dt;
    float* dA;
    float* dD;
    float* d_dt_bias;
    float* dB;
    float* dC;
    float* dh0;
} ssm_bwd_args;

/* One token for every (b,d) channel ("MambaRecurrence ... step(state, x_t)
 * -> (state', y_t)"): state [B,D,N] fp32 is updated in place and y_t [B,D]
 * written. x_t, z_t (nullable), dt_t [B,D]; Bm_t, Cm_t [B,N]. Uses the very
 * same per-token arithmetic as ssm_scan_fwd, so stepping from a state the
 * forward passed through reproduces the forward's outputs bit for bit.
 * workspace: nullable; when given (>= 256 bytes) non-finite outputs are
 * latched in its status word.
 * nsplit: lanes per channel, 1 or 2 (each lane takes one or both halves of
 * the readout); 4 runs as 2; 0 = automatic. */
typedef struct {
    int64_t B, D, N;
    int32_t io_dtype;
    int32_t delta_softplus;
    const void* x_t;
    const void* z_t;
    const void* Bm_t;
    const void* Cm_t;
    const float* dt_t;
    const float* dt_bias;
    const float* A;
    const float* Dskip;
    float* state;
    void* y_t;
    void* workspace;
    int32_t nsplit;
    int32_t pad_;
    /* Elements from one batch row of Bm_t to the next (the same for Cm_t);
     * 0 = N. Same rules as ssm_fwd_args.bc_stride. */
    int64_t bc_stride;
} ssm_step_args;

int ssm_scan_fwd(const ssm_fwd_args* args, void* stream);
int ssm_scan_bwd(const ssm_bwd_args* args, void* stream);
int ssm_step(const ssm_step_args* args, void* stream);

/* The paper has no counterpart to this entry point. It is ssm_scan_fwd for
 * callers that cannot allocate device memory (code running inside an
 * allocator or memory-pool callback, a process whose device memory another
 * component plans in full, a plug-in handed only its input and output
 * tensors): the chunk carries along L, which ssm_scan_fwd keeps in the
 * caller's workspace, live in an 8 MiB array compiled into the library,
 * reserved on every GPU that loads it until the process exits. Nothing is
 * allocated. Arguments and results are those of ssm_scan_fwd, except:
 * workspace is optional and, when given (>= 256 bytes), only receives the
 * status word; groups == 0 picks at most the L-groups whose carries fit the
 * array; an explicit groups that does not fit returns SSM_ERR_SCRATCH_LIMIT
 * before anything runs. The first call in each CUDA context (for the
 * runtime's primary contexts: once per device) looks up the array's address
 * with that device current; make it before any stream capture. All calls
 * share the array: calls that overlap on the GPU race and must be
 * serialised. */
int ssm_scan_fwd_noalloc(const ssm_fwd_args* args, void* stream);

/* Gradient of A_log for A = -exp(A_log) (the analytic-VJP commit: "A_log
 * (via A=-exp(A_log) => dA_log = dA.A)"): dA_log[i] = dA[i] * A[i] for
 * i < n, fp32 device arrays; dA_log may alias dA. Asynchronous on stream. */
int ssm_dA_log_grad(const float* dA, const float* A, float* dA_log, int64_t n, void* stream);

/* The library's FMA-pipe 2^x (the Cody-Waite split and degree-6 polynomial
 * that a kernel can use instead of the MUFU ex2 where the XU pipe binds):
 * y[i] = 2^x[i] for i < n, fp32 device arrays, relative error below 2^-23
 * for -125.5 <= x <= 127 and 0 below -125.5. For tests and error-bound
 * checks; asynchronous on stream. */
int ssm_exp2_fma(const float* x, float* y, int64_t n, void* stream);

/* Causal depthwise conv1d + SiLU, the step in front of the scan
 * (rustytorch commit log, "MambaBlock" S6 forward commit: "in_proj -> causal
 * depthwise conv1d -> SiLU -> x_proj -> ..."; the MambaRecurrence commit
 * carries the conv-ring state between steps). Per (b, d) channel, with the
 * K-1 inputs before t = 0 in state_in (NULL = zeros):
 *   x[t] = silu(bias[d] + sum_{k<K} w[d,k] * xin[t-(K-1)+k])
 * xin, x [B,L,D] in the I/O dtype (SSM_F32 or SSM_BF16); w [D,K] fp32 with
 * K in 1..4 (else SSM_ERR_UNSUPPORTED); bias [D] fp32 (NULL = 0); state_in,
 * state_out [B,D,K-1] fp32, oldest input first (state_out, nullable, gets
 * the last K-1 inputs). D must be a multiple of 8 and every pointer 16-byte
 * aligned (else SSM_ERR_ALIGNMENT). x must not alias xin (chunks read the
 * K-1 inputs before their start; SSM_ERR_INVALID_ARG). state_out may be
 * state_in (every ring entry is read before any is written; each channel's
 * tokens then go to one warp): with L = 1 that is the conv-ring step of
 * decoding.
 * workspace: nullable; when given (>= 256 bytes) non-finite outputs are
 * latched in its status word (ssm_poll_status). Asynchronous on `stream`;
 * the caller owns every buffer. */
typedef struct {
    int64_t B, L, D, K;
    int32_t io_dtype;
    int32_t pad_;
    const void* xin;
    const float* w;
    const float* bias;
    const float* state_in;
    void* x;
    float* state_out;
    void* workspace;
} ssm_conv_args;

/* Reverse pass of ssm_conv1d_fwd for loss = <dx, x>.
 * f: the forward's arguments (xin, w, bias, state_in are read; f.x and
 *   f.state_out are not touched). dx [B,L,D] I/O dtype.
 * Outputs: dxin [B,L,D] I/O dtype (must alias neither dx nor xin: chunks
 *   read K-1 tokens past their end); dw [D,K] and dbias [D]
 *   fp32, OVERWRITTEN (zeroed on the stream first; summed over batch and
 *   tokens; dbias nullable); dstate_in [B,D,K-1] fp32 (nullable) = the
 *   gradient of the initial conv state. */
typedef struct {
    ssm_conv_args f;
    const void* dx;
    void* dxin;
    float* dw;
    float* dbias;
    float* dstate_in;
} ssm_conv_bwd_args;

int ssm_conv1d_fwd(const ssm_conv_args* args, void* stream);
int ssm_conv1d_bwd(const ssm_conv_bwd_args* args, void* stream);

/* The dt projection with its softplus fused into the GEMM epilogue, on the
 * tensor cores ("MambaBlock" S6 forward commit: "delta=softplus(dt.dt_proj
 * +dt_bias)", dt being the first dt_rank columns of the x_proj output):
 *   delta[m,d] = softplus(bias[d] + sum_{r<R} a[m,r] * w[d,r])    (softplus = 1)
 *   delta[m,d] = bias[d] + sum_{r<R} a[m,r] * w[d,r]              (softplus = 0)
 * M = batch * tokens. a [M,R] bf16, rows a_stride elements apart (0 = R), so
 * a may be the first R columns of the x_proj output [M, R + 2N]; w [D,R]
 * bf16 (the projection's weight); bias [D] fp32 (NULL = 0); delta [M,D]
 * fp32, which ssm_scan_fwd then takes as dt with delta_softplus = 0 and no
 * dt_bias. R a multiple of 16 in 16..256 (else SSM_ERR_UNSUPPORTED); D a
 * multiple of 8, a_stride * 2 bytes and every pointer 16-byte aligned (else
 * SSM_ERR_ALIGNMENT). Products are fp32-accumulated from the bf16 operands.
 * workspace: nullable status word (non-finite outputs; SSM_ERR_TIMEOUT if
 * the tensor core's completion never arrived). Asynchronous on `stream`. */
typedef struct {
    int64_t M, D, R;
    int64_t a_stride;
    int32_t softplus;
    int32_t pad_;
    const void* a;
    const void* w;
    const float* bias;
    float* delta;
    void* workspace;
} ssm_dtproj_args;

/* Reverse pass up to the pre-activation, for the gradient ddelta [M,D] fp32
 * arriving at delta: dpre[m,d] = ddelta[m,d] * sigmoid(pre[m,d]) (ddelta
 * itself when softplus = 0), the pre-activation recomputed on the tensor
 * cores; dbias [D] (nullable) = sum over m of dpre, OVERWRITTEN. dpre may be
 * ddelta (in place). The gradients of a and w are the plain products
 * dpre @ w and dpre^T @ a (the caller's GEMMs). f.delta is not used. */
typedef struct {
    ssm_dtproj_args f;
    const float* ddelta;
    float* dpre;
    float* dbias;
} ssm_dtproj_bwd_args;

int ssm_dtproj_fwd(const ssm_dtproj_args* args, void* stream);
int ssm_dtproj_bwd(const ssm_dtproj_bwd_args* args, void* stream);

/* Bytes of workspace a fwd or bwd call of this shape needs (>= 256). */
size_t ssm_scan_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N);
/* fp32 elements of the checkpoint buffer: B * ceil(L/8) * N * D. */
int64_t ssm_scan_ckpt_elems(int64_t B, int64_t L, int64_t D, int64_t N);
/* Tokens between checkpoints (8). */
int ssm_scan_ckpt_interval(void);
/* Synchronises `stream`, reads and clears the workspace status word.
 * Returns SSM_OK, SSM_ERR_TIMEOUT, SSM_ERR_NONFINITE, or SSM_ERR_CUDA. */
int ssm_poll_status(void* workspace, void* stream);
/* Zeroes the workspace status word on `stream` (asynchronous). */
int ssm_clear_status(void* workspace, void* stream);
/* Static English description of a status code. */
const char* ssm_status_string(int code);
/* Launches of the library's own kernels made by the most recent
 * fwd / bwd / step / dA_log / conv / dtproj / noalloc call on this host
 * thread. */
int ssm_last_launch_count(void);

/* Testing hook for the bounded waits (no counterpart on the pages). Arms,
 * for the next ssm_scan_fwd call on this host thread only, a staging fault
 * in its main forward kernel: every warp arms the barrier of its tile `tile`
 * (counted from the start of its L-group) without issuing that tile's
 * copies, and every wait of that kernel gives up after wait_ns nanoseconds
 * (0: the default of one second). The call returns SSM_OK; the warps stop at
 * that tile, wait (bounded) for the copies they still have in flight and
 * leave, y / h_last / ckpt are not valid, and ssm_poll_status then returns
 * SSM_ERR_TIMEOUT. tile < 0 disarms. Returns SSM_ERR_INVALID_ARG for
 * wait_ns above 10 s. */
int ssm_debug_arm_wait_fault(int64_t tile, uint64_t wait_ns);

#ifdef __cplusplus
}
#endif
#endif /* SSM_SCAN_H */
