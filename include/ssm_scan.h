/*
 * ssm_scan.h -- C ABI of the B300 (sm_103a) selective-scan library.
 *
 * The operation is the selective state-space recurrence of Mamba: a
 * diagonal linear recurrence whose step size Delta and input/output maps
 * B, C are given per token ("Mamba", elemedex.maurosantelli.com.ar, section
 * "How it works": h_t = Abar h_{t-1} + Bbar x_t, y_t = C h_t; "State Spaces,
 * Selectively - Mamba", papermap explainer, Chapter 02 "The Discretized
 * View": Delta, B, C are functions of the input, Abar and Bbar derive from
 * (Delta, A, B)).  For every channel (b, d) and state index n, over tokens
 * t = 0 .. L-1, starting from h = 0:
 *
 *     v        = delta[b,d,t] + delta_bias[d]            (bias optional)
 *     Delta    = delta_softplus ? softplus(v) : v
 *     h[n]     = exp(Delta * A[d,n]) * h[n] + Delta * B[b,t,n] * u[b,d,t]
 *     y[b,d,t] = (sum_n C[b,t,n] * h[n] + D[d] * u[b,d,t]) * silu(z[b,d,t])
 *
 * exp(Delta A) is the zero-order-hold decay ("Mamba remembers by forgetting,
 * read closely", interactiveml.org: the scalar update weights the old state
 * by exp(-Delta)); Delta*B*u is the first-order input term.  softplus,
 * delta_bias, the skip term D and the silu(z) output gate follow the usual
 * Mamba layer ("output gate", sghael.github.io Mamba page, "Simplifications
 * and limits"; "multiplicative gate", elemedex entry) and are optional.
 *
 * Layouts (row-major, contiguous, all device memory):
 *     u, delta, z, y   (batch, dim, seqlen)   seqlen fastest
 *     B, C             (batch, seqlen, dstate) one token's B row is contiguous
 *     A                (dim, dstate)          fp32
 *     D, delta_bias    (dim)                  fp32
 *     last_state/state (batch, dim, dstate)   fp32
 *   Single-token step: x, delta, z, y (batch, dim); B, C (batch, dstate).
 * u, delta, z, B, C and y share the I/O element type (fp32 or bf16); the
 * recurrence and the state are always fp32; bf16 outputs are rounded to
 * nearest even once, at the store.
 *
 * Ownership and execution: the caller owns every buffer.  Every pointer is
 * a device pointer (or a host-mapped pointer the device can read), except
 * for ssm_scan_fwd_host, which takes host buffers.  Each call validates its
 * arguments on the host, enqueues work on the caller's stream and returns;
 * none synchronises the device.  Outputs must not alias inputs (state, the
 * only in/out buffer, excepted).  The library prints nothing.
 * Allocation and state kept by the library:
 *   - ssm_scan_fwd, ssm_scan_fwd_ex, ssm_scan_bwd, ssm_scan_bwd_ex, ssm_state_step,
 *     ssm_scan_fwd_noalloc allocate nothing; their scratch is the caller's
 *     workspace (ssm_scan_fwd_noalloc: a fixed buffer inside the library).
 *   - ssm_scan_fwd_host allocates its device staging buffers on the caller's
 *     stream (cudaMallocAsync, returned with cudaFreeAsync) and keeps two
 *     CUDA streams per device, created at its first call and held until exit.
 *   - Per device, the library caches the SM count and the occupancy of each
 *     kernel instance it has launched (read-only facts of the device), and
 *     ssm_scan_fwd_noalloc keeps its buffer's device address.
 * Calls on different streams with disjoint outputs and workspaces may run
 * concurrently.
 *
 * Errors: 0 on success, else a negative ssm_status.  Argument errors are
 * detected on the host before anything is enqueued.  A launch error is
 * reported as SSM_ERR_CUDA (the CUDA error is left for the caller's next
 * CUDA call to see, as the runtime does).  Faults inside a kernel surface
 * at the caller's next synchronisation, as for any CUDA kernel.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ssm_status {
    SSM_OK = 0,
    SSM_ERR_NULL_ARG = -1,      /* a required pointer is NULL */
    SSM_ERR_BAD_DIMS = -2,      /* a size is out of range or overflows */
    SSM_ERR_UNSUPPORTED_N = -3, /* dstate is not 1, 2, 4, 8 or 16 */
    SSM_ERR_BAD_DTYPE = -4,     /* unknown I/O element type */
    SSM_ERR_MISALIGNED = -5,    /* a pointer is not aligned to its element size */
    SSM_ERR_CUDA = -6,          /* the CUDA runtime refused the launch */
    SSM_ERR_WORKSPACE = -7,     /* workspace missing, too small or misaligned */
    SSM_ERR_ALIAS = -8,         /* an output overlaps an input */
    SSM_ERR_TIMEOUT = -9,       /* a bounded on-device wait gave up */
    SSM_ERR_TOO_LARGE = -10,    /* needs more scratch than ssm_scan_fwd_noalloc holds */
    SSM_ERR_BAD_OPTION = -11,   /* an option (a field of ssm_scan_opts, an input_term) is out of range */
    SSM_ERR_DEVICE = -12        /* a -DSSM_DEBUG build's bounds check failed on the device */
} ssm_status;

typedef enum ssm_io_dtype { SSM_IO_F32 = 0, SSM_IO_BF16 = 1 } ssm_io_dtype;

/* Problem sizes.  seqlen is ignored by ssm_state_step. */
typedef struct ssm_dims {
    int64_t batch;   /* Bt >= 1 */
    int64_t dim;     /* D >= 1: channels per batch row */
    int64_t dstate;  /* N in {1, 2, 4, 8, 16}: state entries per channel */
    int64_t seqlen;  /* L >= 0: tokens */
    int32_t io;      /* ssm_io_dtype of u, delta, z, B, C, y */
    int32_t chunk;   /* >= 0.  ssm_scan_fwd: 0: library default schedule.
                        chunk >= seqlen: a cap on the work of one CTA, in
                        tokens of a channel group: the scan then runs on at most
                        ceil(groups * seqlen / chunk) CTAs, splitting a group's
                        tokens between two CTAs where the ranges fall.  Every
                        channel's arithmetic is unchanged: outputs are bitwise
                        equal to the default schedule's.
                        0 < chunk < seqlen: the chunked schedule, with chunks of
                        chunk tokens (rounded up to 32): every chunk's affine
                        map is computed in parallel by walking the chunk back
                        from its end (the walk stops once the product of the
                        decays passed is below 2^-40 for every state, where
                        the earlier tokens no longer change the fp32 result),
                        the maps are composed into carry-ins, and the chunks
                        are scanned from those; outputs agree up to fp32
                        rounding order.  The default schedule takes it by
                        itself for long sequences over few channels.
                        ssm_scan_bwd, ssm_scan_bwd_ex: 0 < chunk < seqlen
                        cuts the sequence into chunks of chunk tokens
                        (rounded up to 32) whose backward passes run side by
                        side, each from the state before it and the adjoint
                        after it (both composed from per-chunk maps found by
                        walks that stop where the decay product is below
                        2^-40); chunk >= seqlen: one chunk; 0: the library
                        chunks long sequences (>= 8192 tokens) over few
                        channels by itself.  Gradients agree with the
                        unchunked pass up to fp32 rounding order. */
} ssm_dims;

/*
 * Forward selective scan (the definition above) over every channel.
 *
 *   dims           sizes; see ssm_dims
 *   u, delta       (batch, dim, seqlen) I/O type; required (when seqlen is 0,
 *                  u, delta, B, C, z and y hold no elements and may be NULL)
 *   A              (dim, dstate) fp32; required.  A <= 0 is the intended use
 *                  (decaying state); other values are computed but not tuned
 *   B, C           (batch, seqlen, dstate) I/O type; required
 *   D              (dim) fp32 skip weights, or NULL for no skip term
 *   z              (batch, dim, seqlen) I/O type gate input, or NULL for no gate
 *   delta_bias     (dim) fp32, or NULL for zero bias
 *   delta_softplus nonzero: Delta = softplus(delta + bias); zero: Delta = delta + bias
 *   y              (batch, dim, seqlen) I/O type output; required
 *   last_state     (batch, dim, dstate) fp32 final state h after token L-1, or
 *                  NULL to skip writing it
 *   workspace      device scratch of at least ssm_scan_fwd_workspace_size()
 *                  bytes, 256-byte aligned; may be NULL when that size is 0.
 *                  Its contents on entry do not matter (the call clears what it
 *                  needs with cudaMemsetAsync on `stream`); the call owns it
 *                  until the enqueued work finishes, so concurrent calls need
 *                  separate workspaces.  The scan splits the token range of
 *                  some channel groups between two CTAs and hands the state
 *                  over through the workspace; that hand-over waits at most
 *                  about a second.  ssm_scan_fwd_status reports the outcome
 *                  (SSM_OK, or SSM_ERR_TIMEOUT if a hand-over gave up; the
 *                  affected outputs are then NaN).
 *   stream         cudaStream_t to enqueue on (NULL: the legacy default stream)
 *
 * Pointers of the I/O type must be aligned to the element size; the library
 * picks 16-byte vector and bulk-copy paths by itself when every row allows it.
 * Returns SSM_OK or a negative ssm_status.
 */
SSM_API int ssm_scan_fwd(const ssm_dims* dims,
                 const void* u, const void* delta, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, int delta_softplus,
                 void* y, float* last_state,
                 void* workspace, size_t workspace_bytes,
                 void* stream);

/* The input term Bbar u of the state update. */
typedef enum ssm_input_term {
    /* Bbar u = Delta B u: the first-order form (the default). */
    SSM_INPUT_DELTA_B = 0,
    /* Bbar u = (exp(Delta A) - 1) / A * B u: the exact zero-order hold of a
     * diagonal A, Delta B u in the limit A = 0.  With A = -1 and B = 1 this is
     * the scalar update h_t = exp(-Delta_t) h_{t-1} + (1 - exp(-Delta_t)) x_t
     * of "Mamba remembers by forgetting, read closely" (interactiveml.org,
     * its recurrence and its selective_scan listing). */
    SSM_INPUT_ZOH = 1
} ssm_input_term;

/* Options of ssm_scan_fwd_ex.  A zero-initialised struct (or a NULL pointer)
 * gives exactly ssm_scan_fwd. */
typedef struct ssm_scan_opts {
    int32_t input_term;        /* ssm_input_term */
    /* The block's short convolution fused into the scan ("Mamba", elemedex
     * entry, "How it works": the block is a linear projection, a short
     * convolution, the selective SSM and a multiplicative gate; sghael.github.io
     * Mamba page, "Simplifications and limits").  0: off, u is the scan input.
     * 1..4: u is the convolution's input x and the scan runs on
     *   u'[b,d,t] = silu(sum_{k<K} conv_weight[d,k] x[b,d,t-K+1+k] + conv_bias[d])
     * (causal, depthwise, width K = conv_width), computed in the scan's
     * prologue in fp32; u' takes u's place everywhere, the D u skip term
     * included, and never goes through memory unless u_out asks for it. */
    int32_t conv_width;
    /* (batch, dim, dstate) fp32 state before token 0, or NULL for zero.  It
     * may be the same buffer as last_state (the state is then continued in
     * place), but may overlap no other output. */
    const float* h0;
    const float* conv_weight;  /* (dim, conv_width) fp32 taps, oldest input first; required with conv */
    const float* conv_bias;    /* (dim) fp32, or NULL for none */
    /* (batch, dim, conv_width - 1) I/O type: the inputs x before token 0,
     * oldest first, or NULL for zeros. */
    const void* conv_state;
    /* (batch, dim, seqlen) I/O type output: the convolution's output u'
     * (rounded to the I/O type), or NULL to skip writing it. */
    void* u_out;
    /* Polls (about 256 ns apart) a CTA makes for the state handed over by the
     * CTA before it before giving up with SSM_ERR_TIMEOUT; 0: the default,
     * 2^22 (about a second).  Must be >= 0. */
    int32_t wait_limit;
    /* Test hook, 0 in normal use: nonzero makes every CTA withhold the flag
     * that publishes its hand-over, so that a CTA waiting for one gives up
     * after wait_limit polls, writes NaN to the outputs of the channels it
     * could not finish and leaves SSM_ERR_TIMEOUT for ssm_scan_fwd_status.
     * Nothing faults or hangs; the device stays usable. */
    int32_t test_skip_handoff;
} ssm_scan_opts;

/*
 * ssm_scan_fwd with options: the exact zero-order-hold input term, an initial
 * state, and the fused short convolution (see ssm_scan_opts).  Every other
 * argument, the workspace (ssm_scan_fwd_workspace_size gives its size for
 * these dims whatever the options) and the errors are those of ssm_scan_fwd;
 * an option out of range returns SSM_ERR_BAD_OPTION.
 */
SSM_API int ssm_scan_fwd_ex(const ssm_dims* dims, const ssm_scan_opts* opts,
                 const void* u, const void* delta, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, int delta_softplus,
                 void* y, float* last_state,
                 void* workspace, size_t workspace_bytes,
                 void* stream);

/*
 * The device-side outcome of the last ssm_scan_fwd / ssm_scan_fwd_ex call
 * that used `workspace` (workspace_bytes as passed to it).  Blocks: it
 * synchronises `stream` (the call's stream), then reads the workspace's
 * header.  Returns SSM_OK; SSM_ERR_TIMEOUT if a bounded hand-over wait gave
 * up (the outputs of the affected channels are NaN); SSM_ERR_DEVICE if a
 * -DSSM_DEBUG build's bounds check failed (that access was skipped); or
 * SSM_ERR_CUDA if the synchronisation or the copy failed.  A call whose
 * workspace size is 0 runs no bounded wait: pass workspace = NULL and
 * get SSM_OK.
 */
SSM_API int ssm_scan_fwd_status(const void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace ssm_scan_fwd needs for these sizes (may be 0).
 * Returns SSM_OK or a negative ssm_status (bad dims). */
SSM_API int ssm_scan_fwd_workspace_size(const ssm_dims* dims, size_t* bytes);

/*
 * Backward selective scan: the gradients for training.  Given dy =
 * dLoss/dy (and optionally dlast_state = dLoss/dlast_state) of a forward
 * scan with the same inputs and a zero initial state, writes the gradients
 * of the loss with respect to every input.  The forward pass stores nothing
 * for it; the backward pass recomputes the forward states on chip instead of
 * reading an expanded state from memory ("State Spaces, Selectively -
 * Mamba", papermap interactive explainer, "The hardware-aware scan": the
 * states are recomputed in the backward pass rather than stored).
 *
 *   dims, u, delta, A, B, C, D, z, delta_bias, delta_softplus
 *                  as for ssm_scan_fwd (device pointers)
 *   dy             (batch, dim, seqlen) fp32; required
 *   dlast_state    (batch, dim, dstate) fp32, or NULL for zero
 *   du, ddelta     (batch, dim, seqlen) fp32; required.  ddelta is the
 *                  gradient with respect to the raw delta (before bias and
 *                  softplus)
 *   dz             (batch, dim, seqlen) fp32; required when z is given
 *   dA             (dim, dstate) fp32; required
 *   dB, dC         (batch, seqlen, dstate) fp32; required
 *   dD, ddelta_bias (dim) fp32, or NULL to skip (ignored when D, resp.
 *                  delta_bias, is NULL)
 *   dh0            (batch, dim, dstate) fp32 gradient with respect to the
 *                  initial state, or NULL
 *   workspace      device scratch of ssm_scan_bwd_workspace_size() bytes
 *                  (the state at every 8th token; with chunks, the states
 *                  and adjoints at the chunk boundaries), 16-byte aligned
 *   stream         cudaStream_t to enqueue on
 *
 * All gradients are fp32 whatever the I/O type.  dA, dB, dC, dD and
 * ddelta_bias are sums over channels or over the batch, accumulated with
 * fp32 atomics: their rounding order, and so their last bits, may vary from
 * run to run.  The call clears them on `stream` first.  Returns SSM_OK or a
 * negative ssm_status.
 */
SSM_API int ssm_scan_bwd(const ssm_dims* dims,
                 const void* u, const void* delta, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, int delta_softplus,
                 const float* dy, const float* dlast_state,
                 float* du, float* ddelta, float* dz, float* dA,
                 float* dB, float* dC, float* dD, float* ddelta_bias, float* dh0,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * ssm_scan_bwd for the forward scan ssm_scan_fwd_ex runs with
 * ssm_scan_opts.h0 = h0 and ssm_scan_opts.input_term = input_term
 * ("Mamba remembers by forgetting, read closely", interactiveml.org: the
 * selective_scan recurrence started from a given state, and its exact
 * zero-order-hold discretisation).
 *   h0          (batch, dim, dstate) fp32 initial state (device), or NULL
 *               for zero.  The recomputed forward states start from h0, so
 *               every gradient includes its effect (dA and ddelta through
 *               h_(-1)); dh0 is the gradient with respect to h0.
 *   input_term  an ssm_input_term.  With SSM_INPUT_ZOH the input weight
 *               w = (exp(Delta A) - 1) / A of every state is differentiated
 *               too: dw/dDelta = exp(Delta A), dw/dA = (Delta exp(Delta A) -
 *               w) / A (Delta^2 / 2 at A = 0); out of range:
 *               SSM_ERR_BAD_OPTION.
 *   grad_io     the ssm_io_dtype of dy, du, ddelta and dz: SSM_IO_F32 (as
 *               for ssm_scan_bwd), or dims->io: dy is then read in the I/O
 *               type and du, ddelta, dz written in it (bf16: the fp32
 *               values rounded to nearest even once), so that a bf16
 *               training step needs no conversion pass; anything else:
 *               SSM_ERR_BAD_DTYPE.  dy, du, ddelta, dz must be aligned to
 *               that type's size.  dlast_state, dA, dB, dC, dD,
 *               ddelta_bias and dh0 are fp32 either way.
 * h0 = NULL, SSM_INPUT_DELTA_B and SSM_IO_F32 is ssm_scan_bwd.  The fused convolution
 * of ssm_scan_opts has no backward here.  Other arguments, workspace and
 * errors as for ssm_scan_bwd.
 */
SSM_API int ssm_scan_bwd_ex(const ssm_dims* dims,
                 const void* u, const void* delta, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, int delta_softplus,
                 const void* dy, const float* dlast_state, const float* h0,
                 int input_term, int grad_io,
                 void* du, void* ddelta, void* dz, float* dA,
                 float* dB, float* dC, float* dD, float* ddelta_bias, float* dh0,
                 void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace ssm_scan_bwd needs for these sizes (may be 0). */
SSM_API int ssm_scan_bwd_workspace_size(const ssm_dims* dims, size_t* bytes);

/*
 * ssm_scan_fwd on HOST buffers: every pointer (u, delta, A, B, C, D, z,
 * delta_bias, y, last_state) is host memory, with the layouts and meanings of
 * ssm_scan_fwd.  The call takes device memory on the current device with
 * cudaMallocAsync on `stream` (returned with cudaFreeAsync when the work is
 * done) and cuts the problem into slices (a batch row, or a range of its
 * channels) whose copies in, scans and copies out overlap on two internal
 * streams of the library joined to `stream` by events; one cudaMemcpyAsync
 * per tensor per slice.  It returns once everything is enqueued: the outputs
 * are valid, and the host buffers may be reused, when `stream` has completed
 * (e.g. cudaStreamSynchronize).  Pinned host memory (cudaHostAlloc,
 * cudaHostRegister) lets the copies run asynchronously and overlap; pageable
 * memory gives the same results with copies staged by the driver.  Each
 * slice's scan is ssm_scan_fwd over the slice, so the outputs equal those of
 * ssm_scan_fwd on device copies of the inputs bit for bit whenever the same
 * kernel serves both (it does except where the full problem would have taken
 * the chunked long-sequence schedule).  Returns SSM_OK or a negative
 * ssm_status; SSM_ERR_CUDA when an allocation or an enqueue fails (after
 * waiting for what was already enqueued).
 */
SSM_API int ssm_scan_fwd_host(const ssm_dims* dims,
                 const void* u, const void* delta, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, int delta_softplus,
                 void* y, float* last_state, void* stream);

/*
 * ssm_scan_fwd without a workspace argument, for callers that cannot allocate
 * device memory when they call the scan (for example an inference engine's
 * plugin confined to a memory plan fixed in advance, or a real-time path
 * where allocation is forbidden).  The source pages have no counterpart to
 * this entry point; it exists only for such callers.
 *
 * The scratch the scan needs lives in one fixed buffer inside the library,
 * ssm_scan_fwd_noalloc_max_scratch() bytes (4 MiB) on every device that loads
 * the library, held until the process exits.  The call allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine.  Problems whose
 * ssm_scan_fwd_workspace_size() exceeds the buffer are refused with
 * SSM_ERR_TOO_LARGE before anything is enqueued (at N = 16 the buffer holds
 * the carries of about 64,000 channels, e.g. batch 4 x 16000 channels).
 *
 * The first call on a device looks up the buffer's device address on that
 * device (cudaGetSymbolAddress, with the device current); make that first
 * call before any stream capture.  Every call shares the one buffer: calls
 * whose work overlaps on the GPU (different streams, or host threads racing)
 * race on it and give wrong results, so serialise them, e.g. on one stream.
 * The call clears the part of the buffer that must start at zero, on
 * `stream`, before the scan reads it; ssm_scan_fwd_noalloc_status reads the
 * status it leaves there.  Arguments, outputs and errors are otherwise those
 * of ssm_scan_fwd.
 */
SSM_API int ssm_scan_fwd_noalloc(const ssm_dims* dims,
                 const void* u, const void* delta, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, int delta_softplus,
                 void* y, float* last_state, void* stream);

/* Size in bytes of ssm_scan_fwd_noalloc's built-in scratch buffer. */
SSM_API size_t ssm_scan_fwd_noalloc_max_scratch(void);

/* ssm_scan_fwd_status for the last ssm_scan_fwd_noalloc call on the current
 * device (whose status lives in the built-in buffer): synchronises `stream`,
 * then reads it.  Allocates nothing. */
SSM_API int ssm_scan_fwd_noalloc_status(void* stream);

/*
 * One token of recurrent (generation) mode: the same update with L = 1,
 * starting from `state` and writing the new state back in place.
 * Recurrent mode costs the same for every token and keeps no cache that
 * grows ("Mamba", sghael.github.io, "Training without stepping token by
 * token"; papermap explainer, "The hardware-aware scan": inference is a pure
 * recurrence, O(1) per token).
 *
 *   state          (batch, dim, dstate) fp32, read and overwritten; required
 *   x, delta, z, y (batch, dim) I/O type (z may be NULL)
 *   B, C           (batch, dstate) I/O type
 *   A, D, delta_bias, delta_softplus: as for ssm_scan_fwd
 *
 * Running ssm_state_step for tokens 0..k-1 from a zero state reproduces the
 * scan's outputs y[..., t] and, after token k-1, the scan's last_state for
 * the first k tokens (up to fp32 rounding order).
 */
SSM_API int ssm_state_step(const ssm_dims* dims, float* state,
                   const void* x, const void* delta, const float* A,
                   const void* B, const void* C, const float* D, const void* z,
                   const float* delta_bias, int delta_softplus,
                   void* y, void* stream);

/*
 * Diagnostic, not part of the scan: enqueue a throughput probe of the
 * special-function unit's 2^x.  It launches `blocks` x `threads` threads
 * that each evaluate iters * 8 dependent 2^x chains and writes nothing
 * (`sink`, a device buffer of at least `threads` floats, is only named so the
 * work cannot be optimised away).  The caller times the launch on `stream`;
 * the number of 2^x evaluations is blocks * threads * iters * 8.
 * threads must be a multiple of 32 in [32, 1024]; blocks and iters >= 1.
 */
SSM_API int ssm_probe_ex2(int32_t blocks, int32_t threads, int32_t iters, float* sink,
                          void* stream);

/* Static text for a status code (never NULL). */
SSM_API const char* ssm_status_string(int status);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
SSM_API int ssm_version(void);

/* Identifier of the sources and compiler flags the library was built from
 * (a hash written in at build time; static text, never NULL).  The build
 * script compares it with the sources on disk to decide whether to rebuild. */
SSM_API const char* ssm_build_id(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
