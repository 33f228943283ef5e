/*
 * ssm_scan.h -- C ABI of the B300 (sm_103a) Mamba S6 selective scan (forward,
 * the forward with the Mamba-block prologue, and the backward pass).
 *
 * The operation (pages "State-space models", rayaq.ca, sections
 * "Discretization", "Mamba: selection", "The parallel scan" and
 * "Implementation"; "Structured State Space Models and Mamba", llms.blog,
 * sections "Discretization Mechanics", the S6 section and "The GPU Memory
 * Hierarchy and Kernel Fusion"): for every batch row b, channel d, step t and
 * state n,
 *
 *   step_t  = softplus(delta[b,t,d] + delta_bias[d])   (or without softplus)
 *   Abar    = exp(step_t * A[d,n])                      zero-order hold, diagonal A
 *   Bbar x  = step_t * B[.,t,n] * x[b,t,d]              the fused scan's input term
 *             (bbar_mode 1: (Abar - 1) / A[d,n] * B[.,t,n] * x[b,t,d], exact ZOH)
 *   h_t[n]  = Abar * h_{t-1}[n] + Bbar x                h_{-1} = 0 or a given state
 *   y_t     = sum_n C[.,t,n] h_t[n] + D[d] x[b,t,d]
 *   out     = y_t * silu(z[b,t,d])                      when a gate z is given
 *
 * The expanded state (batch, L, dim, N) never reaches device memory: only out
 * and the final state are written.
 *
 * Conventions for every entry point:
 *  - Pointers to tensors are DEVICE pointers on the current CUDA device,
 *    contiguous row-major, 16-byte aligned, owned by the caller.  The library
 *    never frees or retains them past the call's completion on `stream`.
 *  - Calls are asynchronous: they enqueue work on `stream` (a cudaStream_t;
 *    NULL is the legacy default stream) and return once it is enqueued.
 *  - Return value: SSM_OK (0) or a negative ssm_status; argument errors are
 *    detected on the host before anything is enqueued.
 *  - No CPU fallback: without a usable GPU every call fails with SSM_ERR_CUDA.
 *  - The forward entry points are deterministic: identical inputs give
 *    bitwise-identical outputs.  The backward pass is not: its sums over
 *    channels use fp32 atomic additions, whose rounding order varies.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of x, delta, z, out and of time-varying B, C. */
typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

/* Layout of B and C. */
typedef enum {
  SSM_BC_TIME_VARYING = 0, /* (batch, seqlen, dstate), io dtype, shared by all channels
                              ("Mamba: selection": all channels share B_t and C_t) */
  SSM_BC_PER_CHANNEL = 1   /* (dim, dstate), fp32, constant in time (an LTI system,
                              "Recurrence and convolution") */
} ssm_bc_layout;

typedef enum {
  SSM_OK = 0,
  SSM_ERR_NULL = -1,        /* a required pointer is NULL */
  SSM_ERR_DIMS = -2,        /* batch, dim or dstate <= 0, seqlen < 0, dstate > 64,
                               an unknown enum value, or state_in with final_state NULL */
  SSM_ERR_ALIGN = -3,       /* a tensor pointer is not 16-byte aligned */
  SSM_ERR_UNSUPPORTED = -4, /* a mode this build does not implement */
  SSM_ERR_CUDA = -5,        /* a CUDA runtime error (no device, launch failure, ...) */
  SSM_ERR_OVERLAP = -6,     /* out or final_state overlaps another tensor */
  SSM_ERR_NOMEM = -7,       /* the workspace could not be allocated */
  SSM_ERR_DEVICE = -8,      /* a kernel reported an internal inconsistency */
  SSM_ERR_TIMEOUT = -9,     /* a kernel gave up a bounded wait for its own copies */
  SSM_ERR_SCRATCH = -10     /* ssm_selective_scan_fwd_noalloc: the call needs more than
                               SSM_NOALLOC_SCRATCH_BYTES of workspace */
} ssm_status;

typedef struct {
  int64_t batch;          /* b  >= 1 */
  int64_t seqlen;         /* L  >= 0; L == 0 only sets final_state (see below) */
  int64_t dim;            /* D  >= 1, channels (d_inner) */
  int64_t dstate;         /* N  in 1..64 */
  int32_t io_dtype;       /* ssm_dtype */
  int32_t bc_layout;      /* ssm_bc_layout */
  int32_t delta_softplus; /* 1: step = softplus(delta + bias); 0: step = delta + bias */
  int32_t state_in;       /* 1: final_state holds h_{-1} on entry (resume / recurrent step) */
  int32_t bbar_mode;      /* 0: Bbar = step * B (the fused scan's input term);
                             1: exact zero-order hold, Bbar = (exp(step A) - 1) / A * B
                             (the limit step * B where A = 0) */
  int32_t reserved;       /* must be 0 */
} ssm_dims;

/*
 * Selective-scan forward.
 *
 *   x, delta, z, out : (batch, seqlen, dim), io dtype
 *   A                : (dim, dstate) fp32, the diagonal of each channel's A (negative
 *                      for a stable system; any value is accepted)
 *   B, C             : see ssm_bc_layout
 *   D                : (dim) fp32 skip weights, or NULL (no skip)
 *   z                : gate input, or NULL (no gate)
 *   delta_bias       : (dim) fp32, added before softplus, or NULL (no bias)
 *   final_state      : (batch, dim, dstate) fp32, or NULL when state_in == 0.  On
 *                      return (in stream order) it holds h_{L-1}; with state_in it is
 *                      read first as h_{-1}.  With seqlen == 0 it keeps h_{-1}
 *                      (state_in) or is zero-filled.
 * out must not overlap any input; final_state must not overlap any other tensor.
 * The state is accumulated in fp32 for both io dtypes; bf16 outputs are rounded to
 * nearest even.  Long sequences are split into chunks scanned in parallel; the
 * chunk carries live in a workspace that the library takes from its own
 * stream-ordered memory pool on `stream` and returns to it in stream order.
 */
int ssm_selective_scan_fwd(const void* x, const void* delta, const float* A,
                           const void* B, const void* C, const float* D,
                           const void* z, const float* delta_bias, void* out,
                           float* final_state, const ssm_dims* dims,
                           cudaStream_t stream);

/*
 * Selective-scan forward with the Mamba-block prologue fused into its load stage
 * (page "State-space models", section "Mamba: selection", the block description:
 * a depthwise causal convolution of width 4 and a silu on the branch that feeds the
 * SSM).  Per batch row b, channel d and step t:
 *
 *   u[b,t,d] = silu( sum_{k=0..3} conv_w[d,k] * x[b,t-k,d] + conv_b[d] )
 *
 * and the scan of ssm_selective_scan_fwd then runs on u in place of x (both the
 * input term and the D skip take u).  u is formed in fp32 and never stored.
 *
 *   conv_w     : (dim, 4) fp32; tap k multiplies the input k steps back
 *   conv_b     : (dim) fp32, or NULL (no bias)
 *   conv_state : (batch, dim, 3) fp32, or NULL.  With dims->state_in it is read
 *                first as the three inputs before the sequence (x[-3], x[-2],
 *                x[-1], oldest first; zeros without state_in).  On return (in
 *                stream order) it holds the last three inputs of the sequence,
 *                extended by that history when seqlen < 3 (seqlen == 0 keeps it,
 *                or zero-fills it without state_in).  It must not overlap any
 *                other tensor.
 * All other arguments as ssm_selective_scan_fwd.  Built for time-varying B and C
 * (SSM_BC_TIME_VARYING) and bbar_mode 0; other forms return SSM_ERR_UNSUPPORTED.
 * A long sequence run in pieces with state_in and both states carried gives the
 * result of one call over the whole sequence.
 */
int ssm_conv_selective_scan_fwd(const void* x, const float* conv_w, const float* conv_b,
                                float* conv_state, const void* delta, const float* A,
                                const void* B, const void* C, const float* D,
                                const void* z, const float* delta_bias, void* out,
                                float* final_state, const ssm_dims* dims,
                                cudaStream_t stream);

/*
 * Selective-scan backward: the gradients of ssm_selective_scan_fwd (bbar_mode 0,
 * time-varying B and C, dstate <= 16) with the expanded state rebuilt rather than
 * stored (page "State-space models", section "The parallel scan": Mamba's kernel
 * recomputes the state in the backward pass).  With gy_t = dout_t * silu(z_t) and
 * the adjoint state lam_t = C_t gy_t + Abar_{t+1} lam_{t+1} (lam_{L-1} = C gy +
 * dfinal_state), for every b, t, d, n:
 *
 *   dx      = sum_n lam step B + gy D          ddelta = d(step)/d(delta) * (
 *   dA[d,n] = sum_{b,t} lam h_{t-1} Abar step       sum_n lam (h_{t-1} Abar A + B x) )
 *   dB[b,t,n] = sum_d lam step x               dC[b,t,n] = sum_d gy h_t
 *   dD[d]   = sum_{b,t} gy x                   ddelta_bias[d] = sum_{b,t} ddelta
 *   dz      = dout y silu'(z)                  dh_init = Abar_0 lam_0
 *
 *   x, delta, A, B, C, D, z, delta_bias : as ssm_selective_scan_fwd (dims likewise;
 *                  dims->state_in is not used: h_init says whether there is one)
 *   h_init       : (batch, dim, dstate) fp32 initial state, or NULL (zeros)
 *   dout         : (batch, seqlen, dim) io dtype, gradient of out
 *   dfinal_state : (batch, dim, dstate) fp32 gradient of the final state, or NULL
 *   dx, ddelta   : (batch, seqlen, dim) io dtype, written
 *   dz           : (batch, seqlen, dim) io dtype, written; required when z is given
 *   dA           : (dim, dstate) fp32; dB, dC: (batch, seqlen, dstate) fp32;
 *   dD, ddelta_bias : (dim) fp32 or NULL -- these sums are overwritten (zeroed first)
 *   dh_init      : (batch, dim, dstate) fp32 or NULL
 * No output may overlap an input or another output.  Sums over channels are
 * accumulated with fp32 atomic additions, so their rounding order is not fixed.
 * Other forms return SSM_ERR_UNSUPPORTED.  Long sequences are chunked; the
 * workspace (chunk carries and a state checkpoint every 4 steps:
 * ceil(seqlen / 4) * batch * dim * padded dstate fp32) comes from the library's
 * stream-ordered pool.
 */
int ssm_selective_scan_bwd(const void* x, const void* delta, const float* A,
                           const void* B, const void* C, const float* D,
                           const void* z, const float* delta_bias,
                           const float* h_init, const void* dout,
                           const float* dfinal_state, void* dx, void* ddelta,
                           float* dA, float* dB, float* dC, float* dD, void* dz,
                           float* ddelta_bias, float* dh_init, const ssm_dims* dims,
                           cudaStream_t stream);

/* Bytes of the fixed workspace of ssm_selective_scan_fwd_noalloc (16 MiB). */
#define SSM_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * Selective-scan forward that allocates no device memory.
 *
 * The source pages have no counterpart to this entry point: it exists for callers that
 * cannot let a library allocate device memory (an application whose arena owns all
 * device memory, a serving loop that allows no allocation after warm-up, an allocator
 * that must not be entered from the calling thread).  Arguments, layouts, results and
 * errors are those of ssm_selective_scan_fwd, with these differences:
 *  - The chunk-carry workspace lives in one fixed device array of
 *    SSM_NOALLOC_SCRATCH_BYTES inside the library, present on every GPU that loads it
 *    until the process exits.  When the automatic chunk count would need more (long
 *    sequences with many chunks: about (chunks - 1) * batch * dim * (2 dstate + 1) * 4
 *    bytes, plus batch * dim * dstate * 4 with state_in), the call uses fewer chunks,
 *    down to one (no workspace).  A chunk count forced with ssm_set_option("chunks")
 *    whose workspace does not fit returns SSM_ERR_SCRATCH and launches nothing.
 *  - The first call on a device asks the runtime for the array's address (once per
 *    device, with that device current); make that first call before any stream
 *    capture.
 *  - All calls on a device share the array and the array keeps the last call's
 *    contents; each call clears the part that must start at zero (its chunk-carry
 *    flags) with a cudaMemsetAsync on `stream` before its kernel.  Calls that may
 *    overlap on the GPU (different streams without ordering) race on it: order them
 *    on one stream.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 */
int ssm_selective_scan_fwd_noalloc(const void* x, const void* delta, const float* A,
                                   const void* B, const void* C, const float* D,
                                   const void* z, const float* delta_bias, void* out,
                                   float* final_state, const ssm_dims* dims,
                                   cudaStream_t stream);

/* Waits for `stream` and returns SSM_OK, SSM_ERR_CUDA if the stream reports a CUDA
 * error, or SSM_ERR_TIMEOUT / SSM_ERR_DEVICE if a kernel of this library raised the
 * device status word since the last check (the word is then cleared).  Every wait
 * inside a kernel is bounded: a copy that never lands ends the kernel with
 * SSM_ERR_TIMEOUT instead of hanging the GPU. */
int ssm_check_status(cudaStream_t stream);

/* Static description of a status code. Never NULL. */
const char* ssm_status_string(int code);

/* Returns the unused memory of the library's per-device pools to the driver.
 * Waits for all work on every device the library has used.  The pools keep the
 * blocks that calls free, so that repeated calls allocate nothing; after a large
 * backward call (its state checkpoints take ceil(seqlen / 4) * batch * dim *
 * padded dstate * 4 bytes, 5.4 GB for a 131072-step, 2560-channel layer) this
 * gives that memory back. */
int ssm_release_workspace(void);

/* Device memory the library's pool holds on the current device (bytes reserved from
 * the driver, in use or kept for reuse; 0 before the first pooled call), or a
 * negative ssm_status. */
int64_t ssm_workspace_reserved_bytes(void);

/* Number of kernels this library has launched in this process. */
uint64_t ssm_kernel_launches(void);

/*
 * Tuning knobs (process-wide, for benchmarks and tests):
 *   "chunks"        force the number of sequence chunks (0 = automatic)
 *   "min_chunk_len" smallest automatic chunk length in steps (default 64)
 *   "lanes"         force the lanes per channel G (1, 2 or 4; 0 = automatic).
 *                   Each channel's states are split over G threads.  A G the build
 *                   lacks for this state count makes calls fail with
 *                   SSM_ERR_UNSUPPORTED.
 *   "lane_threads"  automatic G for bf16 inputs: the fewest lanes giving
 *                   batch * dim * G >= this (default 32768); G = 1 when no G reaches
 *                   it.  fp32 inputs use G = 1.
 *   "ctas_per_sm"   automatic chunking: cut the sequence only when the channels give
 *                   fewer than this many CTAs per SM (default 3); the chunk count then
 *                   fills that many CTAs per SM in one wave
 *   "pow_path"      1 (default): channels whose A row is (n+1) * A[d,0] take one
 *                   exponential per step and form the other decays as its powers;
 *                   0: always one exponential per state
 *   "tma"           1 (default): use the TMA-pipelined kernel where tensor maps can
 *                   describe the tensors; 0: always the generic kernel
 *   "inject_stall"  failure injection for tests (0 = off): with value k, the copy
 *                   producer of every CTA stops before its tile k - 1, so the waits
 *                   for that tile run out (every wait of a kernel is bounded by 2 s);
 *                   the kernels return and ssm_check_status reports SSM_ERR_TIMEOUT.
 *                   Leave it 0 otherwise.
 *   "one_launch"    0 (default): the cross-chunk carry is an aggregate pass (each
 *                   chunk's end state from zero and its step sum) and a fold in the
 *                   output pass, two launches; 1: one launch with decoupled lookback
 *                   (pages "State-space models", The parallel scan; "Structured State
 *                   Space Models and Mamba", Hardware-Aware Parallel Associative Scan):
 *                   chunks take tickets from a counter, publish their aggregates with
 *                   flags and fold their predecessors' aggregates in a fixed order, so
 *                   results stay bitwise repeatable.  Flag waits are bounded (2 s,
 *                   SSM_ERR_TIMEOUT).
 *   "hold_chunk"    failure injection for tests (0 = off, with "one_launch" 1): with
 *                   value k, chunk k - 1 never publishes its aggregate, so the flag
 *                   waits of its successors run out.  Leave it 0 otherwise.
 *   "ssd_legacy"    0 (default): ssm_ssd_fwd runs the tcgen05 kernel; 1: the earlier
 *                   mma.sync kernel (kept for comparison).
 *   "ssd_split"     0 (default): ssm_ssd_fwd chooses how many parts each sequence is
 *                   cut into (1 when the sequences fit the resident CTAs); 1, 2 or 4
 *                   force it (at most the chunks of the sequence).  Other values:
 *                   SSM_ERR_DIMS.
 *   "ssd_hold_part" failure injection for tests (0 = off): with value k and the
 *                   sequences cut into parts, the first part of unit k - 1 never
 *                   hands its state over, so the wait of the next part runs out (2 s,
 *                   SSM_ERR_TIMEOUT).  Leave it 0 otherwise.
 * Returns SSM_ERR_DIMS for an unknown name or a negative value.
 */
int ssm_set_option(const char* name, int64_t value);

/*
 * Per-kernel device timing.  While enabled, every launch is bracketed by CUDA events
 * recorded on the launch stream.  ssm_profile_read() waits for them, writes up to
 * `max` rows (kernel name, launches, total milliseconds) and clears the record; it
 * returns the number of kernel kinds seen, or a negative ssm_status.
 */
int ssm_profile_enable(int on);
int ssm_profile_read(const char** names, int64_t* launches, double* total_ms, int max);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
