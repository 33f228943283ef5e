/*
 * ssm_ssd.h -- C ABI of the B300 (sm_103a) Mamba-2 state-space-duality (SSD)
 * layer, forward.
 *
 * The operation (pages "State-space models", rayaq.ca, section "The parallel
 * scan": Mamba-2 restricts A to a scalar times the identity per head, which turns
 * the scan into blocks of matrix products on the tensor cores; "State Space
 * Models: Mamba and Beyond", aicomputerinstitute.com, section "Beyond Mamba:
 * state-space duality and hybrid architectures": one scalar A per attention-style
 * head, larger state sizes N; "Structured State Space Models and Mamba",
 * llms.blog, section "State Space Duality and Mamba-2": the same map is the
 * masked attention Y = (L o (C B^T)) V with a 1-semiseparable decay mask L).  For
 * every batch row b, head h (reading group g = h / (nheads / ngroups)), step t,
 * channel p of the head and state n:
 *
 *   step_t   = softplus(dt[b,t,h] + dt_bias[h])     (or without softplus)
 *   h_t[p,n] = exp(step_t A[h]) h_{t-1}[p,n] + step_t B[b,t,g,n] x[b,t,h,p]
 *   y_t[p]   = sum_n C[b,t,g,n] h_t[p,n] + D[h] x[b,t,h,p]
 *   out      = y_t * silu(z[b,t,h,p])               when a gate z is given
 *
 * It is the S6 scan of ssm_scan.h with the decay, the step and D tied per head
 * and B, C shared by the heads of a group.  The kernel evaluates it chunk by
 * chunk (128 steps) in the dual form: within a chunk the masked product
 * (L o C B^T)(step x) on the 5th-generation tensor cores (tcgen05, accumulators in
 * tensor memory, inputs staged by TMA); across chunks the (P, N) state of the
 * head, carried in tensor memory.  When the (batch row, head, 32-channel block)
 * sequences outnumber the CTAs the GPU holds at once, each sequence is cut into 2
 * or 4 parts of consecutive chunks taken in order by persistent CTAs; a part hands
 * its end state (fp32, P x N per block) to the next through a workspace that the
 * call takes from the library's stream-ordered pool and returns (SSM_ERR_NOMEM if it
 * cannot), with a release flag the next part waits for (bounded, 2 s).  The result
 * is bitwise the same for any number of parts.
 *
 * Conventions as in ssm_scan.h: device pointers on the current device,
 * contiguous row-major, 16-byte aligned, owned by the caller; the call enqueues
 * on `stream` and returns; status codes are ssm_status; no CPU fallback;
 * identical inputs give bitwise-identical outputs.
 */
#ifndef SSM_SSD_H
#define SSM_SSD_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#include "ssm_scan.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int64_t batch;     /* b >= 1 (at most 65535)                                    */
  int64_t seqlen;    /* L >= 0; L == 0 only writes final_state (h_{-1} or zeros)  */
  int64_t nheads;    /* H >= 1                                                    */
  int64_t headdim;   /* P, channels per head; this build: 64                      */
  int64_t ngroups;   /* G >= 1, dividing H; heads h*G/H .. share B and C          */
  int64_t dstate;    /* N; this build: 64, 128 or 256                             */
  ssm_dtype io_dtype;   /* x, dt, B, C, z, out; this build: SSM_BF16               */
  int32_t dt_softplus;  /* 1: step = softplus(dt + dt_bias); 0: step = dt + dt_bias */
  int32_t state_in;     /* 1: final_state holds h_{-1} on entry                     */
  int32_t reserved;     /* must be 0                                               */
} ssm_ssd_dims;

/*
 * Mamba-2 SSD forward.
 *   x          : (batch, seqlen, nheads, headdim), io dtype
 *   dt         : (batch, seqlen, nheads), io dtype, the raw step before bias
 *   A          : (nheads) fp32, one decay rate per head (negative for a stable layer)
 *   B, C       : (batch, seqlen, ngroups, dstate), io dtype
 *   D          : (nheads) fp32 or NULL (no skip term)
 *   z          : (batch, seqlen, nheads, headdim), io dtype, or NULL (no gate)
 *   dt_bias    : (nheads) fp32 or NULL
 *   out        : (batch, seqlen, nheads, headdim), io dtype; must not overlap an input
 *   final_state: (batch, nheads, headdim, dstate) fp32 or NULL; with
 *                dims->state_in it is read first as h_{-1} (required then); it is
 *                overwritten with h_{L-1}.  Must not overlap any other tensor.
 * x, dt, A, B, C and out are required when seqlen > 0 (an empty tensor may come
 * with a NULL address).
 * Returns SSM_OK or: SSM_ERR_NULL (a required pointer or dims is NULL),
 * SSM_ERR_DIMS (a size out of range, ngroups not dividing nheads, an unknown flag
 * value, state_in without final_state), SSM_ERR_ALIGN, SSM_ERR_OVERLAP,
 * SSM_ERR_UNSUPPORTED (io dtype, headdim or dstate this build does not cover),
 * SSM_ERR_CUDA (launch failure or no usable device), SSM_ERR_NOMEM (the workspace
 * of a call whose sequences are cut into parts).  A wait inside the kernel
 * that does not end within 2 s leaves the call's outputs undefined; the kernel
 * then frees what it holds and returns, and ssm_check_status reports
 * SSM_ERR_TIMEOUT.
 * Arithmetic: bf16 operands on the tensor cores with fp32 accumulation.  The
 * operands formed inside the kernel (the masked decay matrix, the decay-weighted
 * inputs and the carried state, all fp32) enter as a pair of bf16 values (value
 * and remainder), about 16 significant bits; step sizes, decays and the state
 * are kept in fp32.
 */
int ssm_ssd_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                const float* D, const void* z, const float* dt_bias, void* out,
                float* final_state, const ssm_ssd_dims* dims, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SSD_H */
