// Library-internal entry shared by the public C entry points of libssmscan.
#pragma once

#include <stddef.h>

#include "ssm_scan.h"

namespace ssm_internal {

// Runs one selective-scan call.  With scratch == nullptr the chunk-carry workspace
// comes from the library's memory pool; otherwise it is taken from the caller's
// scratch_bytes of device memory at `scratch` and nothing is allocated.  conv: the
// block prologue on x, or null.
// The Mamba-block prologue applied to x before the scan: taps (dim, 4), bias (dim)
// or null, and the (batch, dim, 3) input history (read with dims->state_in, written
// when not null).
struct ConvPrologue {
  const float* w;
  const float* b;
  float* state;
};

int scan_forward(const void* x, const void* delta, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* delta_bias, void* out,
                 float* final_state, const ssm_dims* dims, cudaStream_t stream, void* scratch,
                 size_t scratch_bytes, const ConvPrologue* conv);

// Counts one kernel launch of the library (read by ssm_kernel_launches).
void count_launch();

// The library's stream-ordered memory pool of device dev (workspaces are taken from it
// with cudaMallocFromPoolAsync and returned with cudaFreeAsync).
cudaError_t workspace_pool(int dev, cudaMemPool_t* out);

// Device address of the status word the kernels raise (read by ssm_check_status), or
// null if the runtime cannot give it.
int* status_word();

// Options of the SSD layer (ssm_set_option forwards names it does not know): returns
// true if the name is one of them.
bool set_ssd_option(const char* name, int64_t value);

}  // namespace ssm_internal
