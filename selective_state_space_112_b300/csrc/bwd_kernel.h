// Backward-pass kernels of the selective scan (bwd_kernel.cu): parameters and lookup.
#pragma once

#include "scan_tile.cuh"

namespace ssm {

struct BwdParams {
  const void* x;
  const void* delta;
  const void* z;         // nullable
  const float* A;        // (dim, N)
  const void* B;         // (batch, L, N) io dtype
  const void* C;
  const float* Dskip;    // nullable
  const float* bias;     // nullable
  const float* h_init;   // nullable: zeros
  const void* dout;      // (batch, L, dim) io dtype
  const float* dfinal;   // nullable: zeros
  void* dx;
  void* ddelta;
  void* dz;              // written when z is given
  float* dA;             // accumulated (zeroed by the host)
  float* dB;             // (batch, L, N), accumulated
  float* dC;
  float* dD;             // nullable, accumulated
  float* dbias;          // nullable, accumulated
  float* dh_init;        // nullable
  const float* ws_H;     // forward chunk aggregates (end states), chunks 0 .. nchunks-2
  const float* ws_S;     // forward chunk step sums
  float* ws_M;           // reverse aggregates of the sub-chunks of chunks 1 .. nchunks-1
  float* ws_S2;          // their step sums
  float* ws_ck;          // state checkpoints, (ceil(L / seg), batch, dim, S)
  int64_t batch, seqlen, dim;
  int dstate;
  int nchunks;
  int64_t chunk_len;
  int rsub;              // sub-chunks per chunk of the reverse aggregate pass
  int64_t rsub_len;      // chunk_len / rsub
  int delta_softplus;
};

typedef void (*BwdFn)(BwdParams);

struct BwdKernels {
  BwdFn reverse_aggregate = nullptr;
  BwdFn main = nullptr;
  int seg = 0;  // steps per checkpoint segment
};

// S = padded state count (2, 4, 8 or 16), one lane per channel.
BwdKernels lookup_bwd(int io_bf16, int S);

}  // namespace ssm
