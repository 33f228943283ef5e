// Recurrent step (sequence length 1) of the selective scan: h <- Abar h + Bbar x from
// a stored state (Bbar = step B, or the exact ZOH (Abar - 1) / A B), y = C . h + D x,
// gated ("State-space models", section "Recurrence and convolution": the recurrent
// view generates one token per step with constant work; the state (batch, dim, N) is
// read and written once).
//
// Design: the work is one pass over the state, so the kernel is laid out for the
// state's bandwidth: one thread per (batch row, channel, 4 consecutive states), the
// state moved as one 16-byte vector per thread (G = padded N / 4 consecutive threads
// per channel, whole 64-byte rows per channel for N = 16).  Each thread forms the
// channel's step size itself (G-fold redundant scalar work, free next to the state
// traffic), and the G shares of C . h meet by warp shuffles.  With the Mamba-block
// prologue (CONV) the input is u = silu(w0 x + w1 x_{-1} + w2 x_{-2} + w3 x_{-3} + b)
// from the stored three-input history, which the channel's first thread then shifts.
#include <cuda_runtime.h>

#include "kernel_table.cuh"

namespace ssm {

template <typename IO, int G, bool LTI, bool CONV>
__global__ void __launch_bounds__(256) step_kernel(const __grid_constant__ TmaMaps, const ScanParams p) {
  constexpr bool MFORM = LTI || !IO::kFastDecay;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int g = threadIdx.x % G;
  const int64_t ch = gid / G;  // (batch row, channel) index
  const int64_t Dm = p.dim;
  const int N = p.dstate;
  const bool valid = ch < p.batch * Dm;
  const int64_t cc = valid ? ch : 0;
  const int64_t b = cc / Dm, d = cc - b * Dm;

  float xv = IO::load(p.x, cc);  // x[b, 0, d]: (batch, 1, dim) is row-major (batch, dim)
  [[maybe_unused]] float hist[3] = {0.f, 0.f, 0.f};  // x_{-3}, x_{-2}, x_{-1}
  const float x_raw = xv;
  if (CONV) {
    if (p.conv_hist_in)
      for (int j = 0; j < 3; ++j) hist[j] = p.conv_hist_in[cc * 3 + j];
    const float4 w = *reinterpret_cast<const float4*>(p.conv_w + d * 4);
    const float pre = fmaf(w.x, x_raw, fmaf(w.y, hist[2], fmaf(w.z, hist[1], fmaf(w.w, hist[0],
                                                                               p.conv_b ? p.conv_b[d] : 0.f))));
    xv = silu(pre);
  }
  const float v = IO::load(p.delta, cc) + (p.bias ? p.bias[d] : 0.f);
  const float dt = p.delta_softplus ? softplus<std::is_same<IO, F32>::value>(v) : v;

  const int n0 = 4 * g;
  float hv[4], a[4], bv[4], cv[4];
  const bool vec = (N % 4 == 0) && n0 < N;  // whole 16-byte quads
  const int64_t srow = cc * N;
  if (vec) {
    const float4 h4 = p.h_init ? *reinterpret_cast<const float4*>(p.h_init + srow + n0)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 a4 = *reinterpret_cast<const float4*>(p.A + d * N + n0);
    hv[0] = h4.x; hv[1] = h4.y; hv[2] = h4.z; hv[3] = h4.w;
    a[0] = a4.x; a[1] = a4.y; a[2] = a4.z; a[3] = a4.w;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + j;
      hv[j] = (n < N && p.h_init) ? p.h_init[srow + n] : 0.f;
      a[j] = n < N ? p.A[d * N + n] : 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int n = n0 + j;
    if (LTI) {
      bv[j] = n < N ? static_cast<const float*>(p.B)[d * N + n] : 0.f;
      cv[j] = n < N ? static_cast<const float*>(p.C)[d * N + n] : 0.f;
    } else {
      bv[j] = n < N ? IO::load(p.B, b * N + n) : 0.f;
      cv[j] = n < N ? IO::load(p.C, b * N + n) : 0.f;
    }
  }
  float y = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // decay: Abar - 1 by accurate expm1 (fp32 and constant-coefficient inputs), else Abar
    const float e = MFORM ? expm1f(dt * a[j]) : ex2(dt * a[j] * kLog2e);
    // input factor: step (fused scan) or exact ZOH (Abar - 1) / A, step where A = 0
    const float q = p.bbar_mode ? (a[j] != 0.f ? (MFORM ? e : e - 1.f) / a[j] : dt) : dt;
    const float bx = q * xv * bv[j];
    hv[j] = MFORM ? hv[j] + fmaf(e, hv[j], bx) : fmaf(e, hv[j], bx);
    y = fmaf(cv[j], hv[j], y);
  }
#pragma unroll
  for (int off = 1; off < G; off <<= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
  if (CONV) __syncwarp();  // every thread has read the history before it is shifted

  if (!valid) return;
  if (CONV && g == 0 && p.conv_state_out) {
    p.conv_state_out[cc * 3] = hist[1];
    p.conv_state_out[cc * 3 + 1] = hist[2];
    p.conv_state_out[cc * 3 + 2] = x_raw;
  }
  if (p.final_state) {
    if (vec) {
      *reinterpret_cast<float4*>(p.final_state + srow + n0) = make_float4(hv[0], hv[1], hv[2], hv[3]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (n0 + j < N) p.final_state[srow + n0 + j] = hv[j];
    }
  }
  if (g == 0) {
    y = fmaf(p.Dskip ? p.Dskip[d] : 0.f, xv, y);
    if (p.z) y *= silu(IO::load(p.z, cc));
    IO::store(p.out, cc, y);
  }
}

template <typename IO, bool LTI, bool CONV>
KernelInfo step_info(int G) {
  KernelInfo k;
  switch (G) {
    case 1: k.fn = step_kernel<IO, 1, LTI, CONV>; break;
    case 2: k.fn = step_kernel<IO, 2, LTI, CONV>; break;
    case 4: k.fn = step_kernel<IO, 4, LTI, CONV>; break;
    case 8: k.fn = step_kernel<IO, 8, LTI, CONV>; break;
    case 16: k.fn = step_kernel<IO, 16, LTI, CONV>; break;
    default: return k;
  }
  k.nt = 256;
  k.ch = 256 / G;
  k.t = 1;
  k.smem = 0;
  return k;
}

KernelInfo lookup_step(int io_bf16, bool lti, int G, bool conv) {
  if (conv) {  // the prologue form: time-varying B and C
    if (lti) return KernelInfo();
    return io_bf16 ? step_info<BF16, false, true>(G) : step_info<F32, false, true>(G);
  }
  if (io_bf16) return lti ? step_info<BF16, true, false>(G) : step_info<BF16, false, false>(G);
  return lti ? step_info<F32, true, false>(G) : step_info<F32, false, false>(G);
}

}  // namespace ssm
