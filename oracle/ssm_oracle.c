/*
 * Float64 CPU oracle for the Mamba (S6) selective scan and the Mamba-2 SSD layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * reference that the CUDA kernels are checked against.  Only the test suite,
 * the package smoke check and the benchmark's CPU-baseline leg may load it;
 * the product path never calls it and shares no code, header or table with
 * it.  It steps the recurrence directly, in the order the pages state it,
 * with no blocking, fusion or reordering.
 *
 * Sources (web pages on state-space models and Mamba):
 *  - "State-space models" (rayaq.ca), sections "Discretization" (Euler,
 *    bilinear, ZOH rules), "Recurrence and convolution" (unrolled sum from
 *    h_{-1} = 0, kernel K_k = C Abar^k Bbar), "Mamba: selection" (softplus
 *    step size, diagonal A, B_t and C_t shared by all channels) and
 *    "Implementation" (shapes x, delta: (batch, L, D); A: (D, N);
 *    B, C: (batch, L, N); h: (batch, D, N); the note that the fused scan uses
 *    Bbar = delta * B).
 *  - "Structured State Space Models and Mamba" (llms.blog), sections
 *    "Discretization Mechanics" (h_k = Abar h_{k-1} + Bbar x_k,
 *    y_k = C h_k + D x_k), "The Linear Time-Invariance Bottleneck and the
 *    Selective State Space (S6)" (Delta_t = softplus(Linear(x_t) + bias))
 *    and "Hardware-Aware Parallel Associative Scan".
 *
 * Every floating-point value is widened to double by the caller (the stored
 * fp32 or bf16 values, exactly); all arithmetic here is IEEE double with the
 * C library's exp / expm1 / log1p.
 *
 * Parity pins: every function here is pinned by tests/test_oracle_pins.py
 * against the pages' worked examples, closed forms, the LTI convolution
 * identity and brute force on tiny inputs.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(v) = log(1 + e^v), written so that neither branch overflows.
 * ("State-space models", section "Mamba: selection": softplus keeps the step
 * positive.) */
double oracle_softplus(double v) {
  return fmax(v, 0.0) + log1p(exp(-fabs(v)));
}

/* silu(z) = z * sigmoid(z), the output gate of the Mamba block
 * ("State-space models", section "Mamba: selection", block description). */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* Scalar discretisation of h' = a h + b u with step dt
 * ("State-space models", section "Discretization"):
 *   rule 0  Euler:             abar = 1 + dt a,            bbar = dt b
 *   rule 1  bilinear (Tustin): abar = (1 + dt a/2)/(1 - dt a/2),
 *                              bbar = dt b / (1 - dt a/2)
 *   rule 2  ZOH, exact:        abar = e^{dt a},            bbar = (e^{dt a} - 1)/a * b
 *                              (limit dt b as a -> 0)
 *   rule 3  ZOH with the simplified input term used by the fused scan:
 *                              abar = e^{dt a},            bbar = dt b
 * Returns 0, or -1 for an unknown rule. */
int oracle_discretize_scalar(double a, double b, double dt, int rule,
                             double* abar, double* bbar) {
  switch (rule) {
    case 0:
      *abar = 1.0 + dt * a;
      *bbar = dt * b;
      return 0;
    case 1: {
      double left = 1.0 - 0.5 * dt * a;
      *abar = (1.0 + 0.5 * dt * a) / left;
      *bbar = dt * b / left;
      return 0;
    }
    case 2:
      *abar = exp(dt * a);
      *bbar = (a != 0.0) ? expm1(dt * a) / a * b : dt * b;
      return 0;
    case 3:
      *abar = exp(dt * a);
      *bbar = dt * b;
      return 0;
    default:
      return -1;
  }
}

/*
 * Selective scan, stepped directly.
 *
 * Layouts (row-major, contiguous):
 *   x, delta, z, out : (batch, seqlen, dim)
 *   A                : (dim, dstate)
 *   B, C             : (batch, seqlen, dstate) when per_channel_bc == 0
 *                      (time-varying, shared by every channel of a batch row)
 *                      (dim, dstate) when per_channel_bc == 1 (LTI)
 *   D, delta_bias    : (dim), either may be NULL (treated as 0)
 *   z                : may be NULL (no gate)
 *   state            : (batch, dim, dstate); read as h_{-1} when state_in,
 *                      otherwise h_{-1} = 0; always overwritten with h_{L-1}.
 *                      May be NULL when state_in == 0 (final state dropped).
 *
 * For each batch row b and channel d, with h = h_{-1}:
 *   v     = delta[b,t,d] + bias[d]
 *   dt    = softplus(v) if delta_softplus else v
 *   abar  = exp(dt * A[d,n])
 *   bbar  = dt * B[.,n]                       (bbar_mode 0)
 *         = expm1(dt * A[d,n]) / A[d,n] * B   (bbar_mode 1, exact ZOH)
 *   h[n]  = abar * h[n] + bbar * x[b,t,d]
 *   y     = sum_n C[.,n] h[n] + D[d] x[b,t,d]
 *   out   = y * silu(z[b,t,d])  (or y without a gate)
 * Returns 0, or -1 on bad sizes.
 */
int oracle_selective_scan_f64(const double* x, const double* delta,
                              const double* A, const double* B,
                              const double* C, const double* D,
                              const double* z, const double* delta_bias,
                              double* out, double* state, int64_t batch,
                              int64_t seqlen, int64_t dim, int64_t dstate,
                              int per_channel_bc, int delta_softplus,
                              int state_in, int bbar_mode, int nthreads) {
  if (batch < 0 || seqlen < 0 || dim < 0 || dstate <= 0 || dstate > 4096)
    return -1;
  if (state_in && state == NULL) return -1;
  if (bbar_mode != 0 && bbar_mode != 1) return -1;
  const int64_t nchan = batch * dim;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t ch = 0; ch < nchan; ++ch) {
    const int64_t b = ch / dim;
    const int64_t d = ch % dim;
    double h[4096];
    for (int64_t n = 0; n < dstate; ++n)
      h[n] = state_in ? state[(b * dim + d) * dstate + n] : 0.0;

    for (int64_t t = 0; t < seqlen; ++t) {
      const int64_t i = (b * seqlen + t) * dim + d; /* (b, t, d) */
      const double v = delta[i] + (delta_bias ? delta_bias[d] : 0.0);
      const double dt = delta_softplus ? oracle_softplus(v) : v;
      const double xv = x[i];
      const double* Bv = per_channel_bc ? &B[d * dstate]
                                        : &B[(b * seqlen + t) * dstate];
      const double* Cv = per_channel_bc ? &C[d * dstate]
                                        : &C[(b * seqlen + t) * dstate];
      double y = 0.0;
      for (int64_t n = 0; n < dstate; ++n) {
        const double a = A[d * dstate + n];
        const double abar = exp(dt * a);
        double bbar;
        if (bbar_mode == 0)
          bbar = dt * Bv[n];
        else
          bbar = (a != 0.0) ? expm1(dt * a) / a * Bv[n] : dt * Bv[n];
        h[n] = abar * h[n] + bbar * xv;
        y += Cv[n] * h[n];
      }
      y += (D ? D[d] : 0.0) * xv;
      if (z) y *= silu(z[i]);
      out[i] = y;
    }
    if (state)
      for (int64_t n = 0; n < dstate; ++n)
        state[(b * dim + d) * dstate + n] = h[n];
  }
  return 0;
}

/*
 * Convolution kernel of a linear time-invariant diagonal SSM
 * ("State-space models", section "Recurrence and convolution":
 * K_k = C Abar^k Bbar).  Per channel d with constant step dt[d]:
 *   K[d,k] = sum_n C[d,n] * exp(k * dt[d] * A[d,n]) * bbar[d,n],
 * bbar = dt B (bbar_mode 0) or the exact ZOH term (bbar_mode 1).
 * Abar^k is taken as exp(k dt a), its exact value for a diagonal A.
 * K is (dim, seqlen).  Returns 0, or -1 on bad sizes.
 */
int oracle_lti_kernel(const double* A, const double* B, const double* C,
                      const double* dt, double* K, int64_t dim,
                      int64_t dstate, int64_t seqlen, int bbar_mode) {
  if (dim < 0 || dstate <= 0 || seqlen < 0) return -1;
  for (int64_t d = 0; d < dim; ++d) {
    for (int64_t k = 0; k < seqlen; ++k) {
      double s = 0.0;
      for (int64_t n = 0; n < dstate; ++n) {
        const double a = A[d * dstate + n];
        const double bb = (bbar_mode == 0 || a == 0.0)
                              ? dt[d] * B[d * dstate + n]
                              : expm1(dt[d] * a) / a * B[d * dstate + n];
        s += C[d * dstate + n] * exp((double)k * dt[d] * a) * bb;
      }
      K[d * seqlen + k] = s;
    }
  }
  return 0;
}

/*
 * Causal, zero-padded linear convolution of x with a per-channel kernel, plus
 * the skip term ("State-space models", section "Recurrence and convolution";
 * "Structured State Space Models and Mamba", LTI unroll
 * y_k = sum_{j<=k} C Abar^{k-j} Bbar x_j):
 *   out[b,t,d] = sum_{k=0..t} K[d,k] x[b,t-k,d] + D[d] x[b,t,d].
 * x, out: (batch, seqlen, dim); K: (dim, seqlen); D may be NULL.
 */
int oracle_causal_conv(const double* x, const double* K, const double* D,
                       double* out, int64_t batch, int64_t seqlen,
                       int64_t dim, int nthreads) {
  if (batch < 0 || seqlen < 0 || dim < 0) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  const int64_t nchan = batch * dim;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t ch = 0; ch < nchan; ++ch) {
    const int64_t b = ch / dim;
    const int64_t d = ch % dim;
    for (int64_t t = 0; t < seqlen; ++t) {
      double s = 0.0;
      for (int64_t k = 0; k <= t; ++k)
        s += K[d * seqlen + k] * x[(b * seqlen + (t - k)) * dim + d];
      const int64_t i = (b * seqlen + t) * dim + d;
      out[i] = s + (D ? D[d] : 0.0) * x[i];
    }
  }
  return 0;
}

/*
 * Prologue of the Mamba block on the branch that feeds the SSM
 * ("State-space models", section "Mamba: selection", the block description:
 * a depthwise causal convolution of width 4 and a silu).  Per batch row b and
 * channel d, with W = width taps (lag k multiplies the input k steps back):
 *   pre[b,t,d] = sum_{k=0..W-1} w[d,k] * x[b,t-k,d] + cb[d]
 *   u[b,t,d]   = silu(pre[b,t,d])
 * Inputs before the sequence (t-k < 0) come from hist[b,d,0..W-2], the W-1
 * inputs preceding the sequence, oldest first; zero when hist is NULL.
 * hist_out (may be NULL, may alias hist) receives the last W-1 inputs of the
 * history-extended sequence, oldest first, for a call that continues it.
 * cb may be NULL (no bias).  x, u: (batch, seqlen, dim); w: (dim, W).
 * Returns 0, or -1 on bad sizes.
 */
int oracle_conv_silu(const double* x, const double* w, const double* cb,
                     const double* hist, double* u, double* hist_out,
                     int64_t batch, int64_t seqlen, int64_t dim,
                     int64_t width, int nthreads) {
  if (batch < 0 || seqlen < 0 || dim < 0 || width < 1 || width > 64) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  const int64_t nchan = batch * dim;
  const int64_t H = width - 1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t ch = 0; ch < nchan; ++ch) {
    const int64_t b = ch / dim;
    const int64_t d = ch % dim;
    double past[64];
    for (int64_t j = 0; j < H; ++j)
      past[j] = hist ? hist[(b * dim + d) * H + j] : 0.0;
    /* input at step tau of the history-extended sequence, tau >= -H */
#define XS(tau) ((tau) < 0 ? past[H + (tau)] : x[(b * seqlen + (tau)) * dim + d])
    for (int64_t t = 0; t < seqlen; ++t) {
      double pre = cb ? cb[d] : 0.0;
      for (int64_t k = 0; k < width; ++k) pre += w[d * width + k] * XS(t - k);
      u[(b * seqlen + t) * dim + d] = silu(pre);
    }
    if (hist_out)
      for (int64_t j = 0; j < H; ++j)
        hist_out[(b * dim + d) * H + j] = XS(seqlen - H + j);
#undef XS
  }
  return 0;
}

/*
 * Gradients of the selective-scan forward (bbar_mode 0, time-varying B and C),
 * the backward pass with the states rebuilt rather than stored ("State-space
 * models", section "The parallel scan": Mamba's kernel recomputes the expanded
 * state in the backward pass).  Reverse-mode differentiation of the recurrence as
 * oracle_selective_scan_f64 states it.  Per batch row b and channel d:
 *
 *   forward:  dt_t = softplus(v_t) (or v_t), v_t = delta_t + bias;
 *             a_t[n] = exp(dt_t A[n]);  h_t = a_t h_{t-1} + dt_t B_t x_t;
 *             y_t = C_t . h_t + D x_t;  out_t = y_t silu(z_t)
 *   reverse:  gy_t = dout_t silu(z_t)  (dout_t without a gate)
 *             lam_t = C_t gy_t + a_{t+1} lam_{t+1},  lam_{L-1} = C gy + dfinal
 *             dA[n]   += lam_t[n] h_{t-1}[n] a_t[n] dt_t
 *             ddt_t    = sum_n lam_t[n] (h_{t-1}[n] a_t[n] A[n] + B_t[n] x_t)
 *             dx_t     = sum_n lam_t[n] dt_t B_t[n] + gy_t D
 *             dB_t[n] += lam_t[n] dt_t x_t          (summed over channels)
 *             dC_t[n] += gy_t h_t[n]                (summed over channels)
 *             dz_t     = dout_t y_t silu'(z_t),  silu'(z) = s (1 + z (1 - s)), s = sigmoid(z)
 *             ddelta_t = ddt_t sigmoid(v_t) (softplus) or ddt_t;  dbias += ddelta_t
 *             dD      += gy_t x_t;   dh0 = a_0 lam_0
 *
 * h0 (batch, dim, N) may be NULL (zeros); dfinal (batch, dim, N) may be NULL
 * (zeros); z, D, delta_bias may be NULL.  Outputs dx, ddelta, dz (when z),
 * (batch, L, dim); dA (dim, N); dB, dC (batch, L, N); dD, dbias (dim); dh0
 * (batch, dim, N) -- dz, dD, dbias, dh0 may be NULL.  The shared gradients
 * (dA, dB, dC, dD, dbias) are zeroed here and summed over channels.
 * Returns 0, or -1 on bad sizes.
 */
int oracle_selective_scan_bwd_f64(
    const double* x, const double* delta, const double* A, const double* B,
    const double* C, const double* D, const double* z, const double* delta_bias,
    const double* h0, const double* dout, const double* dfinal, double* dx,
    double* ddelta, double* dA, double* dB, double* dC, double* dD, double* dz,
    double* dbias, double* dh0, int64_t batch, int64_t seqlen, int64_t dim,
    int64_t dstate, int delta_softplus, int nthreads) {
  if (batch < 0 || seqlen < 0 || dim < 0 || dstate <= 0 || dstate > 64) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  const int64_t N = dstate, L = seqlen;
  for (int64_t i = 0; i < dim * N; ++i) dA[i] = 0.0;
  for (int64_t i = 0; i < batch * L * N; ++i) dB[i] = dC[i] = 0.0;
  for (int64_t d = 0; d < dim; ++d) {
    if (dD) dD[d] = 0.0;
    if (dbias) dbias[d] = 0.0;
  }
  const int64_t nchan = batch * dim;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t ch = 0; ch < nchan; ++ch) {
    const int64_t b = ch / dim;
    const int64_t d = ch % dim;
    /* forward, keeping every state: hs[(t + 1) N + n] = h_t[n], hs[n] = h_{-1}[n] */
    double* hs = (double*)malloc(sizeof(double) * (size_t)(L + 1) * N);
    double* dts = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double* vs = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    for (int64_t n = 0; n < N; ++n) hs[n] = h0 ? h0[(b * dim + d) * N + n] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
      const int64_t i = (b * L + t) * dim + d;
      vs[t] = delta[i] + (delta_bias ? delta_bias[d] : 0.0);
      dts[t] = delta_softplus ? oracle_softplus(vs[t]) : vs[t];
      for (int64_t n = 0; n < N; ++n)
        hs[(t + 1) * N + n] = exp(dts[t] * A[d * N + n]) * hs[t * N + n] +
                              dts[t] * B[(b * L + t) * N + n] * x[i];
    }
    /* reverse */
    double lam_next[64], a_next[64];
    for (int64_t n = 0; n < N; ++n) {
      lam_next[n] = dfinal ? dfinal[(b * dim + d) * N + n] : 0.0;
      a_next[n] = 1.0; /* the final-state gradient enters lam_{L-1} undecayed */
    }
    double sD = 0.0, sbias = 0.0;
    for (int64_t t = L - 1; t >= 0; --t) {
      const int64_t i = (b * L + t) * dim + d;
      const double* Bt = &B[(b * L + t) * N];
      const double* Ct = &C[(b * L + t) * N];
      const double sz = z ? 1.0 / (1.0 + exp(-z[i])) : 1.0;
      const double gy = z ? dout[i] * z[i] * sz : dout[i];
      double ddt = 0.0, gx = 0.0, y = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        const double a = exp(dts[t] * A[d * N + n]);
        const double lam = Ct[n] * gy + a_next[n] * lam_next[n];
        const double hprev = hs[t * N + n], hcur = hs[(t + 1) * N + n];
#pragma omp atomic
        dA[d * N + n] += lam * hprev * a * dts[t];
        ddt += lam * (hprev * a * A[d * N + n] + Bt[n] * x[i]);
        gx += lam * dts[t] * Bt[n];
#pragma omp atomic
        dB[(b * L + t) * N + n] += lam * dts[t] * x[i];
#pragma omp atomic
        dC[(b * L + t) * N + n] += gy * hcur;
        y += Ct[n] * hcur;
        lam_next[n] = lam;
        a_next[n] = a;
      }
      y += (D ? D[d] : 0.0) * x[i];
      dx[i] = gx + gy * (D ? D[d] : 0.0);
      if (z && dz) dz[i] = dout[i] * y * sz * (1.0 + z[i] * (1.0 - sz));
      const double sv = delta_softplus ? 1.0 / (1.0 + exp(-vs[t])) : 1.0;
      ddelta[i] = ddt * sv;
      sbias += ddt * sv;
      sD += gy * x[i];
    }
    if (dh0)
      for (int64_t n = 0; n < N; ++n) dh0[(b * dim + d) * N + n] = a_next[n] * lam_next[n];
    if (dD) {
#pragma omp atomic
      dD[d] += sD;
    }
    if (dbias) {
#pragma omp atomic
      dbias[d] += sbias;
    }
    free(hs);
    free(dts);
    free(vs);
  }
  return 0;
}

/*
 * Mamba-2 state-space-duality (SSD) layer, forward, stepped as a recurrence
 * ("State-space models", section "The parallel scan": Mamba-2 restricts A to a
 * scalar times the identity per head; "State Space Models: Mamba and Beyond",
 * section "Beyond Mamba: state-space duality and hybrid architectures": A is a
 * scalar per attention-style head; "Structured State Space Models and Mamba",
 * section "State Space Duality and Mamba-2": the same map written as masked
 * attention Y = (L o (C B^T)) V, which the tests use as a pin).
 *
 * Shapes: x, z, out: (batch, L, H, P); dt: (batch, L, H); A, D, dt_bias: (H);
 * B, C: (batch, L, G, N), head h reading group h / (H / G); state:
 * (batch, H, P, N), read as h_{-1} when state_in, else h_{-1} = 0; written with
 * h_{L-1} when not NULL.  For each batch row b, head h, step t:
 *   s      = dt[b,t,h] + dt_bias[h];  step = softplus(s) if dt_softplus else s
 *   a      = exp(step * A[h])                      one decay for the whole head
 *   h[p,n] = a * h[p,n] + step * B[b,t,g,n] * x[b,t,h,p]
 *   y[p]   = sum_n C[b,t,g,n] h[p,n] + D[h] x[b,t,h,p]
 *   out    = y * silu(z[b,t,h,p])  (or y without a gate)
 * Returns 0, or -1 on bad sizes.
 */
int oracle_ssd_f64(const double* x, const double* dt, const double* A,
                   const double* B, const double* C, const double* D,
                   const double* z, const double* dt_bias, double* out,
                   double* state, int64_t batch, int64_t seqlen, int64_t nheads,
                   int64_t headdim, int64_t ngroups, int64_t dstate,
                   int dt_softplus, int state_in, int nthreads) {
  if (batch < 0 || seqlen < 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 ||
      dstate <= 0 || nheads % ngroups != 0)
    return -1;
  if (state_in && state == NULL) return -1;
  const int64_t per_group = nheads / ngroups;
  const int64_t P = headdim, N = dstate, H = nheads;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < batch * H; ++bh) {
    const int64_t b = bh / H, h = bh % H, g = h / per_group;
    double* hs = (double*)malloc((size_t)(P * N) * sizeof(double));
    if (!hs) {
#pragma omp atomic write
      bad = 1;
      continue;
    }
    for (int64_t i = 0; i < P * N; ++i)
      hs[i] = state_in ? state[(b * H + h) * P * N + i] : 0.0;
    for (int64_t t = 0; t < seqlen; ++t) {
      const double s = dt[(b * seqlen + t) * H + h] + (dt_bias ? dt_bias[h] : 0.0);
      const double step = dt_softplus ? oracle_softplus(s) : s;
      const double a = exp(step * A[h]);
      const double* Bv = &B[((b * seqlen + t) * ngroups + g) * N];
      const double* Cv = &C[((b * seqlen + t) * ngroups + g) * N];
      const int64_t row = ((b * seqlen + t) * H + h) * P;
      for (int64_t p = 0; p < P; ++p) {
        const double xv = x[row + p];
        double y = 0.0;
        for (int64_t n = 0; n < N; ++n) {
          hs[p * N + n] = a * hs[p * N + n] + step * Bv[n] * xv;
          y += Cv[n] * hs[p * N + n];
        }
        y += (D ? D[h] : 0.0) * xv;
        if (z) y *= silu(z[row + p]);
        out[row + p] = y;
      }
    }
    if (state)
      for (int64_t i = 0; i < P * N; ++i) state[(b * H + h) * P * N + i] = hs[i];
    free(hs);
  }
  return bad ? -1 : 0;
}

/* Number of threads OpenMP would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
