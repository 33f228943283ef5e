// Selective-scan forward kernels for sm_103a (B300).
//
// What is computed (pages "State-space models", sections "Discretization",
// "Mamba: selection", "The parallel scan", "Implementation"; "Structured State
// Space Models and Mamba", sections "Discretization Mechanics", S6, "The GPU
// Memory Hierarchy and Kernel Fusion"):
//   step = softplus(delta + bias); Abar = exp(step * A[d,n]); h = Abar h + step B x;
//   y = C . h + D x; out = y * silu(z).
//
// Design (B300):
//  * One thread owns one channel (b, d) and NPT of its N states (TPC threads per
//    channel when N > 16).  The state lives in registers for the whole chunk; Abar,
//    Bbar and h never touch memory: only out and the final state are written.
//  * Fast kernel: tiles of T steps x 128 channels of x / delta / z and T x N of
//    B / C arrive through a 3-stage TMA (cp.async.bulk.tensor) pipeline completed
//    on mbarriers, so DRAM latency is hidden by copies in flight, not by registers.
//    B_t / C_t are shared by the whole CTA: widened to fp32 once per tile into a
//    padded, double-buffered table and read back as broadcast float4 loads.
//    The generic kernel (shapes a tensor map cannot describe) streams the same data
//    with plain coalesced loads and a register prefetch ring.
//  * States are processed in pairs with packed f32x2 arithmetic (FMUL2 / FFMA2),
//    halving the issue slots of the per-state work.
//  * Long sequences are cut into chunks scanned by different CTAs.  The carry between
//    chunks uses the associative combine of the per-step maps ("The parallel scan":
//    (a1, b1) then (a2, b2) = (a1 a2, a2 b1 + b2)): an aggregate pass writes each
//    chunk's sum of steps S (prod Abar = exp(A S)) and its end state from a zero
//    start; the output pass folds the aggregates of the preceding chunks into its
//    starting state.  The kernel boundary orders the passes: no CTA waits on another.
//  * On B300 each ex2 also occupies two FP32-pipe issue slots, so the scan is bound
//    by the FP32 pipe.  Channels whose A row is (n+1) * A[d,0] (S4D-real) take one
//    exponential per step and form the other decays as its powers.
//  * Precision: bf16 inputs form Abar with MUFU ex2.  fp32 inputs carry m = Abar - 1
//    (accurate expm1; powers composed as (1+a)(1+b) - 1 = a + b + ab) and update
//    h <- h + (m h + Bbar x), because near Abar = 1 the fp32 grid itself (spacing
//    6e-8) would misstate a decay rate 1 - Abar ~ 1e-5 by up to 0.3%.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>

namespace ssm {

constexpr int kThreads = 128;  // threads per CTA
constexpr int kTB = 32;        // generic kernel: steps per shared-memory block of B_t / C_t
constexpr int kPF = 4;         // generic kernel: prefetch distance in steps
constexpr int kStages = 3;     // fast kernel: TMA pipeline depth
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr long long kSpinLimit = 1ll << 26;  // bounded mbarrier waits

enum : int { kStatusOk = 0, kStatusTimeout = 1 };

struct ScanParams {
  const void* x;
  const void* delta;
  const void* z;        // nullable
  void* out;
  const float* A;       // (dim, N)
  const void* B;        // (batch, L, N) io dtype, or (dim, N) fp32
  const void* C;
  const float* Dskip;   // nullable
  const float* bias;    // nullable
  float* final_state;   // nullable; written by the last chunk of the output pass
  const float* h_init;  // nullable; initial state (batch, dim, N)
  float* ws_H;          // (nchunks-1, batch, dim, N) chunk end states from the aggregate pass
  float* ws_S;          // (nchunks-1, batch, dim) chunk step sums
  float* ws_h0;         // copy of h_init for the output pass when nchunks > 1
  int* status;          // device status word
  int64_t batch, seqlen, dim;
  int dstate;
  int nchunks;
  int64_t chunk_len;
  int delta_softplus;
  int pow_path;
};

struct TmaMaps {
  CUtensorMap x, delta, z, B, C;
};

// ------------------------------------------------------------------ element access

struct F32 {
  static constexpr int kBytes = 4;
  static constexpr bool kFastDecay = false;  // decays carried as Abar - 1 (accurate)
  static __device__ __forceinline__ float load(const void* p, int64_t i) {
    return __ldg(static_cast<const float*>(p) + i);
  }
  static __device__ __forceinline__ float lds(const unsigned char* p) {
    return *reinterpret_cast<const float*>(p);
  }
  static __device__ __forceinline__ void store(void* p, int64_t i, float v) {
    static_cast<float*>(p)[i] = v;
  }
};

struct BF16 {
  static constexpr int kBytes = 2;
  static constexpr bool kFastDecay = true;   // decays formed with MUFU ex2
  static __device__ __forceinline__ float widen(unsigned short v) {
    return __uint_as_float(static_cast<unsigned>(v) << 16);  // exact
  }
  static __device__ __forceinline__ float load(const void* p, int64_t i) {
    return widen(__ldg(static_cast<const unsigned short*>(p) + i));
  }
  static __device__ __forceinline__ float lds(const unsigned char* p) {
    return widen(*reinterpret_cast<const unsigned short*>(p));
  }
  static __device__ __forceinline__ void store(void* p, int64_t i, float v) {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  }
};

// ------------------------------------------------------------------------ math

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// softplus(v) = log(1 + e^v).  ACCURATE: relative error ~1e-7 (libm log1pf);
// otherwise the MUFU lg2 form, absolute error ~1e-7 (enough for bf16 inputs).
template <bool ACCURATE>
__device__ __forceinline__ float softplus(float v) {
  if (v > 15.f) return v + ex2(-v * kLog2e);  // log1p(e^v) = v + log1p(e^-v), e^-v < 4e-7
  const float e = ex2(v * kLog2e);
  if (ACCURATE) return log1pf(e);
  return lg2(1.f + e) * kLn2;
}

// silu(z) = z * sigmoid(z)
__device__ __forceinline__ float silu(float z) {
  return __fdividef(z, 1.f + ex2(-z * kLog2e));
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Per-channel constants of the state update, held in registers for the whole chunk.
template <int NPT>
struct ChannelConsts {
  float2 A2[NPT / 2];   // A * log2(e), state pairs
  float A2base;         // A[d,0] * log2(e)          (powers path)
  float A2first;        // A[d, first state] * log2e (powers path, TPC > 1)
  float Ar[NPT];        // A                          (expm1 paths)
  float Bc[NPT], Cc[NPT];
};

// (1 + x)(1 + y) - 1 without forming the products near 1: the composition of two
// decays carried as Abar - 1, exact in relative terms up to two roundings.
__device__ __forceinline__ float mcomb(float x, float y) { return fmaf(x, y, x + y); }

// m[e-1] = (1 + m1)^e - 1 for e = 1..NPT, by repeated halving (depth <= 2 log2 NPT).
template <int NPT>
__device__ __forceinline__ void mpowers(float m1, float (&m)[NPT]) {
  m[0] = m1;
#pragma unroll
  for (int e = 2; e <= NPT; ++e) m[e - 1] = (e & 1) ? mcomb(m[e - 2], m1) : mcomb(m[e / 2 - 1], m[e / 2 - 1]);
}

// One step of one channel: update the NPT states, return this thread's share of
// C . h (0 in the aggregate pass).  Brow / Crow: fp32 rows of this thread's states
// (unused for constant-coefficient channels, whose B and C sit in k).
//
// MFORM (fp32 inputs and constant-coefficient channels) carries m = Abar - 1 =
// expm1(step A), accurate to a few ulp even when Abar is within 1e-5 of 1, and
// updates h <- h + (m h + Bbar x): the decay of a long-memory channel keeps its full
// relative precision, which an fp32 Abar itself cannot hold.  Otherwise (bf16 inputs)
// Abar = 2^(step A log2 e) from MUFU ex2 and h <- Abar h + Bbar x.
template <int NPT, int TPC, bool POW, bool LTI, bool OUT, bool MFORM>
__device__ __forceinline__ float step_states(float dt, float u, const float* __restrict__ Brow,
                                             const float* __restrict__ Crow,
                                             float2 (&h)[NPT / 2], const ChannelConsts<NPT>& k) {
  const float2 dt2 = f2(dt, dt), u2 = f2(u, u);
  float2 a[NPT / 2];  // Abar, or Abar - 1 in MFORM
  if (MFORM) {
    if (POW && TPC == 1) {
      float m[NPT];
      mpowers<NPT>(expm1f(dt * k.Ar[0]), m);
#pragma unroll
      for (int i = 0; i < NPT / 2; ++i) a[i] = f2(m[2 * i], m[2 * i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < NPT / 2; ++i) a[i] = f2(expm1f(dt * k.Ar[2 * i]), expm1f(dt * k.Ar[2 * i + 1]));
    }
  } else if (POW) {
    // A[d,n] = (n+1) A[d,0]:  Abar_n = r^(n+1), r = exp(step A[d,0])
    const float r = ex2(dt * k.A2base);
    const float r2 = r * r;
    const float first = (TPC == 1) ? r : ex2(dt * k.A2first);
    a[0] = f2(first, first * r);
    const float2 st = f2(r2, r2);
#pragma unroll
    for (int i = 1; i < NPT / 2; ++i) a[i] = __fmul2_rn(a[i - 1], st);
  } else {
#pragma unroll
    for (int i = 0; i < NPT / 2; ++i) {
      const float2 g = __fmul2_rn(dt2, k.A2[i]);
      a[i] = f2(ex2(g.x), ex2(g.y));
    }
  }
  auto update = [&](int i, float2 b) {
    const float2 ub = __fmul2_rn(u2, b);
    h[i] = MFORM ? __fadd2_rn(h[i], __ffma2_rn(a[i], h[i], ub)) : __ffma2_rn(a[i], h[i], ub);
  };
  float2 ya = f2(0.f, 0.f), yb = f2(0.f, 0.f);
#pragma unroll
  for (int q = 0; q < NPT / 4; ++q) {
    const int i0 = 2 * q, i1 = 2 * q + 1;
    float4 b4, c4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (LTI) {
      b4 = make_float4(k.Bc[4 * q], k.Bc[4 * q + 1], k.Bc[4 * q + 2], k.Bc[4 * q + 3]);
      c4 = make_float4(k.Cc[4 * q], k.Cc[4 * q + 1], k.Cc[4 * q + 2], k.Cc[4 * q + 3]);
    } else {
      b4 = *reinterpret_cast<const float4*>(Brow + 4 * q);
      if (OUT) c4 = *reinterpret_cast<const float4*>(Crow + 4 * q);
    }
    update(i0, f2(b4.x, b4.y));
    update(i1, f2(b4.z, b4.w));
    if (OUT) {
      ya = __ffma2_rn(f2(c4.x, c4.y), h[i0], ya);
      yb = __ffma2_rn(f2(c4.z, c4.w), h[i1], yb);
    }
  }
  return OUT ? (ya.x + ya.y) + (yb.x + yb.y) : 0.f;
}

// Load the channel constants; returns whether this channel's A row is (n+1) A[d,0].
template <int NPT, int TPC, bool LTI>
__device__ __forceinline__ bool load_consts(const ScanParams& p, int64_t dd, int sub,
                                            ChannelConsts<NPT>& k) {
  const int N = p.dstate;
  const float a0 = p.A[dd * N];
  bool structured = true;
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    const int n = sub * NPT + j;
    const float a = (n < N) ? p.A[dd * N + n] : 0.f;
    if (j & 1) k.A2[j / 2].y = a * kLog2e;
    else k.A2[j / 2].x = a * kLog2e;
    k.Ar[j] = a;
    if (n < N && a != (float)(n + 1) * a0) structured = false;
    if (LTI) {
      k.Bc[j] = (n < N) ? static_cast<const float*>(p.B)[dd * N + n] : 0.f;
      k.Cc[j] = (n < N) ? static_cast<const float*>(p.C)[dd * N + n] : 0.f;
    }
  }
  k.A2base = a0 * kLog2e;
  k.A2first = k.A2[0].x;
  return structured;
}

// Starting state of a chunk: h_init (chunk 0) or the fold of the preceding chunks'
// aggregates, h <- exp(A S_c') h + H_c'.
template <int NPT, int PASS>
__device__ __forceinline__ void start_state(const ScanParams& p, int b, int c, int64_t dd, int sub,
                                            bool valid, float2 (&h)[NPT / 2],
                                            const ChannelConsts<NPT>& k) {
  const int N = p.dstate;
  const int64_t Dm = p.dim;
  float hv[NPT];
#pragma unroll
  for (int j = 0; j < NPT; ++j) hv[j] = 0.f;
  const int64_t sidx = ((int64_t)b * Dm + dd) * N;
  if (c == 0) {
    const float* src = (PASS == 1 && p.nchunks > 1) ? p.ws_h0 : p.h_init;
    if (src) {
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int n = sub * NPT + j;
        if (n < N) hv[j] = src[sidx + n];
      }
      if (PASS == 0 && p.ws_h0 && valid) {
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
          const int n = sub * NPT + j;
          if (n < N) p.ws_h0[sidx + n] = hv[j];
        }
      }
    }
  } else if (PASS == 1) {
    for (int cc = 0; cc < c; ++cc) {
      const int64_t ci = (int64_t)cc * p.batch + b;
      const float S = p.ws_S[ci * Dm + dd];
      const float* H = p.ws_H + (ci * Dm + dd) * N;
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int n = sub * NPT + j;
        const float a2 = (j & 1) ? k.A2[j / 2].y : k.A2[j / 2].x;
        if (n < N) hv[j] = fmaf(ex2(S * a2), hv[j], H[n]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NPT / 2; ++i) h[i] = f2(hv[2 * i], hv[2 * i + 1]);
}

template <int NPT, int PASS>
__device__ __forceinline__ void store_results(const ScanParams& p, int b, int c, int64_t d, int sub,
                                              const float2 (&h)[NPT / 2], float S) {
  const int N = p.dstate;
  const int64_t Dm = p.dim;
  if (PASS == 1) {
    if (c == p.nchunks - 1 && p.final_state) {
      const int64_t sidx = ((int64_t)b * Dm + d) * N;
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int n = sub * NPT + j;
        if (n < N) p.final_state[sidx + n] = (j & 1) ? h[j / 2].y : h[j / 2].x;
      }
    }
  } else {
    const int64_t ci = (int64_t)c * p.batch + b;
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const int n = sub * NPT + j;
      if (n < N) p.ws_H[(ci * Dm + d) * N + n] = (j & 1) ? h[j / 2].y : h[j / 2].x;
    }
    if (sub == 0) p.ws_S[ci * Dm + d] = S;
  }
}

// Step size of one (t, d): softplus(delta + bias), or delta + bias.
template <typename IO>
__device__ __forceinline__ float step_size(const ScanParams& p, float dv, float biasv) {
  const float v = dv + biasv;
  return p.delta_softplus ? softplus<std::is_same<IO, F32>::value>(v) : v;
}

__device__ __forceinline__ void kahan_add(float& S, float& comp, float x) {
  const float y = x - comp;
  const float t = S + y;
  comp = (t - S) - y;
  S = t;
}

// ----------------------------------------------------------------- TMA helpers

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: false if the phase did not complete within kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (long long i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

template <typename IO> struct TileSteps;
template <> struct TileSteps<BF16> { static constexpr int value = 16; };
template <> struct TileSteps<F32> { static constexpr int value = 8; };

// Shared-memory bytes of the fast kernel.
template <typename IO, int NPT, int TPC>
constexpr int tma_smem_bytes() {
  constexpr int T = TileSteps<IO>::value, NST = NPT * TPC, CH = kThreads / TPC;
  constexpr int XB = T * CH * IO::kBytes, BCB = T * NST * IO::kBytes;
  return kStages * (3 * XB + 2 * BCB) + 2 * 2 * T * NST * 4 + kStages * 8;
}

// ------------------------------------------------------------ fast (TMA) kernel

// PASS 0: chunk aggregate (end state from the chunk start, sum of steps).
// PASS 1: output pass (carry-in, y, out, final state).
template <typename IO, int NPT, int TPC, bool LTI, int PASS>
__global__ void __launch_bounds__(kThreads)
scan_tma_kernel(const __grid_constant__ TmaMaps maps, const ScanParams p) {
  constexpr int T = TileSteps<IO>::value, S = kStages, NST = NPT * TPC, CH = kThreads / TPC;
  constexpr int ESZ = IO::kBytes;
  constexpr int XB = T * CH * ESZ, BCB = T * NST * ESZ, STAGE = 3 * XB + 2 * BCB;
  constexpr bool OUT = (PASS == 1);
  constexpr bool MFORM = LTI || !IO::kFastDecay;
  extern __shared__ __align__(128) unsigned char smem[];
  float* conv = reinterpret_cast<float*>(smem + S * STAGE);          // [2][2][T][NST]
  uint64_t* full = reinterpret_cast<uint64_t*>(conv + 2 * 2 * T * NST);

  const int tid = threadIdx.x;
  const int N = p.dstate;
  const int64_t L = p.seqlen, Dm = p.dim;
  const int b = blockIdx.z, c = blockIdx.y;
  const int sub = tid % TPC, lch = tid / TPC;
  const int d0 = blockIdx.x * CH;
  const int64_t d = (int64_t)d0 + lch;
  const bool valid = d < Dm;
  const int64_t dd = valid ? d : Dm - 1;
  const int64_t t0 = (int64_t)c * p.chunk_len;
  const int64_t t1 = min(t0 + p.chunk_len, L);
  const int ntiles = (int)((t1 - t0 + T - 1) / T);
  const bool gate = OUT && (p.z != nullptr);
  const uint32_t tile_bytes = (uint32_t)((2 + (gate ? 1 : 0)) * XB +
                                         (LTI ? 0 : (OUT ? 2 : 1) * T * N * ESZ));

  auto stage = [&](int s) { return smem + s * STAGE; };
  auto issue = [&](int i) {  // one thread: start the copies of tile i
    const int s = i % S;
    const int ts = (int)(t0 + (int64_t)i * T);
    mbar_arrive_expect_tx(&full[s], tile_bytes);
    tma_load_3d(stage(s), &maps.x, d0, ts, b, &full[s]);
    tma_load_3d(stage(s) + XB, &maps.delta, d0, ts, b, &full[s]);
    if (gate) tma_load_3d(stage(s) + 2 * XB, &maps.z, d0, ts, b, &full[s]);
    if (!LTI) {
      tma_load_3d(stage(s) + 3 * XB, &maps.B, 0, ts, b, &full[s]);
      if (OUT) tma_load_3d(stage(s) + 3 * XB + BCB, &maps.C, 0, ts, b, &full[s]);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
  }
  // zero the padded state columns of the widened B / C tables
  for (int e = tid; e < 2 * 2 * T * NST; e += kThreads) conv[e] = 0.f;
  __syncthreads();
  if (tid == 0)
    for (int i = 0; i < S && i < ntiles; ++i) issue(i);

  ChannelConsts<NPT> k;
  const bool structured = load_consts<NPT, TPC, LTI>(p, dd, sub, k);
  const bool use_pow = !LTI && p.pow_path && (IO::kFastDecay || TPC == 1) &&
                       __syncthreads_and(structured || !valid);
  const float biasv = p.bias ? p.bias[dd] : 0.f;
  const float Dv = p.Dskip ? p.Dskip[dd] : 0.f;
  float2 h[NPT / 2];
  start_state<NPT, PASS>(p, b, c, dd, sub, valid, h, k);

  // widen tile i's B / C rows into the fp32 table (i & 1)
  auto widen_bc = [&](int i) {
    if (LTI) return;
    const int s = i % S;
    float* dstB = conv + ((i & 1) * 2) * T * NST;
    const unsigned char* srcB = stage(s) + 3 * XB;
    for (int e = tid; e < T * N; e += kThreads) {
      const int tt = e / N, n = e - tt * N;
      dstB[tt * NST + n] = IO::lds(srcB + e * ESZ);
      if (OUT) dstB[T * NST + tt * NST + n] = IO::lds(srcB + BCB + e * ESZ);
    }
  };

  bool ok = true;
  if (ntiles > 0) ok = mbar_wait(&full[0], 0);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) atomicExch(p.status, kStatusTimeout);
    return;
  }
  widen_bc(0);
  __syncthreads();

  float S_sum = 0.f, S_comp = 0.f;
  int64_t oidx = ((int64_t)b * L + t0) * Dm + d;  // out element of the current step

  auto run = [&](auto pow_tag) {
    constexpr bool POW = decltype(pow_tag)::value;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % S;
      const unsigned char* st = stage(s);
      const float* Bt = conv + ((i & 1) * 2) * T * NST + sub * NPT;
      const float* Ct = Bt + T * NST;
      const int64_t rem = t1 - (t0 + (int64_t)i * T);
      const int nsteps = rem < T ? (int)rem : T;
      auto one_step = [&](int tt) {
        const float xv = IO::lds(st + (tt * CH + lch) * ESZ);
        const float dv = IO::lds(st + XB + (tt * CH + lch) * ESZ);
        const float dt = step_size<IO>(p, dv, biasv);
        const float u = dt * xv;
        float y = step_states<NPT, TPC, POW, LTI, OUT, MFORM>(dt, u, Bt + tt * NST, Ct + tt * NST, h, k);
        if (OUT) {
#pragma unroll
          for (int off = 1; off < TPC; off <<= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
          if (sub == 0 && valid) {
            y = fmaf(Dv, xv, y);
            if (gate) y *= silu(IO::lds(st + 2 * XB + (tt * CH + lch) * ESZ));
            IO::store(p.out, oidx, y);
          }
        } else {
          kahan_add(S_sum, S_comp, dt);
        }
        oidx += Dm;
      };
      if (nsteps == T) {
        // Full tile, in groups of G steps and three phases so that independent work of
        // different steps can overlap: (1) step sizes and inputs, (2) state updates,
        // (3) readout epilogues.
        constexpr int G = 8;
#pragma unroll
        for (int g0 = 0; g0 < T; g0 += G) {
          float dtv[G], uv[G], yv[G];
#pragma unroll
          for (int j = 0; j < G; ++j) {
            const int tt = g0 + j;
            const float xv = IO::lds(st + (tt * CH + lch) * ESZ);
            const float dv = IO::lds(st + XB + (tt * CH + lch) * ESZ);
            dtv[j] = step_size<IO>(p, dv, biasv);
            uv[j] = dtv[j] * xv;
            if (!OUT) kahan_add(S_sum, S_comp, dtv[j]);
          }
#pragma unroll
          for (int j = 0; j < G; ++j) {
            const int tt = g0 + j;
            yv[j] = step_states<NPT, TPC, POW, LTI, OUT, MFORM>(dtv[j], uv[j], Bt + tt * NST,
                                                                Ct + tt * NST, h, k);
          }
          if (OUT) {
#pragma unroll
            for (int j = 0; j < G; ++j) {
              const int tt = g0 + j;
              float y = yv[j];
#pragma unroll
              for (int off = 1; off < TPC; off <<= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
              if (sub == 0 && valid) {
                y = fmaf(Dv, IO::lds(st + (tt * CH + lch) * ESZ), y);
                if (gate) y *= silu(IO::lds(st + 2 * XB + (tt * CH + lch) * ESZ));
                IO::store(p.out, oidx + (int64_t)j * Dm, y);
              }
            }
          }
          oidx += (int64_t)G * Dm;
        }
      } else {
        for (int tt = 0; tt < nsteps; ++tt) one_step(tt);
      }
      // next tile: wait for its copies and widen its B / C rows
      bool okn = true;
      if (i + 1 < ntiles) {
        okn = mbar_wait(&full[(i + 1) % S], ((i + 1) / S) & 1);
        if (okn) widen_bc(i + 1);
      }
      if (__syncthreads_or(!okn)) {  // also: every thread is done with stage s
        if (tid == 0) atomicExch(p.status, kStatusTimeout);
        return false;
      }
      if (tid == 0 && i + S < ntiles) issue(i + S);
    }
    return true;
  };
  const bool done = use_pow ? run(std::true_type{}) : run(std::false_type{});
  if (!done) {
    // drain the copies still in flight (bounded) before the CTA exits
    const int last = ntiles - 1;
    for (int i = max(0, last - S + 1); i <= last; ++i) mbar_wait(&full[i % S], (i / S) & 1);
    return;
  }
  if (valid) store_results<NPT, PASS>(p, b, c, d, sub, h, S_sum);
}

// --------------------------------------------------------------- generic kernel

// Same computation for shapes a tensor map cannot describe (row pitch or B / C rows
// not a multiple of 16 bytes): plain coalesced loads with a register prefetch ring.
template <typename IO, int NPT, int TPC, bool LTI, int PASS>
__global__ void __launch_bounds__(kThreads)
scan_generic_kernel(const ScanParams p) {
  constexpr int NST = NPT * TPC;
  constexpr int CH = kThreads / TPC;
  constexpr bool OUT = (PASS == 1);
  constexpr bool MFORM = LTI || !IO::kFastDecay;

  __shared__ __align__(16) float sB[2][kTB * NST];
  __shared__ __align__(16) float sC[OUT ? 2 : 1][OUT ? kTB * NST : 4];

  const int N = p.dstate;
  const int64_t L = p.seqlen, Dm = p.dim;
  const int b = blockIdx.z, c = blockIdx.y;
  const int sub = threadIdx.x % TPC;
  const int64_t d = (int64_t)blockIdx.x * CH + threadIdx.x / TPC;
  const bool valid = d < Dm;
  const int64_t dd = valid ? d : Dm - 1;
  const int64_t t0 = (int64_t)c * p.chunk_len;
  const int64_t t1 = min(t0 + p.chunk_len, L);

  ChannelConsts<NPT> k;
  const bool structured = load_consts<NPT, TPC, LTI>(p, dd, sub, k);
  const bool use_pow = !LTI && p.pow_path && (IO::kFastDecay || TPC == 1) &&
                       __syncthreads_and(structured || !valid);
  const float biasv = p.bias ? p.bias[dd] : 0.f;
  const float Dv = p.Dskip ? p.Dskip[dd] : 0.f;
  float2 h[NPT / 2];
  start_state<NPT, PASS>(p, b, c, dd, sub, valid, h, k);

  if (!LTI) {
    for (int i = threadIdx.x; i < 2 * kTB * NST; i += kThreads) {
      (&sB[0][0])[i] = 0.f;
      if (OUT) (&sC[0][0])[i] = 0.f;
    }
    __syncthreads();
  }
  constexpr int kBCPerThread = (kTB * NST + kThreads - 1) / kThreads;
  float rB[kBCPerThread], rC[kBCPerThread];
  const int64_t bc_row0 = (int64_t)b * L;
  auto fetch_bc = [&](int64_t tb) {
#pragma unroll
    for (int j = 0; j < kBCPerThread; ++j) {
      const int e = threadIdx.x + j * kThreads;
      const int tt = e / N, n = e - tt * N;
      const int64_t t = tb + tt;
      const bool okk = (e < kTB * N) && (t < t1);
      rB[j] = okk ? IO::load(p.B, (bc_row0 + t) * N + n) : 0.f;
      if (OUT) rC[j] = okk ? IO::load(p.C, (bc_row0 + t) * N + n) : 0.f;
    }
  };
  auto stash_bc = [&](int buf) {
#pragma unroll
    for (int j = 0; j < kBCPerThread; ++j) {
      const int e = threadIdx.x + j * kThreads;
      if (e < kTB * N) {
        const int tt = e / N, n = e - tt * N;
        sB[buf][tt * NST + n] = rB[j];
        if (OUT) sC[buf][tt * NST + n] = rC[j];
      }
    }
  };
  if (!LTI) {
    fetch_bc(t0);
    stash_bc(0);
    __syncthreads();
  }

  const int64_t row = (int64_t)b * L;
  float rx[kPF], rd[kPF], rz[kPF];
  const bool gate = OUT && (p.z != nullptr);
#pragma unroll
  for (int j = 0; j < kPF; ++j) {
    const int64_t t = t0 + j;
    const bool okk = t < t1;
    const int64_t i = (row + (okk ? t : t0)) * Dm + dd;
    rx[j] = okk ? IO::load(p.x, i) : 0.f;
    rd[j] = okk ? IO::load(p.delta, i) : 0.f;
    rz[j] = (okk && gate) ? IO::load(p.z, i) : 0.f;
  }

  float S_sum = 0.f, S_comp = 0.f;
  int buf = 0;
  int64_t cur_i = (row + t0) * Dm + dd;
  int64_t pf_i = cur_i + kPF * Dm;

  auto body = [&](auto pow_tag) {
    constexpr bool POW = decltype(pow_tag)::value;
    for (int64_t tb = t0; tb < t1; tb += kTB) {
      const int64_t tend = min(tb + kTB, t1);
      const bool more = tend < t1;
      if (!LTI && more) fetch_bc(tend);
      const float* Bblk = sB[buf] + sub * NPT;
      const float* Cblk = sC[OUT ? buf : 0] + sub * NPT;
      for (int64_t tg = tb; tg < tend; tg += kPF) {
#pragma unroll
        for (int j = 0; j < kPF; ++j) {
          const int64_t t = tg + j;
          const float xv = rx[j], dv = rd[j], zv = rz[j];
          if (t + kPF < t1) {  // refill this ring slot with step t + kPF
            rx[j] = IO::load(p.x, pf_i);
            rd[j] = IO::load(p.delta, pf_i);
            if (gate) rz[j] = IO::load(p.z, pf_i);
          }
          pf_i += Dm;
          if (t < tend) {
            const float dt = step_size<IO>(p, dv, biasv);
            const float u = dt * xv;
            const int r = (int)(t - tb) * NST;
            float y = step_states<NPT, TPC, POW, LTI, OUT, MFORM>(dt, u, Bblk + r, Cblk + r, h, k);
            if (OUT) {
#pragma unroll
              for (int off = 1; off < TPC; off <<= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
              if (sub == 0 && valid) {
                y = fmaf(Dv, xv, y);
                if (gate) y *= silu(zv);
                IO::store(p.out, cur_i, y);
              }
            } else {
              kahan_add(S_sum, S_comp, dt);
            }
          }
          cur_i += Dm;
        }
      }
      if (!LTI && more) {
        stash_bc(buf ^ 1);
        __syncthreads();
        buf ^= 1;
      }
    }
  };
  if (use_pow) body(std::true_type{});
  else body(std::false_type{});

  if (valid) store_results<NPT, PASS>(p, b, c, d, sub, h, S_sum);
}

}  // namespace ssm
