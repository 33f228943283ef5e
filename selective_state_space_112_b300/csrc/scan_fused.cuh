// Selective-scan forward for sm_103a, two channels per lane, with the carry across
// sequence chunks formed in the same launch by a decoupled lookback.
//
// What is computed is the scan of scan_tile.cuh (pages "State-space models",
// sections "Discretization", "Mamba: selection", "The parallel scan",
// "Implementation"; "Structured State Space Models and Mamba", sections
// "Discretization Mechanics", the S6 section, "Hardware-Aware Parallel Associative
// Scan" and "The GPU Memory Hierarchy and Kernel Fusion"):
//   step = softplus(delta + bias); Abar = exp(step * A[d,n]); h = Abar h + step B x;
//   y = C . h + D x; out = y * silu(z).
// This kernel serves time-varying B and C, the fused scan's input term and padded
// state counts S = 4, 8, 16 held by one lane per channel.
//
// Design:
//  * Each lane of a consumer warp owns two adjacent channels (64 channels per warp).
//    The B and C rows of a step are shared by all channels, so a lane loads each row
//    once from shared memory for both of its channels: half the shared-memory traffic
//    per state update of one channel per lane, which together with the exponential
//    unit bounded the one-channel layout.  The per-(step, channel) work (softplus,
//    step * x, D x, silu gate, conversions) runs on the channel pair in f32x2 form.
//  * One producer warp feeds four consumer warps through a 4-stage ring of tiles
//    (x, delta, z: T steps x 256 channels; B, C: T x N) filled by TMA tensor copies and
//    completed on mbarriers; it widens the B and C rows to fp32 planes once per tile
//    and, after the consumers have written y over x in the stage, stores the y tile
//    with one TMA tensor store.  Every wait is bounded (2 s by %globaltimer).
//  * Sequence chunks (when batch x channels alone cannot fill the GPU).  A CTA takes
//    a ticket from a counter when it starts; tickets are given out chunk by chunk, so
//    a CTA only ever waits for CTAs that started before it.  With the associative
//    combine of the per-step maps ("The parallel scan": (a1, b1) then (a2, b2) =
//    (a1 a2, a2 b1 + b2), here (exp(A S1), H1) then (exp(A S2), H2) = (exp(A (S1 +
//    S2)), exp(A S2) H1 + H2) with S the sum of the steps):
//      phase 1  the CTA scans its chunk from a zero state (the first chunk from the
//               initial state) and publishes, per consumer warp, the chunk's step sum S
//               and end state H with a flag (1: aggregate; the first chunk publishes its
//               end state as an inclusive prefix, flag 2);
//      lookback each warp walks back over the preceding chunks of its channels,
//               folding aggregates until it meets an inclusive prefix, which gives its
//               carry-in; it publishes its own inclusive prefix exp(A S) h_in + H
//               (flag 2) so that later chunks stop there;
//      phase 2  the CTA scans its chunk again from the carry-in, writing out (and the
//               last chunk the final state).
//    The last chunk skips phase 1 (no one reads its aggregate).  The producer fetches
//    phase 2's first tiles while the consumers look back.  Only the per-chunk
//    aggregates and prefixes ((N + 1) and N floats per channel) and the flags touch
//    memory; Abar, Bbar and the states of every step stay on chip.
//  * Steps past the end of the sequence get step = 0 and u = 0 (an identity step).
//  * Precision as scan_tile.cuh: bf16 inputs form Abar with MUFU ex2; fp32 inputs
//    carry Abar - 1 (accurate expm1) and update h <- h + ((Abar - 1) h + Bbar x); rows
//    of A of the S4D-real form (n+1) A[d,0] take one exponential per step and channel.
#pragma once

#include "scan_tile.cuh"

namespace ssm {

struct FusedParams {
  const void* x;
  const void* delta;
  const void* z;          // nullable
  void* out;
  const float* A;         // (dim, N)
  const void* B;          // (batch, L, N) io dtype
  const void* C;
  const float* Dskip;     // nullable
  const float* bias;      // nullable
  float* final_state;     // nullable; written by the last chunk
  const float* h_init;    // nullable; initial state (batch, dim, N)
  // chunk carry (nchunks > 1): flags and ticket counter are zeroed before the launch
  unsigned* flags;        // (nchunks - 1, batch, nwb): 0 nothing, 1 aggregate, 2 prefix
  unsigned* ticket;       // counter of started CTAs
  float* agg_S;           // (nchunks - 1, batch, dim) step sums
  float* agg_H;           // (nchunks - 1, batch, dim, N) end states from a zero start
  float* pre_H;           // (nchunks - 1, batch, dim, N) inclusive prefixes (true end states)
  float* ws_h0;           // (batch, dim, N) copy of h_init kept by the first chunk, or null
  int* status;            // device status word
  int64_t batch, seqlen, dim;
  int dstate;
  int nchunks;
  int ncb;                // channel blocks (CTAs) per batch row
  int nwb;                // warp blocks (64 channels) per batch row
  int64_t chunk_len;
  int delta_softplus;
  int pow_path;
  int stall_tile;         // failure injection: the producer stops before this tile (-1 off)
  int hold_chunk;         // failure injection: this chunk never publishes (-1 off)
};

template <typename IO, int S>
struct FGeo {
  static constexpr int K = 2;                        // channels per lane
  static constexpr int NW = 4;                       // consumer warps
  static constexpr int NT = 32 * (NW + 1);
  static constexpr int CW = 32 * K;                  // channels per consumer warp
  static constexpr int CH = NW * CW;                 // channels per CTA (TMA box width)
  static constexpr int ESZ = IO::kBytes;
  static constexpr int T = ESZ == 2 ? 16 : 8;        // steps per tile
  static constexpr int ST = 4;                       // stages
  static constexpr int al(int v) { return (v + 127) / 128 * 128; }
  static constexpr int XB = al(T * CH * ESZ);        // one x / delta / z tile
  static constexpr int BB = al(T * S * ESZ);         // one raw B / C tile
  static constexpr int FB = al(T * S * 4);           // one fp32 B / C plane
  static constexpr int OFF_F = 3 * XB + 2 * BB;
  static constexpr int STAGE = OFF_F + 2 * FB;
  static constexpr int OFF_BAR = ST * STAGE;
  static constexpr int BYTES = OFF_BAR + 3 * ST * 8 + 16;
  static constexpr int R = 4;                        // steps per group of phases A/B/C
  static_assert(T % R == 0 && kChunkAlign % T == 0, "whole groups per tile, whole tiles per chunk");
  static_assert(S % 2 == 0 && S <= 16, "states are updated in pairs");
};

// Two adjacent values of the io dtype from shared memory, widened to fp32.
template <typename IO>
__device__ __forceinline__ float2 lds2(const unsigned char* p) {
  if (IO::kBytes == 2) return bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(p));
  return *reinterpret_cast<const float2*>(p);
}

// Two adjacent values stored in the io dtype (bf16: round to nearest even).
template <typename IO>
__device__ __forceinline__ void sts2(unsigned char* p, float2 v) {
  if (IO::kBytes == 2) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
  } else {
    *reinterpret_cast<float2*>(p) = v;
  }
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Lane 0 polls a flag until it reaches `want` or more (bounded by kWaitNs); the value
// seen (0 if the wait ran out) is returned to every lane of the warp.
__device__ __forceinline__ unsigned wait_flag(const unsigned* f, unsigned want, int lane) {
  unsigned v = 0;
  if (lane == 0) {
    v = ld_acquire(f);
    if (v < want) {
      const uint64_t start = globaltimer_ns();
      for (long long i = 0; i < kSpinLimit && v < want; ++i) {
        __nanosleep(64);
        v = ld_acquire(f);
        if (globaltimer_ns() - start > kWaitNs) break;
      }
    }
    if (v < want) v = 0;
  }
  return __shfl_sync(0xffffffffu, v, 0);
}

template <typename IO, int S>
__global__ void __launch_bounds__(FGeo<IO, S>::NT, 2)
scan_fused_kernel(const __grid_constant__ TmaMaps maps, const FusedParams p) {
  using Gm = FGeo<IO, S>;
  constexpr int NW = Gm::NW, CH = Gm::CH, CW = Gm::CW, T = Gm::T, ST = Gm::ST, R = Gm::R;
  constexpr int ESZ = Gm::ESZ, XB = Gm::XB, BB = Gm::BB, FB = Gm::FB;
  constexpr bool MFORM = !IO::kFastDecay;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Gm::OFF_BAR);
  uint64_t* ready = full + ST;
  uint64_t* empty = ready + ST;
  unsigned* tk_smem = reinterpret_cast<unsigned*>(empty + ST);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.dstate;
  const int64_t L = p.seqlen, Dm = p.dim;

  // ---- work item: chunk-major tickets when chunked, else the block index
  unsigned item = blockIdx.x;
  if (p.nchunks > 1) {
    if (tid == 0) *tk_smem = atomicAdd(p.ticket, 1u);
  }
  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&ready[s], 1);
      mbar_init(&empty[s], NW);
    }
    mbar_fence_init();
  }
  for (int s = 0; s < ST; ++s)
    for (int e = tid; e < 2 * FB / 4; e += Gm::NT)
      reinterpret_cast<float*>(smem + s * Gm::STAGE + Gm::OFF_F)[e] = 0.f;
  __syncthreads();
  if (p.nchunks > 1) item = *tk_smem;
  const int per_chunk = (int)(p.batch * p.ncb);
  const int chunk = (int)(item / per_chunk);
  const int rem = (int)(item - (unsigned)chunk * per_chunk);
  const int b = rem / p.ncb;
  const int cb = rem - b * p.ncb;
  if (chunk >= p.nchunks) return;  // cannot happen: the grid holds one ticket per CTA
  const int c0 = cb * CH;
  const int64_t t0 = (int64_t)chunk * p.chunk_len;
  const int64_t t1 = min(t0 + p.chunk_len, L);
  const int ntiles = (int)((t1 - t0 + T - 1) / T);
  const bool last = chunk == p.nchunks - 1;
  const int n1 = last ? 0 : ntiles;  // phase-1 tiles (the aggregate); then ntiles phase-2 tiles
  const int nv = n1 + ntiles;
  const bool gate = p.z != nullptr;
  auto stage = [&](int v) { return smem + (v % ST) * Gm::STAGE; };

  // ======================================================= producer warp
  if (warp == NW) {
    const bool sp = p.delta_softplus != 0;
    const uint32_t bytes1 = (uint32_t)(2 * T * CH * ESZ + T * N * ESZ);
    const uint32_t bytes2 = (uint32_t)((2 + (gate ? 1 : 0)) * T * CH * ESZ + 2 * T * N * ESZ);
    int issued = 0, released = 0;
    // waits until the consumers release virtual tile j; for a phase-2 tile, stores its
    // y tile (clipped at the sequence end and the last channel)
    auto release = [&](int j) {
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&empty[j % ST], (j / ST) & 1);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      released = j + 1;
      if (j >= n1 && lane == 0) {
        tma_store_3d(&maps.out, stage(j), c0, (int)(t0 + (int64_t)(j - n1) * T), b);
        bulk_commit();
        bulk_wait_read<0>();
      }
      return true;
    };
    auto issue = [&](int j) {
      if (j >= ST && !release(j - ST)) return false;
      unsigned char* st = stage(j);
      const bool ph2 = j >= n1;
      const int ts = (int)(t0 + (int64_t)(ph2 ? j - n1 : j) * T);
      if (lane == 0) {
        uint64_t* bar = &full[j % ST];
        mbar_arrive_expect_tx(bar, ph2 ? bytes2 : bytes1);
        tma_load_3d(st, &maps.x, c0, ts, b, bar);
        tma_load_3d(st + XB, &maps.delta, c0, ts, b, bar);
        tma_load_3d(st + 3 * XB, &maps.B, 0, ts, b, bar);
        if (ph2) {
          if (gate) tma_load_3d(st + 2 * XB, &maps.z, c0, ts, b, bar);
          tma_load_3d(st + 3 * XB + BB, &maps.C, 0, ts, b, bar);
        }
      }
      issued = j + 1;
      return true;
    };
    // widen the raw B (and, in phase 2, C) rows to fp32 planes; with softplus, rows
    // past the sequence end get delta = -inf (step 0: an identity step)
    auto prepare = [&](int v) {
      unsigned char* st = stage(v);
      const bool ph2 = v >= n1;
      float* fb = reinterpret_cast<float*>(st + Gm::OFF_F);
      constexpr int VE = 16 / ESZ;
      constexpr int PER_PLANE = T * S / VE;
      for (int c = lane; c < (ph2 ? 2 : 1) * PER_PLANE; c += 32) {
        const int plane = c / PER_PLANE, e = (c - plane * PER_PLANE) * VE;
        const uint4 w = *reinterpret_cast<const uint4*>(st + 3 * XB + plane * BB + e * ESZ);
        float4* dst = reinterpret_cast<float4*>(fb + plane * (FB / 4) + e);
        if (ESZ == 2) {
          const float2 a0 = bf16x2_to_f2(w.x), a1 = bf16x2_to_f2(w.y);
          const float2 a2 = bf16x2_to_f2(w.z), a3 = bf16x2_to_f2(w.w);
          dst[0] = make_float4(a0.x, a0.y, a1.x, a1.y);
          dst[1] = make_float4(a2.x, a2.y, a3.x, a3.y);
        } else {
          dst[0] = make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                               __uint_as_float(w.w));
        }
      }
      if (sp) {
        const int i = ph2 ? v - n1 : v;
        const int valid = (int)min((int64_t)T, t1 - (t0 + (int64_t)i * T));
        unsigned char* dl = st + XB;
        for (int e = valid * CH + lane; e < T * CH; e += 32) {
          if (ESZ == 2) *reinterpret_cast<unsigned short*>(dl + 2 * e) = 0xFF80u;
          else *reinterpret_cast<uint32_t*>(dl + 4 * e) = 0xFF800000u;
        }
      }
    };
    bool ok = true;
    int waited = 0;
    for (int j = 0; j < ST - 1 && j < nv && ok; ++j) ok = issue(j);
    for (int v = 0; v < nv && ok; ++v) {
      if (v == p.stall_tile) break;  // injected stall: tile v is never handed over
      bool landed = true;
      if (lane == 0) landed = mbar_wait(&full[v % ST], (v / ST) & 1);
      if (!__shfl_sync(0xffffffffu, landed, 0)) {
        ok = false;
        break;
      }
      waited = v + 1;
      prepare(v);
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ready[v % ST]);
      if (v + ST - 1 < nv) ok = issue(v + ST - 1);
    }
    for (int j = released; j < nv && ok; ++j) ok = release(j);
    if (lane == 0) bulk_wait<0>();
    if (!ok && lane == 0) atomicExch(p.status, kStatusTimeout);
    if (lane == 0)
      for (int j = waited; j < issued; ++j) mbar_wait(&full[j % ST], (j / ST) & 1);
    return;
  }

  // ======================================================= consumer warps
  const int cl = warp * CW + 2 * lane;  // first of the lane's two channels within the CTA
  const int64_t d0 = (int64_t)c0 + cl;
  const bool val0 = d0 < Dm, val1 = d0 + 1 < Dm;
  const int64_t dd0 = val0 ? d0 : Dm - 1, dd1 = val1 ? d0 + 1 : Dm - 1;
  const int wb = (c0 + warp * CW) / CW;  // this warp's block of 64 channels in the row

  // per-channel constants: A (x log2 e for the ex2 form), the S4D-real test
  float2 Ak[2][S / 2];
  bool structured = true;
  float a00[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int64_t dd = k ? dd1 : dd0;
    a00[k] = p.A[dd * N];
#pragma unroll
    for (int j = 0; j < S; ++j) {
      const float a = (j < N) ? p.A[dd * N + j] : 0.f;
      const float v = MFORM ? a : a * kLog2e;
      if (j & 1) Ak[k][j / 2].y = v;
      else Ak[k][j / 2].x = v;
      if (j < N && a != (float)(j + 1) * a00[k]) structured = false;
    }
  }
  const bool use_pow = p.pow_path && __all_sync(0xffffffffu, structured || !val0);
  const float2 bias2 = p.bias ? f2(p.bias[dd0], p.bias[dd1]) : f2(0.f, 0.f);
  const float2 D2 = p.Dskip ? f2(p.Dskip[dd0], p.Dskip[dd1]) : f2(0.f, 0.f);

  // initial state of the chunk's first scan: the initial state for the first chunk
  // (which, when the sequence is chunked, keeps a copy for its second scan: the last
  // chunk overwrites final_state, which may be the buffer h_init points to), else 0
  float2 h[2][S / 2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int64_t sidx = ((int64_t)b * Dm + (k ? dd1 : dd0)) * N;
#pragma unroll
    for (int i = 0; i < S / 2; ++i) {
      float v0 = 0.f, v1 = 0.f;
      if (chunk == 0 && p.h_init) {
        if (2 * i < N) v0 = p.h_init[sidx + 2 * i];
        if (2 * i + 1 < N) v1 = p.h_init[sidx + 2 * i + 1];
        if (p.ws_h0 && (k ? val1 : val0)) {
          if (2 * i < N) p.ws_h0[sidx + 2 * i] = v0;
          if (2 * i + 1 < N) p.ws_h0[sidx + 2 * i + 1] = v1;
        }
      }
      h[k][i] = f2(v0, v1);
    }
  }

  float2 Ssum = f2(0.f, 0.f), Scomp = f2(0.f, 0.f);  // phase 1: the chunk's step sums

  // One phase over its tiles (virtual tiles v0 .. v0 + ntiles - 1).  OUT: phase 2
  // (readout, gate, y into the stage); otherwise phase 1 (state and step sum only).
  auto run = [&](auto pow_tag, auto out_tag, int v0) -> bool {
    constexpr bool POW = decltype(pow_tag)::value;
    constexpr bool OUT = decltype(out_tag)::value;
    for (int i = 0; i < ntiles; ++i) {
      const int v = v0 + i;
      if (!mbar_wait(&ready[v % ST], (v / ST) & 1)) return false;
      unsigned char* st = stage(v);
      const int64_t ts = t0 + (int64_t)i * T;
      const int nvalid = (int)min((int64_t)T, t1 - ts);
      const float* bplane = reinterpret_cast<const float*>(st + Gm::OFF_F);
      const float* cplane = bplane + FB / 4;
#pragma unroll
      for (int r0 = 0; r0 < T; r0 += R) {
        auto xo = [&](int q) { return ((r0 + q) * CH + cl) * ESZ; };
        float2 xv[R], dq[R], p1[R], uv[R];
        // phase A: per (step, channel pair) work
#pragma unroll
        for (int q = 0; q < R; ++q) {
          xv[q] = lds2<IO>(st + xo(q));
          dq[q] = __fadd2_rn(lds2<IO>(st + XB + xo(q)), bias2);
        }
        if (p.delta_softplus) {
#pragma unroll
          for (int q = 0; q < R; ++q)
            dq[q] = f2(softplus<!IO::kFastDecay>(dq[q].x), softplus<!IO::kFastDecay>(dq[q].y));
        } else {
#pragma unroll
          for (int q = 0; q < R; ++q)
            if (r0 + q >= nvalid) dq[q] = f2(0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < R; ++q) {
          uv[q] = __fmul2_rn(dq[q], xv[q]);
          p1[q] = dq[q];
          if (POW)
            p1[q] = MFORM ? f2(expm1f(dq[q].x * a00[0]), expm1f(dq[q].y * a00[1]))
                          : f2(ex2(dq[q].x * a00[0] * kLog2e), ex2(dq[q].y * a00[1] * kLog2e));
        }
        if (!OUT) {
          float2 tsum[R];
#pragma unroll
          for (int q = 0; q < R; ++q) tsum[q] = dq[q];
#pragma unroll
          for (int w = 1; w < R; w *= 2)
#pragma unroll
            for (int q = 0; q + w < R; q += 2 * w) tsum[q] = __fadd2_rn(tsum[q], tsum[q + w]);
          kahan_add(Ssum.x, Scomp.x, tsum[0].x);
          kahan_add(Ssum.y, Scomp.y, tsum[0].y);
        }
        // phase B: the state updates, B and C rows loaded once for both channels
        float2 yv[R];
#pragma unroll
        for (int q = 0; q < R; ++q) {
          const int t = r0 + q;
          float2 bv[S / 2], cv[S / 2];
          load_row<F32, S>(reinterpret_cast<const unsigned char*>(bplane + t * S), bv);
          if (OUT) load_row<F32, S>(reinterpret_cast<const unsigned char*>(cplane + t * S), cv);
          float yk[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float pk = k ? p1[q].y : p1[q].x;
            const float uk = k ? uv[q].y : uv[q].x;
            float2 a[S / 2];
            if (POW) {
              float pw[S];
              pw[0] = pk;
#pragma unroll
              for (int e = 2; e <= S; ++e) {
                const float xx = (e & 1) ? pw[e - 2] : pw[e / 2 - 1];
                const float yy = (e & 1) ? pk : pw[e / 2 - 1];
                pw[e - 1] = MFORM ? mcomb(xx, yy) : xx * yy;
              }
#pragma unroll
              for (int j = 0; j < S / 2; ++j) a[j] = f2(pw[2 * j], pw[2 * j + 1]);
            } else if (MFORM) {
#pragma unroll
              for (int j = 0; j < S / 2; ++j)
                a[j] = f2(expm1f(pk * Ak[k][j].x), expm1f(pk * Ak[k][j].y));
            } else {
              const float2 dt2 = f2(pk, pk);
#pragma unroll
              for (int j = 0; j < S / 2; ++j) {
                const float2 e = __fmul2_rn(dt2, Ak[k][j]);
                a[j] = f2(ex2(e.x), ex2(e.y));
              }
            }
            const float2 u2 = f2(uk, uk);
#pragma unroll
            for (int j = 0; j < S / 2; ++j) {
              const float2 ub = __fmul2_rn(u2, bv[j]);
              h[k][j] = MFORM ? __fadd2_rn(h[k][j], __ffma2_rn(a[j], h[k][j], ub))
                              : __ffma2_rn(a[j], h[k][j], ub);
            }
            yk[k] = OUT ? readout<S>(cv, h[k]) : 0.f;
          }
          yv[q] = f2(yk[0], yk[1]);
        }
        if (OUT) {  // phase C: D x, gate, y over x in the stage
#pragma unroll
          for (int q = 0; q < R; ++q) {
            float2 y = __ffma2_rn(D2, xv[q], yv[q]);
            if (gate) {
              const float2 zz = lds2<IO>(st + 2 * XB + xo(q));
              y = __fmul2_rn(y, f2(silu(zz.x), silu(zz.y)));
            }
            sts2<IO>(st + xo(q), y);
          }
        }
      }
      if (OUT) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[v % ST]);
    }
    return true;
  };
  auto fail = [&]() {
    if (lane == 0) atomicExch(p.status, kStatusTimeout);
  };

  if (!last) {
    // ---- phase 1: the chunk's aggregate (the first chunk: its true end state)
    const bool done = use_pow ? run(std::true_type{}, std::false_type{}, 0)
                              : run(std::false_type{}, std::false_type{}, 0);
    if (!done) return fail();
    const int64_t ci = (int64_t)chunk * p.batch + b;
    if (chunk != p.hold_chunk) {
      float* H = (chunk == 0 ? p.pre_H : p.agg_H) + (ci * Dm + d0) * N;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (!(k ? val1 : val0)) continue;
#pragma unroll
        for (int j = 0; j < S / 2; ++j) {
          if (2 * j < N) H[k * N + 2 * j] = h[k][j].x;
          if (2 * j + 1 < N) H[k * N + 2 * j + 1] = h[k][j].y;
        }
      }
      if (chunk != 0) {
        const float2 tot = f2(Ssum.x - Scomp.x, Ssum.y - Scomp.y);
        if (val0) p.agg_S[ci * Dm + d0] = tot.x;
        if (val1) p.agg_S[ci * Dm + d0 + 1] = tot.y;
      }
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        st_release(p.flags + ci * p.nwb + wb, chunk == 0 ? 2u : 1u);
      }
    }
  }

  float2 hin[2][S / 2];  // the chunk's carry-in
  if (chunk == 0) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t sidx = ((int64_t)b * Dm + (k ? dd1 : dd0)) * N;
#pragma unroll
      for (int i = 0; i < S / 2; ++i) {
        if (last) {
          hin[k][i] = h[k][i];  // one chunk: no first scan ran, h holds the initial state
        } else {
          float v0 = 0.f, v1 = 0.f;
          if (p.ws_h0 && (k ? val1 : val0)) {
            if (2 * i < N) v0 = p.ws_h0[sidx + 2 * i];
            if (2 * i + 1 < N) v1 = p.ws_h0[sidx + 2 * i + 1];
          }
          hin[k][i] = f2(v0, v1);
        }
      }
    }
  } else {
    // ---- lookback: fold the preceding chunks' aggregates back to an inclusive prefix
    float2 Hacc[2][S / 2];
    float2 Sacc = f2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int j = 0; j < S / 2; ++j) Hacc[k][j] = f2(0.f, 0.f);
    bool found = false;
    for (int c = chunk - 1; c >= 0 && !found; --c) {
      const int64_t ci = (int64_t)c * p.batch + b;
      const unsigned f = wait_flag(p.flags + ci * p.nwb + wb, 1u, lane);
      if (f == 0) return fail();
      __syncwarp();  // lane 0's acquire orders the other lanes' reads below
      found = f >= 2;
      const float* src = (found ? p.pre_H : p.agg_H) + (ci * Dm + d0) * N;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float sk = k ? Sacc.y : Sacc.x;
#pragma unroll
        for (int j = 0; j < S / 2; ++j) {
          // H_acc += exp(A S_acc) H_c   (the later chunks' decay applied to chunk c)
          const bool v = k ? val1 : val0;
          const float hx = (v && 2 * j < N) ? __ldcg(src + k * N + 2 * j) : 0.f;
          const float hy = (v && 2 * j + 1 < N) ? __ldcg(src + k * N + 2 * j + 1) : 0.f;
          const float2 e = MFORM ? f2(expf(sk * Ak[k][j].x), expf(sk * Ak[k][j].y))
                                 : f2(ex2(sk * Ak[k][j].x), ex2(sk * Ak[k][j].y));
          Hacc[k][j] = __ffma2_rn(e, f2(hx, hy), Hacc[k][j]);
        }
      }
      if (!found) {
        const float s0 = val0 ? __ldcg(p.agg_S + ci * Dm + d0) : 0.f;
        const float s1 = val1 ? __ldcg(p.agg_S + ci * Dm + d0 + 1) : 0.f;
        Sacc = __fadd2_rn(Sacc, f2(s0, s1));
      }
    }
    // the carry-in; then this chunk's inclusive prefix exp(A S) h_in + H for later chunks
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int j = 0; j < S / 2; ++j) hin[k][j] = Hacc[k][j];
    if (!last && chunk != p.hold_chunk) {
      const int64_t ci = (int64_t)chunk * p.batch + b;
      const float2 tot = f2(Ssum.x - Scomp.x, Ssum.y - Scomp.y);
      float* P = p.pre_H + (ci * Dm + d0) * N;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (!(k ? val1 : val0)) continue;
        const float sk = k ? tot.y : tot.x;
#pragma unroll
        for (int j = 0; j < S / 2; ++j) {
          const float2 e = MFORM ? f2(expf(sk * Ak[k][j].x), expf(sk * Ak[k][j].y))
                                 : f2(ex2(sk * Ak[k][j].x), ex2(sk * Ak[k][j].y));
          const float2 v = __ffma2_rn(e, hin[k][j], h[k][j]);
          if (2 * j < N) P[k * N + 2 * j] = v.x;
          if (2 * j + 1 < N) P[k * N + 2 * j + 1] = v.y;
        }
      }
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        st_release(p.flags + ci * p.nwb + wb, 2u);
      }
    }
  }

  // ---- phase 2: the chunk from its carry-in, writing out
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int j = 0; j < S / 2; ++j) h[k][j] = hin[k][j];
  const bool done = use_pow ? run(std::true_type{}, std::true_type{}, n1)
                            : run(std::false_type{}, std::true_type{}, n1);
  if (!done) return fail();
  if (last && p.final_state) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (!(k ? val1 : val0)) continue;
      float* F = p.final_state + ((int64_t)b * Dm + d0 + k) * N;
#pragma unroll
      for (int j = 0; j < S / 2; ++j) {
        if (2 * j < N) F[2 * j] = h[k][j].x;
        if (2 * j + 1 < N) F[2 * j + 1] = h[k][j].y;
      }
    }
  }
}

}  // namespace ssm
