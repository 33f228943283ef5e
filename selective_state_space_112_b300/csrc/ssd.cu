// Mamba-2 SSD layer, forward: the scan with one scalar decay per head, evaluated
// chunk by chunk in its dual (masked-attention) form on the tensor cores.
//
// Pages: "State-space models", section "The parallel scan" (A a scalar times the
// identity per head turns the scan into blocks of matrix products); "Structured
// State Space Models and Mamba", section "State Space Duality and Mamba-2"
// (Y = (L o (Q K^T)) V with a 1-semiseparable decay mask L).
//
// One CTA owns one (batch row, head, block of PB channels) and walks its sequence in
// chunks of Q = 64 steps, carrying that (N, PB) part of the state in fp32 registers.
// With S_i the running sum of step * A inside the chunk, for steps i, j of the chunk:
//   M[i][j]   = (C_i . B_j) exp(S_i - S_j) step_j            j <= i, else 0
//   y_i       = exp(S_i) C_i . h_prev  +  sum_j M[i][j] x_j  +  D x_i
//   h_next    = exp(S_last) h_prev  +  sum_j B_j (exp(S_last - S_j) step_j x_j)^T
// Four products per chunk on the tensor cores (bf16 operands, fp32 accumulation):
// C B^T (Q x Q over N), C h_prev (Q x PB over N), M X (Q x PB over Q) and
// B^T Xw (N x PB over Q).  The operands formed inside the kernel in fp32 (M, Xw and
// the carried state) enter as a pair of bf16 values, hi = bf16(v) and
// lo = bf16(v - hi), with one product each: about 16 significant bits, where one
// bf16 rounding (8 bits) of the state would show in y at the 1e-2 level.  C, B and x
// are bf16 inputs and exact.  Inputs stream through a two-stage cp.async ring.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "scan_internal.h"
#include "ssd_tc.cuh"
#include "ssm_ssd.h"

namespace {

constexpr int Q = 64;          // chunk length in steps
constexpr int P = 64;          // channels per head
constexpr int NWARP = 8;
constexpr int NTHR = NWARP * 32;

template <int N, int PB>
struct SsdSmem {
  static constexpr int XS = PB + 8;  // row stride (bf16 elements) of the x, Xw and state tiles
  static constexpr int MS = Q + 8;   // row stride of the M tile
  static constexpr int BS = N + 8;   // row stride of the B and C tiles
  static constexpr int YS = PB + 4;  // row stride (fp32) of the y tile
  static constexpr int X_BYTES = Q * XS * 2;
  static constexpr int M_BYTES = Q * MS * 2;
  static constexpr int S_BYTES = N * XS * 2;
  static constexpr int BC_BYTES = Q * BS * 2;
  // the gate z rides in the stage (x, B, C, z of one chunk) unless it would not fit
  static constexpr bool Z_SMEM = 2 * (2 * X_BYTES + 2 * BC_BYTES) + 2 * Q * MS * 2 + 2 * X_BYTES +
                                     Q * YS * 4 + 2 * N * XS * 2 + 8 * Q * 4 <= 232448;
  static constexpr int OFF_Z = X_BYTES + 2 * BC_BYTES;
  static constexpr int STAGE = (Z_SMEM ? 2 : 1) * X_BYTES + 2 * BC_BYTES;
  static constexpr int OFF_M = 2 * STAGE;                // M hi, M lo
  static constexpr int OFF_XW = OFF_M + 2 * M_BYTES;     // Xw hi, Xw lo
  static constexpr int OFF_Y = OFF_XW + 2 * X_BYTES;
  static constexpr int OFF_S = OFF_Y + Q * YS * 4;       // state hi, state lo
  static constexpr int OFF_V = OFF_S + 2 * S_BYTES;      // per-step vectors, two chunks
  static constexpr int BYTES = OFF_V + 8 * Q * 4;
  static_assert(BYTES <= 232448, "dynamic shared memory of one CTA");
};

struct SsdParams {
  const __nv_bfloat16* x;
  const __nv_bfloat16* dt;
  const __nv_bfloat16* B;
  const __nv_bfloat16* C;
  const __nv_bfloat16* z;
  const float* A;
  const float* D;
  const float* dt_bias;
  __nv_bfloat16* out;
  float* state;
  int64_t L;
  int H, G, hpg;  // heads, groups, heads per group
  int softplus, state_in;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte global -> shared copy; ok == false fills the 16 bytes with zeros
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// d += a (16 x 16, row) * b (16 x 8, col), bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Addresses of one lane for an ldmatrix.x4 (stride in bf16 elements).
// A operand, 16 x 16 at (m0, k0) of a [m][k] tile.
__device__ __forceinline__ uint32_t a_addr(uint32_t base, int stride, int m0, int k0, int lane) {
  return base + 2u * ((m0 + (lane & 7) + ((lane >> 3) & 1) * 8) * stride + k0 + (lane >> 4) * 8);
}
// A operand, 16 x 16 at (m0, k0), from a [k][m] tile (transposing load).
__device__ __forceinline__ uint32_t a_addr_t(uint32_t base, int stride, int m0, int k0, int lane) {
  return base + 2u * ((k0 + (lane & 7) + (lane >> 4) * 8) * stride + m0 + ((lane >> 3) & 1) * 8);
}
// B operands of the two 8-wide column tiles n0, n0 + 8 over k0..k0+15, from a [n][k] tile.
__device__ __forceinline__ uint32_t b_addr(uint32_t base, int stride, int n0, int k0, int lane) {
  return base + 2u * ((n0 + (lane & 7) + (lane >> 4) * 8) * stride + k0 + ((lane >> 3) & 1) * 8);
}
// The same from a [k][n] tile (transposing load).
__device__ __forceinline__ uint32_t b_addr_t(uint32_t base, int stride, int n0, int k0, int lane) {
  return base + 2u * ((k0 + (lane & 7) + ((lane >> 3) & 1) * 8) * stride + n0 + (lane >> 4) * 8);
}

__device__ __forceinline__ float softplus_f(float v) { return v > 20.f ? v : log1pf(expf(v)); }

// v = hi + lo with both parts bf16 (lo holds what hi rounds away)
__device__ __forceinline__ void split2(float a, float b, __nv_bfloat162& hi, __nv_bfloat162& lo) {
  hi = __floats2bfloat162_rn(a, b);
  const float2 h = __bfloat1622float2(hi);
  lo = __floats2bfloat162_rn(a - h.x, b - h.y);
}
// the gate and the decay mask take the hardware exponential (relative error near
// 2^-21, far inside the 16-bit operands and the bf16 output)
__device__ __forceinline__ float silu_f(float v) { return __fdividef(v, 1.f + __expf(-v)); }

template <int N, int PB>
__global__ void __launch_bounds__(NTHR, 1) ssd_fwd_kernel(const SsdParams p) {
  using Sm = SsdSmem<N, PB>;
  constexpr int XS = Sm::XS, MS = Sm::MS, BS = Sm::BS, YS = Sm::YS;
  constexpr int YNT = PB / 16;  // 8-column tiles of y per warp (two warps across PB)
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, cq = lane & 3;
  const int h = blockIdx.x / (P / PB), pc = (blockIdx.x % (P / PB)) * PB;  // head, first channel
  const int b = blockIdx.y, g = h / p.hpg;
  const int64_t L = p.L;
  const int nch = (int)((L + Q - 1) / Q);
  const float Ah = p.A[h];
  const float Dh = p.D ? p.D[h] : 0.f;
  const float biash = p.dt_bias ? p.dt_bias[h] : 0.f;

  // per-step vectors of a chunk (chunk c in buffer c % 2): S_i, exp(S_i),
  // exp(S_last - S_j) step_j, step_j
  float* const vbuf = reinterpret_cast<float*>(smem + Sm::OFF_V);
  __nv_bfloat16* Ms = reinterpret_cast<__nv_bfloat16*>(smem + Sm::OFF_M);    // hi; lo follows
  __nv_bfloat16* Xws = reinterpret_cast<__nv_bfloat16*>(smem + Sm::OFF_XW);  // hi; lo follows
  float* Ys = reinterpret_cast<float*>(smem + Sm::OFF_Y);
  __nv_bfloat16* Ss = reinterpret_cast<__nv_bfloat16*>(smem + Sm::OFF_S);    // state [n][p], hi; lo follows
  constexpr int M_LO = Sm::M_BYTES / 2, X_LO = Sm::X_BYTES / 2, S_LO = Sm::S_BYTES / 2;  // in elements

  // chunk c's x, B and C rows into stage c % 2 (rows past the end are zeros)
  auto issue = [&](int c) {
    unsigned char* st = smem + (c & 1) * Sm::STAGE;
    const int64_t t0 = (int64_t)c * Q;
    for (int i = tid; i < Q * (PB / 8); i += NTHR) {
      const int r = i / (PB / 8), k = i % (PB / 8);
      const bool ok = t0 + r < L;
      const int64_t t = ok ? t0 + r : t0;
      const int64_t off = (((int64_t)b * L + t) * p.H + h) * P + pc + k * 8;
      cp_async16(smem_u32(st + (r * XS + k * 8) * 2), p.x + off, ok);
      if (Sm::Z_SMEM && p.z) cp_async16(smem_u32(st + Sm::OFF_Z + (r * XS + k * 8) * 2), p.z + off, ok);
    }
    for (int i = tid; i < Q * (N / 8); i += NTHR) {
      const int r = i / (N / 8), k = i % (N / 8);
      const bool ok = t0 + r < L;
      const int64_t t = ok ? t0 + r : t0;
      const int64_t off = (((int64_t)b * L + t) * p.G + g) * N + k * 8;
      cp_async16(smem_u32(st + Sm::X_BYTES + (r * BS + k * 8) * 2), p.B + off, ok);
      cp_async16(smem_u32(st + Sm::X_BYTES + Sm::BC_BYTES + (r * BS + k * 8) * 2), p.C + off, ok);
    }
  };

  // the state tile of this warp: WM warps along N, WN along the CTA's PB channels
  constexpr int WM = (N / 16 < NWARP) ? N / 16 : NWARP;
  constexpr int WN = NWARP / WM;
  constexpr int SMT = N / 16 / WM;  // 16-row tiles per warp
  constexpr int SNT = PB / 8 / WN;  // 8-column tiles per warp
  static_assert(SNT % 2 == 0, "column tiles are loaded in pairs");
  const int sm0 = (warp % WM) * SMT * 16;
  const int sn0 = (warp / WM) * SNT * 8;
  float sacc[SMT][SNT][4];
  const int64_t sbase = ((int64_t)b * p.H + h) * P * N;  // (b, h) block of the (b, H, P, N) state
#pragma unroll
  for (int mt = 0; mt < SMT; ++mt)
#pragma unroll
    for (int nt = 0; nt < SNT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = sm0 + mt * 16 + gq + (e >> 1) * 8, pp = sn0 + nt * 8 + 2 * cq + (e & 1);
        sacc[mt][nt][e] = p.state_in ? p.state[sbase + (int64_t)(pc + pp) * N + n] : 0.f;
      }
  // the state as the bf16 hi / lo operands of the next chunk's readout
  auto store_state = [&]() {
#pragma unroll
    for (int mt = 0; mt < SMT; ++mt)
#pragma unroll
      for (int nt = 0; nt < SNT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int n = sm0 + mt * 16 + gq + hh * 8, pp = sn0 + nt * 8 + 2 * cq;
          __nv_bfloat162 hi, lo;
          split2(sacc[mt][nt][2 * hh], sacc[mt][nt][2 * hh + 1], hi, lo);
          *reinterpret_cast<__nv_bfloat162*>(Ss + n * XS + pp) = hi;
          *reinterpret_cast<__nv_bfloat162*>(Ss + S_LO + n * XS + pp) = lo;
        }
  };
  bool have_state = p.state_in != 0;
  if (have_state) store_state();

  // warp 0: the raw steps of chunk c, two per lane (read one chunk ahead of use)
  auto load_dt = [&](int c, float (&r)[2]) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t t = (int64_t)c * Q + 2 * lane + k;
      r[k] = (c < nch && t < L) ? __bfloat162float(p.dt[((int64_t)b * L + t) * p.H + h]) : 0.f;
    }
  };
  // warp 0: step sizes and running sums S_i of step * A over chunk c
  auto make_v = [&](int c, const float (&r)[2]) {
    float* V = vbuf + (c & 1) * 4 * Q;
    float stp[2], a2[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t t = (int64_t)c * Q + 2 * lane + k;
      float s = 0.f;  // steps past the end: identity
      if (t < L) {
        const float v = r[k] + biash;
        s = p.softplus ? softplus_f(v) : v;
      }
      stp[k] = s;
      a2[k] = s * Ah;
    }
    float incl = a2[0] + a2[1];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    const float c1 = incl, c0 = incl - a2[1];
    const float clast = __shfl_sync(0xffffffffu, incl, 31);
    V[2 * lane] = c0;
    V[2 * lane + 1] = c1;
    V[Q + 2 * lane] = expf(c0);
    V[Q + 2 * lane + 1] = expf(c1);
    V[2 * Q + 2 * lane] = expf(clast - c0) * stp[0];
    V[2 * Q + 2 * lane + 1] = expf(clast - c1) * stp[1];
    V[3 * Q + 2 * lane] = stp[0];
    V[3 * Q + 2 * lane + 1] = stp[1];
  };
  float dtn[2] = {0.f, 0.f};  // warp 0: raw steps of the next chunk
  if (warp == 0) {
    float r0[2];
    load_dt(0, r0);
    make_v(0, r0);
    load_dt(1, dtn);
  }

  issue(0);
  cp_async_commit();
  if (nch > 1) issue(1);
  cp_async_commit();

  for (int c = 0; c < nch; ++c) {
    cp_async_wait1();
    __syncthreads();  // chunk c resident; the previous chunk's readers are done
    const unsigned char* st = smem + (c & 1) * Sm::STAGE;
    const uint32_t xs_u = smem_u32(st), bs_u = smem_u32(st + Sm::X_BYTES),
                   cs_u = smem_u32(st + Sm::X_BYTES + Sm::BC_BYTES);
    const __nv_bfloat16* Xs = reinterpret_cast<const __nv_bfloat16*>(st);
    const int64_t t0 = (int64_t)c * Q;

    const float* cumS = vbuf + (c & 1) * 4 * Q;
    const float* eS = cumS + Q;
    const float* wS = eS + Q;
    const float* sS = wS + Q;

    // Xw[j][p] = x[j][p] exp(S_last - S_j) step_j: the inputs weighted by their decay
    // to the chunk end (hi / lo)
    static_assert(Q * (PB / 8) % NTHR == 0, "whole pieces per thread");
#pragma unroll
    for (int i = tid; i < Q * (PB / 8); i += NTHR) {
      const int r = i / (PB / 8), k = i % (PB / 8);
      const uint4 v = *reinterpret_cast<const uint4*>(Xs + r * XS + k * 8);
      const float wr = wS[r];
      const __nv_bfloat162* pv = reinterpret_cast<const __nv_bfloat162*>(&v);
      uint4 vh, vl;
      __nv_bfloat162* ph = reinterpret_cast<__nv_bfloat162*>(&vh);
      __nv_bfloat162* pl = reinterpret_cast<__nv_bfloat162*>(&vl);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(pv[e]);
        split2(f.x * wr, f.y * wr, ph[e], pl[e]);
      }
      *reinterpret_cast<uint4*>(Xws + r * XS + k * 8) = vh;
      *reinterpret_cast<uint4*>(Xws + X_LO + r * XS + k * 8) = vl;
    }
    // M = (C B^T) o decay mask o step: warp (mt, nh) takes rows 16 mt.., columns 32 nh..
    {
      const int i0 = (warp & 3) * 16, j0 = (warp >> 2) * 32;
      if (j0 <= i0 + 15) {  // blocks wholly above the diagonal are never read
        float acc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll 4
        for (int k0 = 0; k0 < N; k0 += 16) {
          uint32_t a[4];
          ldsm4(a_addr(cs_u, BS, i0, k0, lane), a);
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            uint32_t bb[4];
            ldsm4(b_addr(bs_u, BS, j0 + np * 16, k0, lane), bb);
            mma16816(acc[2 * np], a, bb[0], bb[1]);
            mma16816(acc[2 * np + 1], a, bb[2], bb[3]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int i = i0 + gq + hh * 8, j = j0 + nt * 8 + 2 * cq;
            const float ci = cumS[i];
            const float v0 = (j <= i) ? acc[nt][2 * hh] * __expf(ci - cumS[j]) * sS[j] : 0.f;
            const float v1 = (j + 1 <= i) ? acc[nt][2 * hh + 1] * __expf(ci - cumS[j + 1]) * sS[j + 1] : 0.f;
            __nv_bfloat162 hi, lo;
            split2(v0, v1, hi, lo);
            *reinterpret_cast<__nv_bfloat162*>(Ms + i * MS + j) = hi;
            *reinterpret_cast<__nv_bfloat162*>(Ms + M_LO + i * MS + j) = lo;
          }
      }
    }
    __syncthreads();

    // y = exp(S_i) C_i . h_prev + M x + D x (warp (mt, nh): rows 16 mt.., channels
    // PB / 2 nh..) and h_next = exp(S_last) h_prev + B^T Xw, their k-steps interleaved
    // so that three independent accumulator chains are in flight per warp
    {
      const int i0 = (warp & 3) * 16, p0 = (warp >> 2) * (PB / 2);
      const int mtw = warp & 3;  // the causal product takes k-steps 0..mtw
      float acc[YNT][4], accd[YNT][4];  // C h_prev; M x
#pragma unroll
      for (int nt = 0; nt < YNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = accd[nt][e] = 0.f;
      const float dl = eS[Q - 1];
#pragma unroll
      for (int mt = 0; mt < SMT; ++mt)
#pragma unroll
        for (int nt = 0; nt < SNT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[mt][nt][e] *= dl;
      const uint32_t ss_u = smem_u32(Ss), ms_u = smem_u32(Ms), xw_u = smem_u32(Xws);
      constexpr int KN = N / 16, KQ = Q / 16, KMAX = KN > KQ ? KN : KQ;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const int k0 = k * 16;
        if (k < KN && have_state) {  // C h_prev over states k0..k0+15
          uint32_t a[4];
          ldsm4(a_addr(cs_u, BS, i0, k0, lane), a);
#pragma unroll
          for (int part = 0; part < 2; ++part)  // state hi, lo
#pragma unroll
            for (int np = 0; np < YNT / 2; ++np) {
              uint32_t bb[4];
              ldsm4_t(b_addr_t(ss_u + part * Sm::S_BYTES, XS, p0 + np * 16, k0, lane), bb);
              mma16816(acc[2 * np], a, bb[0], bb[1]);
              mma16816(acc[2 * np + 1], a, bb[2], bb[3]);
            }
        }
        if (k < KQ && k <= mtw) {  // M x over steps k0..k0+15 (causal)
          uint32_t bx[YNT / 2][4];
#pragma unroll
          for (int np = 0; np < YNT / 2; ++np) ldsm4_t(b_addr_t(xs_u, XS, p0 + np * 16, k0, lane), bx[np]);
#pragma unroll
          for (int part = 0; part < 2; ++part) {  // M hi, lo
            uint32_t a[4];
            ldsm4(a_addr(ms_u + part * Sm::M_BYTES, MS, i0, k0, lane), a);
#pragma unroll
            for (int np = 0; np < YNT / 2; ++np) {
              mma16816(accd[2 * np], a, bx[np][0], bx[np][1]);
              mma16816(accd[2 * np + 1], a, bx[np][2], bx[np][3]);
            }
          }
        }
        if (k < KQ) {  // B^T Xw over steps k0..k0+15
          uint32_t a[SMT][4];
#pragma unroll
          for (int mt = 0; mt < SMT; ++mt) ldsm4_t(a_addr_t(bs_u, BS, sm0 + mt * 16, k0, lane), a[mt]);
#pragma unroll
          for (int part = 0; part < 2; ++part)  // Xw hi, lo
#pragma unroll
            for (int np = 0; np < SNT / 2; ++np) {
              uint32_t bb[4];
              ldsm4_t(b_addr_t(xw_u + part * Sm::X_BYTES, XS, sn0 + np * 16, k0, lane), bb);
#pragma unroll
              for (int mt = 0; mt < SMT; ++mt) {
                mma16816(sacc[mt][2 * np], a[mt], bb[0], bb[1]);
                mma16816(sacc[mt][2 * np + 1], a[mt], bb[2], bb[3]);
              }
            }
        }
      }
      const float e0 = eS[i0 + gq], e1 = eS[i0 + gq + 8];
#pragma unroll
      for (int nt = 0; nt < YNT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = i0 + gq + hh * 8, pp = p0 + nt * 8 + 2 * cq;
          const float e = hh ? e1 : e0;
          const float2 xv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Xs + i * XS + pp));
          *reinterpret_cast<float2*>(Ys + i * YS + pp) =
              make_float2(fmaf(Dh, xv.x, fmaf(e, acc[nt][2 * hh], accd[nt][2 * hh])),
                          fmaf(Dh, xv.y, fmaf(e, acc[nt][2 * hh + 1], accd[nt][2 * hh + 1])));
        }
    }
    __syncthreads();  // every read of this stage, of M, Xw and of the state tile is done

    // out = y silu(z), 8 channels per thread and piece (the same pieces this thread
    // copies in, so the stage is read here before this thread refills it)
    for (int i = tid; i < Q * (PB / 8); i += NTHR) {
      const int r = i / (PB / 8), k = i % (PB / 8);
      const int64_t t = t0 + r;
      if (t >= L) continue;
      const int64_t off = (((int64_t)b * L + t) * p.H + h) * P + pc + k * 8;
      const float4 y0 = *reinterpret_cast<const float4*>(Ys + r * YS + k * 8);
      const float4 y1 = *reinterpret_cast<const float4*>(Ys + r * YS + k * 8 + 4);
      float y[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
      if (p.z) {
        const uint4 zv = Sm::Z_SMEM ? *reinterpret_cast<const uint4*>(st + Sm::OFF_Z + (r * XS + k * 8) * 2)
                                    : __ldg(reinterpret_cast<const uint4*>(p.z + off));
        const __nv_bfloat162* zp = reinterpret_cast<const __nv_bfloat162*>(&zv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(zp[e]);
          y[2 * e] *= silu_f(f.x);
          y[2 * e + 1] *= silu_f(f.y);
        }
      }
      uint4 o;
      __nv_bfloat162* op = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) op[e] = __floats2bfloat162_rn(y[2 * e], y[2 * e + 1]);
      *reinterpret_cast<uint4*>(p.out + off) = o;
    }
    if (c + 2 < nch) issue(c + 2);
    cp_async_commit();
    store_state();
    have_state = true;
    if (warp == 0 && c + 1 < nch) {
      make_v(c + 1, dtn);
      load_dt(c + 2, dtn);
    }
  }

  if (p.state) {
#pragma unroll
    for (int mt = 0; mt < SMT; ++mt)
#pragma unroll
      for (int nt = 0; nt < SNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = sm0 + mt * 16 + gq + (e >> 1) * 8, pp = sn0 + nt * 8 + 2 * cq + (e & 1);
          p.state[sbase + (int64_t)(pc + pp) * N + n] = sacc[mt][nt][e];
        }
  }
}

template <int N, int PB>
int launch_ssd(const SsdParams& prm, int64_t batch, cudaStream_t stream) {
  // the dynamic shared-memory limit is raised once per device
  static std::atomic<uint64_t> ready{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(ready.load() & bit)) {
    if (cudaFuncSetAttribute(ssd_fwd_kernel<N, PB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SsdSmem<N, PB>::BYTES) != cudaSuccess)
      return SSM_ERR_CUDA;
    ready.fetch_or(bit);
  }
  ssd_fwd_kernel<N, PB><<<dim3((unsigned)prm.H * (P / PB), (unsigned)batch), NTHR, SsdSmem<N, PB>::BYTES,
                          stream>>>(prm);
  ssm_internal::count_launch();
  return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// ------------------------------------------------ the tcgen05 kernel (ssd_tc.cuh)

std::atomic<int64_t> g_ssd_legacy{0};  // 1: the mma.sync kernel above instead
std::atomic<int64_t> g_ssd_split{0};   // parts per sequence: 0 automatic, else 1, 2 or 4
std::atomic<int64_t> g_ssd_hold{0};    // tests: 1 + unit whose first part never hands over

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A (batch, L, mid, inner) bf16 tensor seen as 5-D: (w values, L rows, inner / w blocks
// of w values, mid, batch).  A box of (w, Q, blocks, 1, 1) lands in shared memory block
// by block, each block Q rows of w values swizzled as the tensor cores read them
// (w = 64 with the 128-byte swizzle, w = 32 with the 64-byte swizzle).
bool encode_tile(CUtensorMap* m, const void* base, int64_t inner, int64_t mid, int64_t L, int64_t batch,
                 int w, int blocks, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn || inner % w) return false;
  const cuuint64_t dims[5] = {(cuuint64_t)w, (cuuint64_t)L, (cuuint64_t)(inner / w), (cuuint64_t)mid,
                              (cuuint64_t)batch};
  const cuuint64_t strides[4] = {(cuuint64_t)(inner * mid * 2), (cuuint64_t)(w * 2), (cuuint64_t)(inner * 2),
                                 (cuuint64_t)(inner * mid * L * 2)};
  const cuuint32_t box[5] = {(cuuint32_t)w, (cuuint32_t)ssd::Q, (cuuint32_t)blocks, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NP, int PB, int N>
int launch_ssd_tc(const SsdParams& prm, int64_t batch, cudaStream_t stream) {
  using Sm = ssd::Smem<NP, PB>;
  static std::atomic<uint64_t> ready{0};
  static std::atomic<int> slots_cache[64];  // resident CTAs per device (0: not yet known)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(ready.load() & bit)) {
    // all of the unified L1 as shared memory: two CTAs of 106 KB per SM at N <= 128
    if (cudaFuncSetAttribute(ssd::ssd_tc_kernel<NP, PB, N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Sm::BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(ssd::ssd_tc_kernel<NP, PB, N>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
      return SSM_ERR_CUDA;
    // CTAs resident per SM, from the kernel's registers (allocated per warp in units of
    // 256), its shared memory (plus the per-block reservation) and its tensor-memory
    // columns (512 per SM).  (The occupancy calculator answers 1 for this kernel at any
    // size, which is not what the SM does: the 4-warp build held two CTAs per SM.)
    cudaFuncAttributes fa;
    int sms = 0, smem_sm = 0, smem_rsv = 0, regs_sm = 0;
    if (cudaFuncGetAttributes(&fa, ssd::ssd_tc_kernel<NP, PB, N>) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess)
      return SSM_ERR_CUDA;
    const int warp_regs = (fa.numRegs * 32 + 255) / 256 * 256;
    int per_sm = std::min(regs_sm / (warp_regs * (ssd::NTHR / 32)), smem_sm / (Sm::BYTES + smem_rsv));
    per_sm = std::min(per_sm, 512 / Sm::TCOLS);
    slots_cache[dev & 63] = std::max(per_sm, 1) * std::max(sms, 1);
    ready.fetch_or(bit);
  }
  const int64_t slots = slots_cache[dev & 63].load();
  ssd::Maps maps;
  std::memset(&maps, 0, sizeof maps);
  if (!encode_tile(&maps.x, prm.x, P, prm.H, prm.L, batch, PB, 1, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode_tile(&maps.B, prm.B, N, prm.G, prm.L, batch, 64, N / 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tile(&maps.C, prm.C, N, prm.G, prm.L, batch, 64, N / 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return SSM_ERR_CUDA;
  ssd::Params p;
  std::memset(&p, 0, sizeof p);
  p.x = prm.x; p.dt = prm.dt; p.z = prm.z; p.A = prm.A; p.D = prm.D; p.dt_bias = prm.dt_bias;
  p.out = prm.out; p.state = prm.state; p.L = prm.L; p.H = prm.H; p.G = prm.G; p.hpg = prm.hpg;
  p.N = N; p.softplus = prm.softplus; p.state_in = prm.state_in; p.batch = (int)batch;
  p.status = ssm_internal::status_word();
  if (!p.status) return SSM_ERR_CUDA;
  // Work: `units` (batch row, head, PB channels) sequences.  When they outnumber the
  // resident CTAs, each is cut into nsplit parts of consecutive chunks taken in order
  // by persistent CTAs, so that the last round is not left mostly empty.  A part costs
  // its chunks plus about two chunk times of pipeline start (measured); nsplit (1, 2 or
  // 4, at most the chunks) minimises rounds x that cost, the smaller on a tie.  Option
  // ssd_split forces it.
  const int64_t units = (int64_t)prm.H * (ssd::P / PB) * batch;
  const int64_t nch = (prm.L + ssd::Q - 1) / ssd::Q;
  if (units * 4 > INT32_MAX) return SSM_ERR_DIMS;
  int nsplit = 1;
  const int64_t forced = g_ssd_split.load();
  if (forced > 0) {
    nsplit = (int)forced;
  } else if (units > slots) {
    auto cost = [&](int64_t n) { return ((n * units + slots - 1) / slots) * ((nch + n - 1) / n + 2); };
    for (int n = 2; n <= 4 && n <= nch; n *= 2)
      if (cost(n) < cost(nsplit)) nsplit = n;
  }
  while (nsplit > 1 && nsplit > nch) nsplit /= 2;
  p.hold_unit = (int)std::min<int64_t>(g_ssd_hold.load(), INT32_MAX) - 1;
  p.units = (int)units;
  p.items = (int)(units * nsplit);
  p.nsplit = nsplit;
  const bool persistent = p.items > slots || nsplit > 1;
  void* ws = nullptr;
  if (persistent) {
    // workspace: the item counter, a flag per (part, unit) and the carries between parts
    const size_t nflag = (size_t)(nsplit - 1) * units;
    const size_t head = ((1 + nflag) * sizeof(int) + 255) / 256 * 256;
    const size_t bytes = head + nflag * PB * N * sizeof(float);
    cudaMemPool_t pool;
    if (ssm_internal::workspace_pool(dev, &pool) != cudaSuccess) return SSM_ERR_CUDA;
    if (cudaMallocFromPoolAsync(&ws, bytes, pool, stream) != cudaSuccess) return SSM_ERR_NOMEM;
    if (cudaMemsetAsync(ws, 0, head, stream) != cudaSuccess) {
      cudaFreeAsync(ws, stream);
      return SSM_ERR_CUDA;
    }
    p.counter = static_cast<int*>(ws);
    p.flags = p.counter + 1;
    p.carry = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + head);
  }
  const int64_t grid = persistent ? std::min<int64_t>(p.items, slots) : p.items;
  ssd::ssd_tc_kernel<NP, PB, N><<<dim3((unsigned)grid), ssd::NTHR, Sm::BYTES, stream>>>(maps, p);
  ssm_internal::count_launch();
  int rc = cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
  if (ws && cudaFreeAsync(ws, stream) != cudaSuccess && rc == SSM_OK) rc = SSM_ERR_CUDA;
  return rc;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

}  // namespace

extern "C" int ssm_ssd_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                           const float* D, const void* z, const float* dt_bias, void* out,
                           float* final_state, const ssm_ssd_dims* dims, cudaStream_t stream) {
  if (!dims) return SSM_ERR_NULL;
  const ssm_ssd_dims d = *dims;
  if (d.batch <= 0 || d.batch > 65535 || d.seqlen < 0 || d.nheads <= 0 || d.nheads > (1 << 29) ||
      d.headdim <= 0 || d.ngroups <= 0 || d.dstate <= 0 || d.nheads % d.ngroups != 0 ||
      (d.io_dtype != SSM_F32 && d.io_dtype != SSM_BF16) || (d.dt_softplus != 0 && d.dt_softplus != 1) ||
      (d.state_in != 0 && d.state_in != 1) || d.reserved != 0)
    return SSM_ERR_DIMS;
  if (d.state_in && !final_state) return SSM_ERR_DIMS;
  if (d.seqlen > 0 && (!x || !dt || !A || !B || !C || !out)) return SSM_ERR_NULL;
  const void* ptrs[] = {x, dt, A, B, C, D, z, dt_bias, out, final_state};
  for (const void* q : ptrs)
    if ((uintptr_t)q % 16) return SSM_ERR_ALIGN;
  if (d.io_dtype != SSM_BF16 || d.headdim != P ||
      (d.dstate != 64 && d.dstate != 128 && d.dstate != 256))
    return SSM_ERR_UNSUPPORTED;

  const size_t act = (size_t)d.batch * d.seqlen * d.nheads * d.headdim * 2;
  const size_t bc = (size_t)d.batch * d.seqlen * d.ngroups * d.dstate * 2;
  const size_t st = (size_t)d.batch * d.nheads * d.headdim * d.dstate * 4;
  const size_t hv = (size_t)d.nheads * 4;
  const struct { const void* p; size_t n; } ins[] = {
      {x, act}, {dt, (size_t)d.batch * d.seqlen * d.nheads * 2}, {A, hv}, {B, bc}, {C, bc},
      {D, hv}, {z, act}, {dt_bias, hv}};
  for (const auto& in : ins) {
    if (overlap(out, act, in.p, in.n)) return SSM_ERR_OVERLAP;
    if (overlap(final_state, st, in.p, in.n)) return SSM_ERR_OVERLAP;
  }
  if (overlap(final_state, st, out, act)) return SSM_ERR_OVERLAP;

  if (d.seqlen == 0) {
    if (final_state && !d.state_in && cudaMemsetAsync(final_state, 0, st, stream) != cudaSuccess)
      return SSM_ERR_CUDA;
    return SSM_OK;
  }

  SsdParams prm;
  memset(&prm, 0, sizeof prm);
  prm.x = static_cast<const __nv_bfloat16*>(x);
  prm.dt = static_cast<const __nv_bfloat16*>(dt);
  prm.B = static_cast<const __nv_bfloat16*>(B);
  prm.C = static_cast<const __nv_bfloat16*>(C);
  prm.z = static_cast<const __nv_bfloat16*>(z);
  prm.A = A;
  prm.D = D;
  prm.dt_bias = dt_bias;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.state = final_state;
  prm.L = d.seqlen;
  prm.H = (int)d.nheads;
  prm.G = (int)d.ngroups;
  prm.hpg = (int)(d.nheads / d.ngroups);
  prm.softplus = d.dt_softplus;
  prm.state_in = d.state_in;
  if (!g_ssd_legacy.load()) {
    switch (d.dstate) {
      case 64: return launch_ssd_tc<128, 32, 64>(prm, d.batch, stream);  // state rows padded to 128
      case 128: return launch_ssd_tc<128, 32, 128>(prm, d.batch, stream);
      default: return launch_ssd_tc<256, 32, 256>(prm, d.batch, stream);
    }
  }
  switch (d.dstate) {
    case 64: return launch_ssd<64, 64>(prm, d.batch, stream);
    case 128: return launch_ssd<128, 64>(prm, d.batch, stream);
    default: return launch_ssd<256, 32>(prm, d.batch, stream);  // half a head per CTA
  }
}

namespace ssm_internal {

bool set_ssd_option(const char* name, int64_t value) {
  if (!std::strcmp(name, "ssd_legacy")) {
    g_ssd_legacy = value ? 1 : 0;
    return true;
  }
  if (!std::strcmp(name, "ssd_hold_part")) {  // failure injection for tests
    if (value < 0) return false;
    g_ssd_hold = value;
    return true;
  }
  if (!std::strcmp(name, "ssd_split")) {  // 0: automatic; 1, 2, 4: parts per sequence
    if (value != 0 && value != 1 && value != 2 && value != 4) return false;
    g_ssd_split = value;
    return true;
  }
  return false;
}

}  // namespace ssm_internal
