// Backward pass of the selective scan with the states rebuilt rather than stored
// (page "State-space models", section "The parallel scan": Mamba's kernel recomputes
// the expanded state in the backward pass).  Reverse-mode differentiation of
//   dt_t = softplus(v_t), v_t = delta_t + bias;  a_t = exp(dt_t A);
//   h_t = a_t h_{t-1} + dt_t B_t x_t;  y_t = C_t . h_t + D x_t;  out_t = y_t silu(z_t)
// with the adjoint state lam_t = C_t gy_t + a_{t+1} lam_{t+1} (gy_t = dout_t silu(z_t)).
//
// Design: one warp per CTA, one lane per channel, all S (= padded N) states of the
// channel in the lane.  The sequence is cut into chunks scanned in parallel; the
// carries in both directions use the associative combine of the per-step maps:
//  * forward: the aggregate pass of the forward kernel (chunk end state from a zero
//    start, chunk step sum S_c) gives h at each chunk start, h <- exp(A S_c) h + H_c;
//  * reverse: bwd_reverse_aggregate gives the adjoint carry of each sub-chunk (rsub
//    per chunk, for more warps) from a zero start at its end,
//    M = sum_s (prod_{r=t0..s} a_r) C_s gy_s, and its step sum S; the carry into a
//    chunk from the right folds the later sub-chunks, mu <- M + exp(A S) mu, from
//    mu = dfinal past the sequence end.
// bwd_main then sweeps its chunk forward once, storing h every SEG steps (HBM
// checkpoints), and walks the segments backwards: it rebuilds the segment's states
// into shared memory and runs the adjoint sweep over them.  Inputs move in tiles of
// SEG steps staged in shared memory, all loads of a tile issued together.  dB, dC
// (summed over channels) leave through a warp reduce-scatter and one atomic add per
// (t, n) per warp; dA, dD and the bias gradient accumulate in registers and are
// added once per lane.
#include <cuda_runtime.h>

#include "bwd_kernel.h"

namespace ssm {

namespace {

constexpr int SEG = 4;  // steps per tile and per rebuilt segment (chunks are multiples of 32)

__device__ __forceinline__ float sigmoidf_(float v) { return 1.f / (1.f + __expf(-v)); }

// Lane i receives the warp sum of v[i] (32 values per lane): recursive halving.
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

// The inputs of SEG steps in shared memory: one column per lane (channel) for the
// per-(step, channel) values, one row per step for B and C (shared by the channels).
// All loads of a tile are issued before any step uses them.
template <int S>
struct Tile {
  float v[SEG][32];  // delta + bias
  float x[SEG][32];
  float g[SEG][32];  // dout
  float z[SEG][32];
  float b[SEG][S];   // zero past N
  float c[SEG][S];
};

// A tile's inputs in flight: issued into registers one tile ahead, stored to shared
// memory when the tile is reached (the loads overlap the previous tile's compute).
template <int S>
struct TileRegs {
  static constexpr int RPL = (SEG * S + 31) / 32;  // B / C row values per lane
  float v[SEG], x[SEG], g[SEG], z[SEG];
  float b[RPL], c[RPL];
};

template <typename IO, int S, bool X, bool G, bool BROW, bool CROW>
__device__ __forceinline__ void fetch_tile(TileRegs<S>& r, const BwdParams& p, int b, int64_t ts, int cnt,
                                           int64_t dd, int lane) {
  const int64_t L = p.seqlen, Dm = p.dim;
#pragma unroll
  for (int k = 0; k < SEG; ++k) {
    if (k < cnt) {
      const int64_t i = ((int64_t)b * L + ts + k) * Dm + dd;
      r.v[k] = IO::load(p.delta, i);
      if (X) r.x[k] = IO::load(p.x, i);
      if (G) {
        r.g[k] = IO::load(p.dout, i);
        if (p.z) r.z[k] = IO::load(p.z, i);
      }
    }
  }
  if (BROW || CROW) {
    const int N = p.dstate;
#pragma unroll
    for (int m = 0; m < TileRegs<S>::RPL; ++m) {
      const int e = lane + 32 * m;
      if (e < cnt * N) {
        const int k = e / N, n = e - k * N;
        const int64_t row = ((int64_t)b * L + ts + k) * N + n;
        if (BROW) r.b[m] = IO::load(p.B, row);
        if (CROW) r.c[m] = IO::load(p.C, row);
      }
    }
  }
}

template <int S, bool X, bool G, bool BROW, bool CROW>
__device__ __forceinline__ void stash_tile(const TileRegs<S>& r, Tile<S>& tl, const BwdParams& p, int cnt,
                                           float biasv, int lane) {
  __syncwarp();  // every lane is done with the previous tile
#pragma unroll
  for (int k = 0; k < SEG; ++k) {
    if (k < cnt) {
      tl.v[k][lane] = r.v[k] + biasv;
      if (X) tl.x[k][lane] = r.x[k];
      if (G) {
        tl.g[k][lane] = r.g[k];
        if (p.z) tl.z[k][lane] = r.z[k];
      }
    }
  }
  if (BROW || CROW) {
    const int N = p.dstate;
#pragma unroll
    for (int m = 0; m < TileRegs<S>::RPL; ++m) {
      const int e = lane + 32 * m;
      if (e < cnt * N) {
        const int k = e / N, n = e - k * N;
        if (BROW) tl.b[k][n] = r.b[m];
        if (CROW) tl.c[k][n] = r.c[m];
      }
    }
  }
  __syncwarp();
}

template <int S>
__device__ __forceinline__ void zero_rows(Tile<S>& tl, int lane) {
  for (int e = lane; e < SEG * S; e += 32) {
    (&tl.b[0][0])[e] = 0.f;
    (&tl.c[0][0])[e] = 0.f;
  }
  __syncwarp();
}

}  // namespace

// Reverse aggregates of the sub-chunks of chunks 1 .. nchunks-1 (rsub per chunk,
// grid.y = sub-chunk index - rsub); a sub-chunk past the sequence end is empty.
template <typename IO, int S>
__global__ void __launch_bounds__(32) bwd_reverse_aggregate(const BwdParams p) {
  __shared__ Tile<S> tl;
  const int lane = threadIdx.x;
  const int64_t L = p.seqlen, Dm = p.dim;
  const int N = p.dstate;
  const int b = blockIdx.z, sub = blockIdx.y + p.rsub;
  const int64_t d = (int64_t)blockIdx.x * 32 + lane;
  const bool valid = d < Dm;
  const int64_t dd = valid ? d : Dm - 1;
  const int64_t t0 = min((int64_t)sub * p.rsub_len, L), t1 = min(t0 + p.rsub_len, L);
  const bool sp = p.delta_softplus != 0;
  float A2[S], m[S];
#pragma unroll
  for (int n = 0; n < S; ++n) {
    A2[n] = n < N ? p.A[dd * N + n] * kLog2e : 0.f;
    m[n] = 0.f;
  }
  const float biasv = p.bias ? p.bias[dd] : 0.f;
  zero_rows(tl, lane);
  float Ssum = 0.f, Scomp = 0.f;
  const int ntile = (int)((t1 - t0 + SEG - 1) / SEG);
  auto tile_at = [&](int j, int64_t& ts, int& cnt) {
    ts = t0 + (int64_t)j * SEG;
    cnt = (int)min((int64_t)SEG, t1 - ts);
  };
  TileRegs<S> rg;
  {
    int64_t ts;
    int cnt;
    tile_at(ntile - 1, ts, cnt);
    fetch_tile<IO, S, false, true, false, true>(rg, p, b, ts, cnt, dd, lane);
  }
  for (int j = ntile - 1; j >= 0; --j) {
    int64_t ts;
    int cnt;
    tile_at(j, ts, cnt);
    stash_tile<S, false, true, false, true>(rg, tl, p, cnt, biasv, lane);
    if (j > 0) {  // the next tile's loads overlap this tile's steps
      int64_t tn;
      int cn;
      tile_at(j - 1, tn, cn);
      fetch_tile<IO, S, false, true, false, true>(rg, p, b, tn, cn, dd, lane);
    }
    float tsum = 0.f;
    for (int k = cnt - 1; k >= 0; --k) {
      const float v = tl.v[k][lane];
      const float dt = sp ? softplus<std::is_same<IO, F32>::value>(v) : v;
      const float g = tl.g[k][lane];
      const float gy = p.z ? g * silu(tl.z[k][lane]) : g;
      const float2 dt2 = make_float2(dt, dt), gy2 = make_float2(gy, gy);
#pragma unroll
      for (int i = 0; i < S / 2; ++i) {
        const float2 e = __fmul2_rn(dt2, make_float2(A2[2 * i], A2[2 * i + 1]));
        const float2 c2 = *reinterpret_cast<const float2*>(&tl.c[k][2 * i]);
        const float2 mm = __fmul2_rn(make_float2(ex2(e.x), ex2(e.y)),
                                     __ffma2_rn(c2, gy2, make_float2(m[2 * i], m[2 * i + 1])));
        m[2 * i] = mm.x;
        m[2 * i + 1] = mm.y;
      }
      tsum += dt;
    }
    kahan_add(Ssum, Scomp, tsum);
  }
  if (!valid) return;
  const int64_t ci = ((int64_t)(sub - p.rsub) * p.batch + b) * Dm + d;
#pragma unroll
  for (int n = 0; n < S; ++n)
    if (n < N) p.ws_M[ci * N + n] = m[n];
  p.ws_S2[ci] = Ssum - Scomp;
}

template <typename IO, int S>
__global__ void __launch_bounds__(32, 16) bwd_main(const BwdParams p) {
  __shared__ float2 hist[SEG + 1][S / 2][32];  // state pairs; row 0: state before the segment
  __shared__ float dts[SEG][32];
  __shared__ Tile<S> tl;
  const int lane = threadIdx.x;
  const int64_t L = p.seqlen, Dm = p.dim;
  const int N = p.dstate;
  const int b = blockIdx.z, chunk = blockIdx.y;
  const int64_t d = (int64_t)blockIdx.x * 32 + lane;
  const bool valid = d < Dm;
  const int64_t dd = valid ? d : Dm - 1;
  const int64_t t0 = (int64_t)chunk * p.chunk_len, t1 = min(t0 + p.chunk_len, L);
  const bool sp = p.delta_softplus != 0;

  float A2[S];
#pragma unroll
  for (int n = 0; n < S; ++n) A2[n] = n < N ? p.A[dd * N + n] * kLog2e : 0.f;
  float2 A2p[S / 2];  // the same, as state pairs for the f32x2 operations
#pragma unroll
  for (int i = 0; i < S / 2; ++i) A2p[i] = make_float2(A2[2 * i], A2[2 * i + 1]);
  const float biasv = p.bias ? p.bias[dd] : 0.f;
  const float Dv = p.Dskip ? p.Dskip[dd] : 0.f;
  const float vm = valid ? 1.f : 0.f;  // absent channels add nothing to dB, dC
  const int64_t sidx = ((int64_t)b * Dm + dd) * N;
  zero_rows(tl, lane);

  // ---- state at the chunk start (forward carry)
  float h[S];
#pragma unroll
  for (int n = 0; n < S; ++n) h[n] = (chunk == 0 && p.h_init && n < N) ? p.h_init[sidx + n] : 0.f;
  for (int cc = 0; cc < chunk; ++cc) {
    const int64_t ci = ((int64_t)cc * p.batch + b) * Dm + dd;
    const float Sc = p.ws_S[ci];
#pragma unroll
    for (int n = 0; n < S; ++n)
      if (n < N) h[n] = fmaf(ex2(Sc * A2[n]), h[n], p.ws_H[ci * N + n]);
  }
  // ---- adjoint carry into the chunk from the right: kap = a_{t1} lam_{t1}
  float kap[S];
#pragma unroll
  for (int n = 0; n < S; ++n) kap[n] = (p.dfinal && n < N) ? p.dfinal[sidx + n] : 0.f;
  for (int sc = p.nchunks * p.rsub - 1; sc >= (chunk + 1) * p.rsub; --sc) {
    const int64_t ci = ((int64_t)(sc - p.rsub) * p.batch + b) * Dm + dd;
    const float Sc = p.ws_S2[ci];
#pragma unroll
    for (int n = 0; n < S; ++n)
      if (n < N) kap[n] = fmaf(ex2(Sc * A2[n]), kap[n], p.ws_M[ci * N + n]);
  }

  // ---- forward sweep: a checkpoint at every segment start
  const int nseg = (int)((t1 - t0 + SEG - 1) / SEG);
  const int64_t seg0 = t0 / SEG;
  auto seg_at = [&](int j, int64_t& ts, int& cnt) {
    ts = t0 + (int64_t)j * SEG;
    cnt = (int)min((int64_t)SEG, t1 - ts);
  };
  TileRegs<S> rg;
  {
    int64_t ts;
    int cnt;
    seg_at(0, ts, cnt);
    fetch_tile<IO, S, true, false, true, false>(rg, p, b, ts, cnt, dd, lane);
  }
  for (int j = 0; j < nseg; ++j) {
    int64_t ts;
    int cnt;
    seg_at(j, ts, cnt);
    if (valid) {
      float* ck = p.ws_ck + (((seg0 + j) * p.batch + b) * Dm + d) * S;
#pragma unroll
      for (int n = 0; n < S; ++n) ck[n] = h[n];
    }
    stash_tile<S, true, false, true, false>(rg, tl, p, cnt, biasv, lane);
    if (j + 1 < nseg) {
      int64_t tn;
      int cn;
      seg_at(j + 1, tn, cn);
      fetch_tile<IO, S, true, false, true, false>(rg, p, b, tn, cn, dd, lane);
    } else {  // the reverse walk starts with the last segment
      fetch_tile<IO, S, true, true, true, true>(rg, p, b, ts, cnt, dd, lane);
    }
    for (int k = 0; k < cnt; ++k) {
      const float v = tl.v[k][lane];
      const float dt = sp ? softplus<std::is_same<IO, F32>::value>(v) : v;
      const float u = dt * tl.x[k][lane];
      const float2 dt2 = make_float2(dt, dt), u2 = make_float2(u, u);
#pragma unroll
      for (int i = 0; i < S / 2; ++i) {
        const float2 e = __fmul2_rn(dt2, A2p[i]);
        const float2 bb = __fmul2_rn(u2, *reinterpret_cast<const float2*>(&tl.b[k][2 * i]));
        const float2 hh = __ffma2_rn(make_float2(ex2(e.x), ex2(e.y)), make_float2(h[2 * i], h[2 * i + 1]), bb);
        h[2 * i] = hh.x;
        h[2 * i + 1] = hh.y;
      }
    }
  }

  // ---- segments in reverse: rebuild the states, then the adjoint sweep
  float2 gA2[S / 2], kap2[S / 2];
#pragma unroll
  for (int i = 0; i < S / 2; ++i) {
    gA2[i] = make_float2(0.f, 0.f);
    kap2[i] = make_float2(kap[2 * i], kap[2 * i + 1]);
  }
  float gD = 0.f, gbias = 0.f;
  for (int j = nseg - 1; j >= 0; --j) {
    int64_t ts;
    int cnt;
    seg_at(j, ts, cnt);
    float2 h2[S / 2];
    {
      const float* ck = p.ws_ck + (((seg0 + j) * p.batch + b) * Dm + dd) * S;
#pragma unroll
      for (int i = 0; i < S / 2; ++i)
        h2[i] = valid ? make_float2(ck[2 * i], ck[2 * i + 1]) : make_float2(0.f, 0.f);
    }
    stash_tile<S, true, true, true, true>(rg, tl, p, cnt, biasv, lane);
    if (j > 0) {
      int64_t tn;
      int cn;
      seg_at(j - 1, tn, cn);
      fetch_tile<IO, S, true, true, true, true>(rg, p, b, tn, cn, dd, lane);
    }
#pragma unroll
    for (int i = 0; i < S / 2; ++i) hist[0][i][lane] = h2[i];
    for (int k = 0; k < cnt; ++k) {
      const float v = tl.v[k][lane];
      const float dt = sp ? softplus<std::is_same<IO, F32>::value>(v) : v;
      dts[k][lane] = dt;
      const float u = dt * tl.x[k][lane];
      const float2 dt2 = make_float2(dt, dt), u2 = make_float2(u, u);
#pragma unroll
      for (int i = 0; i < S / 2; ++i) {
        const float2 e = __fmul2_rn(dt2, A2p[i]);
        const float2 bb = __fmul2_rn(u2, *reinterpret_cast<const float2*>(&tl.b[k][2 * i]));
        h2[i] = __ffma2_rn(make_float2(ex2(e.x), ex2(e.y)), h2[i], bb);
        hist[k + 1][i][lane] = h2[i];
      }
    }
    for (int k = cnt - 1; k >= 0; --k) {
      const int64_t t = ts + k;
      const int64_t i0 = ((int64_t)b * L + t) * Dm + dd;
      const float dt = dts[k][lane], v = tl.v[k][lane];
      const float xv = tl.x[k][lane], g = tl.g[k][lane];
      float zv = 0.f, sz = 1.f;
      if (p.z) {
        zv = tl.z[k][lane];
        sz = sigmoidf_(zv);
      }
      const float gy = p.z ? g * zv * sz : g;
      const float2 dt2 = make_float2(dt, dt), gy2 = make_float2(gy, gy);
      const float2 dtx2 = make_float2(dt * xv * vm, dt * xv * vm), gyv2 = make_float2(gy * vm, gy * vm);
      float2 sA = make_float2(0.f, 0.f), sB = make_float2(0.f, 0.f), y2 = make_float2(0.f, 0.f);
      float red[32];
#pragma unroll
      for (int i = 0; i < S / 2; ++i) {
        const float2 e = __fmul2_rn(dt2, A2p[i]);
        const float2 a = make_float2(ex2(e.x), ex2(e.y));
        const float2 hp = hist[k][i][lane], hc = hist[k + 1][i][lane];
        const float2 bn = *reinterpret_cast<const float2*>(&tl.b[k][2 * i]);
        const float2 cn = *reinterpret_cast<const float2*>(&tl.c[k][2 * i]);
        const float2 lam = __ffma2_rn(cn, gy2, kap2[i]);
        const float2 ga = __fmul2_rn(__fmul2_rn(lam, hp), a);  // gradient of a_t, times a_t
        gA2[i] = __ffma2_rn(ga, dt2, gA2[i]);
        sA = __ffma2_rn(ga, A2p[i], sA);   // sum of ga A log2(e)
        sB = __ffma2_rn(lam, bn, sB);      // sum of lam B
        y2 = __ffma2_rn(cn, hc, y2);
        const float2 tb = __fmul2_rn(lam, dtx2), tc = __fmul2_rn(gyv2, hc);
        red[2 * i] = tb.x;                 // this channel's shares of dB
        red[2 * i + 1] = tb.y;
        red[16 + 2 * i] = tc.x;            // and of dC
        red[16 + 2 * i + 1] = tc.y;
        kap2[i] = __fmul2_rn(a, lam);
      }
#pragma unroll
      for (int n = S; n < 16; ++n) red[n] = red[16 + n] = 0.f;
      const float lamB = sB.x + sB.y;
      const float gx = fmaf(gy, Dv, lamB * dt);
      const float y = fmaf(Dv, xv, y2.x + y2.y);
      const float ddt = fmaf(sA.x + sA.y, kLn2, lamB * xv);
      const float dv = sp ? ddt * sigmoidf_(v) : ddt;
      gbias += dv;
      gD = fmaf(gy, xv, gD);
      if (valid) {
        IO::store(p.dx, i0, gx);
        IO::store(p.ddelta, i0, dv);
        if (p.z) IO::store(p.dz, i0, g * y * sz * fmaf(zv, 1.f - sz, 1.f));
      }
      const float tot = reduce_scatter32(red, lane);
      const int n = lane & 15;
      if (n < N) atomicAdd((lane < 16 ? p.dB : p.dC) + ((int64_t)b * L + t) * N + n, tot);
    }
  }
#pragma unroll
  for (int i = 0; i < S / 2; ++i) {
    kap[2 * i] = kap2[i].x;
    kap[2 * i + 1] = kap2[i].y;
  }
  float gA[S];
#pragma unroll
  for (int i = 0; i < S / 2; ++i) {
    gA[2 * i] = gA2[i].x;
    gA[2 * i + 1] = gA2[i].y;
  }
  if (!valid) return;
  // kap = a_{t0} lam_{t0}: the gradient of the state before the chunk
  if (chunk == 0 && p.dh_init)
#pragma unroll
    for (int n = 0; n < S; ++n)
      if (n < N) p.dh_init[sidx + n] = kap[n];
#pragma unroll
  for (int n = 0; n < S; ++n)
    if (n < N) atomicAdd(p.dA + dd * N + n, gA[n]);
  if (p.dD) atomicAdd(p.dD + dd, gD);
  if (p.dbias) atomicAdd(p.dbias + dd, gbias);
}

template <typename IO, int S>
BwdKernels bwd_kernels() {
  BwdKernels k;
  k.reverse_aggregate = bwd_reverse_aggregate<IO, S>;
  k.main = bwd_main<IO, S>;
  k.seg = SEG;
  return k;
}

BwdKernels lookup_bwd(int io_bf16, int S) {
  switch (S) {
    case 2: return io_bf16 ? bwd_kernels<BF16, 2>() : bwd_kernels<F32, 2>();
    case 4: return io_bf16 ? bwd_kernels<BF16, 4>() : bwd_kernels<F32, 4>();
    case 8: return io_bf16 ? bwd_kernels<BF16, 8>() : bwd_kernels<F32, 8>();
    case 16: return io_bf16 ? bwd_kernels<BF16, 16>() : bwd_kernels<F32, 16>();
    default: return BwdKernels();
  }
}

}  // namespace ssm
