// Mamba-2 SSD layer, forward, on the 5th-generation tensor cores (tcgen05, TMEM).
//
// Pages: "State-space models", section "The parallel scan" (A a scalar times the
// identity per head turns the scan into blocks of matrix products on the tensor
// cores); "Structured State Space Models and Mamba", section "State Space Duality and
// Mamba-2" (Y = (L o (C B^T)) V with a 1-semiseparable decay mask L).
//
// A CTA (eight warps, 256 threads) takes one (batch row, head, block of PB channels) --
// a unit -- or one part of a unit's sequence, and walks it in chunks of Q = 128 steps,
// the (N, PB) state of its channels carried in tensor memory.  When the units outnumber
// the resident CTAs, CTAs persist and take the parts (consecutive chunks) in order from
// a counter: part s of a unit waits for the release flag of part s - 1 and starts from
// the state it left (fp32) in a workspace; taking items in order means the part waited
// for is held by a CTA already running, which never waits on a later item.  The state
// between parts is the sum of its two accumulators, the value every chunk start forms
// anyway, so the result does not depend on the number of parts.  With S_i the running
// sum of step * A inside a chunk:
//   G        = C B^T                                          (Q x Q over N)
//   M[i][j]  = G[i][j] exp(S_i - S_j) step_j   for j <= i, else 0
//   Yd       = M X                                            (Q x PB over Q)
//   Yo       = C h_prev                                       (Q x PB over N)
//   y_i      = Yd_i + exp(S_i) Yo_i + D x_i;   out = y silu(z)
//   h_next   = exp(S_last) h_prev + B^T Xw,   Xw_j = exp(S_last - S_j) step_j x_j
// The four products are tcgen05.mma (kind::f16: bf16 operands, fp32 accumulators in
// TMEM), each accumulator chain issued by one thread (C h_prev and B^T Xw, and the two
// parts of M X, by two threads side by side) and completed on mbarriers.  C, B and x
// arrive by one TMA tensor copy each per chunk, as rows of 128 (C, B) and 64 (x) bytes
// with the hardware swizzle, and enter the products through swizzled shared-memory
// descriptors; Xw and the state copy are written by the threads in the no-swizzle
// core-matrix layout (8 rows x 16 bytes per core matrix).  M never leaves tensor memory:
// each thread reads its row of G, forms its row of M and writes it back over G as the A
// operand of M X.  Threads i and i + 128 own TMEM lane i (row i of every accumulator)
// for the element-wise work, each with half of the columns (of M: alternate blocks).  The state copy and Xw, held as pairs of bf16 parts, enter their
// products as one operand twice as wide (the parts side by side), so that one
// instruction forms both partial products into adjacent accumulator columns; the carried
// state is held as two accumulators (the sum so far, this chunk's low parts).  The two
// parts of M enter as two products (M_hi X onto exp(S_i) C h_prev, M_lo X beside it),
// summed when the outputs are formed.
//
// Order inside a chunk (its G already issued): the threads form Xw, then C h_prev and
// B^T Xw are issued; M is formed once G is done, the scaled C h_prev written as the
// start of M X once those two are done, and M X is issued last.  Then the next chunk's
// copies are issued; while they land the threads form its per-step vectors and state
// copy (neither needs its inputs); then its G is issued, and runs while the threads
// form this chunk's outputs.  The decay factor of M is split as
//   exp(S_i - S_j) = exp(S_i - S_ref) exp(S_ref - S_j),  S_ref = the midpoint of the
// chunk's range of S, so that M costs two multiplies per element; a chunk whose range
// of S is too wide for both factors to stay inside fp32 takes one exponential per
// element instead.  The column blocks right of a warp's diagonal block are zero and
// written as zeros, not formed.
//
// Precision: the operands formed in fp32 enter as a pair of bf16 values (value and
// remainder, about 16 significant bits): M (one bf16 rounding of it alone reached
// 1.7e-2 of floored error on a Gaussian layer), Xw and the state copy (the state
// accumulates over the whole sequence).  Step sizes, decays and the state stay in
// fp32.  Every wait is bounded (2 s); a wait that runs out sets the status word and
// the CTA waits (bounded) for its products in flight, frees its tensor memory and
// leaves.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace ssd {

constexpr int Q = 128;      // steps per chunk (the M dimension of every product)
constexpr int P = 64;       // channels per head
constexpr int NTHR = 256;   // threads per CTA: two per TMEM lane (each with half the columns)
constexpr uint64_t kWaitNs = 2000000000ull;

// 5-D tensor maps (w values, L rows, blocks of w values, head or group, batch row): one
// box of (w, Q, blocks, 1, 1) is a chunk's tile, block by block, each block Q swizzled
// rows of w values (C, B: w = 64, 128-byte swizzle; x: w = PB = 32, 64-byte swizzle).
struct Maps {
  CUtensorMap x;   // box (32, Q, 1, 1, 1)
  CUtensorMap B;   // box (64, Q, N / 64, 1, 1)
  CUtensorMap C;
};

struct Params {
  const __nv_bfloat16* x;
  const __nv_bfloat16* dt;
  const __nv_bfloat16* z;
  const float* A;
  const float* D;
  const float* dt_bias;
  __nv_bfloat16* out;
  float* state;       // (batch, H, P, N) or null
  int* status;
  // work items: each (batch row, head, block of PB channels) -- a unit -- walks its
  // sequence in nsplit parts of consecutive chunks; item k is part k / units of unit
  // k % units.  With counter set, CTAs take items in order from it (a part s > 0 waits
  // for flags[(s - 1) units + u] and starts from the state part s - 1 left in carry
  // [(s - 1) units + u][PB][N]); without it CTA k runs item k alone (nsplit 1).
  int* counter;
  int* flags;
  float* carry;
  int units, items, nsplit;
  int hold_unit;  // failure injection for tests: part 0 of this unit never releases (-1: none)
  int64_t L;
  int batch, H, G, hpg, N;
  int softplus, state_in;
};

// Shared-memory plan of one CTA: NP = N padded to a multiple of 128 (the state rows
// of one product), PB channels.
template <int NP, int PB>
struct Smem {
  static constexpr int C_OFF = 0;                        // C tile  [Q x NP] bf16
  static constexpr int B_OFF = C_OFF + Q * NP * 2;       // B tile  [Q x NP]
  static constexpr int X_OFF = B_OFF + Q * NP * 2;       // x tile  [Q x PB]
  static constexpr int W_OFF = X_OFF + Q * PB * 2;       // Xw hi, lo [Q x PB] each
  static constexpr int H_OFF = W_OFF + 2 * Q * PB * 2;   // state hi, lo [NP x PB] each
  static constexpr int V_OFF = H_OFF + 2 * NP * PB * 2;  // S, step, b (Q floats each), reductions, item
  static constexpr int BAR_OFF = V_OFF + 3 * Q * 4 + 64;
  static constexpr int BYTES = BAR_OFF + 64;
  // TMEM columns: G, then M (hi, lo: two bf16 per column) in its place; C h_hi | C h_lo,
  // then the two M X accumulators in their place; per 128 state rows the state's two
  // accumulators (sum so far | low parts)
  static constexpr int T_G = 0, T_YO = Q, T_H = Q + 2 * PB;
  static constexpr int TUSED = T_H + (NP / 128) * 2 * PB;
  static constexpr int TCOLS = TUSED <= 256 ? 256 : 512;
  static_assert(TUSED <= 512, "tensor memory columns");
  static_assert(BYTES <= 227 * 1024, "shared memory of one CTA");
  static_assert(PB == 32, "x arrives as 64-byte swizzled rows of 32 channels");
  static_assert(B_OFF % 1024 == 0 && X_OFF % 1024 == 0, "swizzled tiles on 1024-byte boundaries");
};

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t par) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(par)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase: false if it did not complete within kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t par) {
  if (mbar_try(bar, par)) return true;
  const uint64_t t0 = gtimer();
  for (long long i = 0; i < (1ll << 30); ++i) {
    if (mbar_try(bar, par)) return true;
    if (gtimer() - t0 > kWaitNs) return false;
  }
  return false;
}

// Shared-memory matrix descriptor: start address, leading-dimension byte offset,
// stride-dimension byte offset, the fixed version bits and the layout (0: no swizzle,
// core matrices of 8 rows x 16 bytes; kSw128 / kSw64: rows of 128 / 64 bytes with their
// 16-byte pieces permuted within groups of 8 rows, as TMA writes them).  No swizzle:
// LBO between core matrices along K, SBO between core matrices along M or N.  Swizzled
// K-major: SBO between groups of 8 rows (LBO unused); swizzled MN-major: LBO between
// blocks of 64 (128 B) or 32 (64 B) M/N values, SBO between groups of 8 K rows.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout = 0) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}
// layout field of a shared-memory descriptor
constexpr uint32_t kSw128 = 2, kSw64 = 4;
constexpr int kAtom = Q * 128;  // one 128-byte-swizzled block: Q rows of 64 bf16 values

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, M x N, K-major (0) or
// MN-major (1) A and B.
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t id, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(id), "r"((uint32_t)acc)
      : "memory");
}

// The same with A (M x 16, K-major) in tensor memory: row m in lane m, two bf16 values
// of K per column (the lower K in the low half), the 8 columns of a K step from tmem_a.
__device__ __forceinline__ void mma_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t db, uint32_t id, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(db), "r"(id), "r"((uint32_t)acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's lane; the load's wait is the caller's
// (tmem_wait_ld on each destination) so that several loads are in flight together.
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Wait for this thread's tensor-memory loads; the registers of r pass through the
// statement so that no use of them is scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                 "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                 "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane, waited for.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld32_nw(taddr, r);
  tmem_wait_ld(r);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// 16 consecutive fp32 columns of this thread's lane, waited for (the wait names the
// destinations, so that no use of them is scheduled before it).
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
        "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15])
      : "r"(ta));
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
        "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
      : "r"(tb));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                 "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                 "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
                 "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                 "+r"(b[14]), "+r"(b[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  uint32_t r[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(v[j]);
  tmem_st32u(taddr, r);
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            int c4, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
      : "memory");
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// v = hi + lo with both parts bf16 (lo holds what hi rounds away)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte offset of row r, column block cb (8 columns) in a no-swizzle core-matrix tile of
// R rows whose column blocks are stored one after another (block cb at cb * R * 16).
__device__ __forceinline__ uint32_t cm(int r, int cb, int R) { return (uint32_t)(cb * R + r) * 16u; }

// NN = N (a compile-time state size: the product loops unroll with constant descriptors)
template <int NP, int PB, int NN>
__global__ void __maxnreg__((Smem<NP, PB>::BYTES <= 110 * 1024 && Smem<NP, PB>::TCOLS <= 256) ? 120 : 255)
    ssd_tc_kernel(const __grid_constant__ Maps maps, const Params p) {
  static_assert(NN % 64 == 0 && NN <= NP, "state size: a multiple of 64, at most the padded rows");
  using Sm = Smem<NP, PB>;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // warps w and w + 4 share lane quarter qw (TMEM lanes 32 qw ..): each takes half of the
  // columns of every element-wise phase (channels HP hf .. HP hf + HP - 1)
  const int qw = warp & 3, hf = warp >> 2;
  constexpr int HP = PB / 2;
  // the item in hand: batch row b, head h, first channel pc, group g (set per item)
  int b = 0, h = 0, pc = 0, g = 0;
  float Ah = 0.f, Dh = 0.f, biash = 0.f;
  const int64_t L = p.L;
  const int nch = (int)((L + Q - 1) / Q);
  constexpr int N = NN, kN = NN / 16;  // K steps over the state dimension
  float* Sv = reinterpret_cast<float*>(smem + Sm::V_OFF);  // S_i of the chunk
  float* stepv = Sv + Q;                                  // step_i
  float* bv = stepv + Q;                                  // exp(S_ref - S_j) step_j
  float* red = bv + Q;                                    // per-warp sums, minima, maxima
  int* item_s = reinterpret_cast<int*>(red + 12);         // the item taken by thread 0
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::BAR_OFF);
  uint32_t* tbase_s = reinterpret_cast<uint32_t*>(bars + 4);
  const uint32_t bar_in = su32(&bars[0]), bar_g = su32(&bars[1]), bar_s = su32(&bars[2]),
                 bar_y = su32(&bars[3]);
  const uint32_t s_base = su32(smem);

  // zero the tiles once (the rows of B past N feed state rows that are never read)
  for (int i = tid; i < Sm::V_OFF / 16; i += NTHR) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {  // C h_prev and B^T Xw, and the two parts of M X, are issued by two threads
    const uint32_t cnt[4] = {1, 1, 2, 2};
    for (int i = 0; i < 4; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(&bars[i])), "r"(cnt[i]) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tbase_s)),
                 "r"(Sm::TCOLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tbase_s;
  const uint32_t lane_t = tmem + ((uint32_t)(qw * 32) << 16);  // this warp's lanes
  bool ok = true;
  int issued = 0;  // products issued and not yet waited for: bit 0 G, 1 C h / B^T Xw, 2 M X
  uint32_t gc = 0;  // chunks this CTA has begun: each takes one phase of every barrier

  // the inputs of chunk c: C, B (Q x N) and x (Q x PB), one tensor copy each, landing in
  // barrier phase par
  const uint32_t in_bytes = (uint32_t)((2 * (N / 8) + PB / 8) * Q * 16);
  bool in_flight = false;  // a tensor copy into the tiles has been issued and not waited for
  uint32_t in_par = 0;     // ... in this phase of bar_in
  auto load_chunk = [&](int c, uint32_t par) {
    in_flight = true;
    in_par = par;
    if (tid != 0) return;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_in), "r"(in_bytes)
                 : "memory");
    const int t0 = c * Q;
    tma_load_5d(s_base + Sm::C_OFF, &maps.C, 0, t0, 0, g, b, bar_in);
    tma_load_5d(s_base + Sm::B_OFF, &maps.B, 0, t0, 0, g, b, bar_in);
    tma_load_5d(s_base + Sm::X_OFF, &maps.x, 0, t0, pc / PB, h, b, bar_in);
  };

  constexpr uint32_t ID_G = idesc(Q, Q, 0, 0);          // C (K-major) x B^T (K-major)
  constexpr uint32_t ID_Y = idesc(Q, PB, 0, 1);         // M (TMEM) x X (MN-major)
  constexpr uint32_t ID_O = idesc(Q, 2 * PB, 0, 1);     // C (K-major) x [h_hi | h_lo] (MN-major)
  constexpr uint32_t ID_S = idesc(128, 2 * PB, 1, 1);   // B^T (MN-major) x [Xw_hi | Xw_lo] (MN-major)
  // operand descriptors at offset 0; a K step adds its byte offset / 16
  // C, B, x arrive 128- (C, B) and 64-byte (x) swizzled; Xw and the state copy are
  // written by the threads without swizzle
  const uint64_t dC = sdesc(s_base + Sm::C_OFF, 16, 1024, kSw128);      // K-major, K = n
  const uint64_t dB = sdesc(s_base + Sm::B_OFF, 16, 1024, kSw128);      // K-major, K = n
  const uint64_t dBt = sdesc(s_base + Sm::B_OFF, kAtom, 1024, kSw128);  // MN-major: M = n, K = j
  const uint64_t dX = sdesc(s_base + Sm::X_OFF, 4096, 512, kSw64);      // MN-major: N = channel, K = j
  const uint64_t dH = sdesc(s_base + Sm::H_OFF, 128, NP * 16);          // MN-major: N = channel, K = n
  const uint64_t dW = sdesc(s_base + Sm::W_OFF, 128, Q * 16);           // MN-major: N = channel, K = j
  // a K step (16 values) of the swizzled K-major tiles: 32 bytes inside a block of 64
  auto kmaj = [](int k) { return (uint32_t)((k >> 2) * kAtom + (k & 3) * 32); };
  auto off16 = [](uint32_t bytes) { return (uint64_t)(bytes >> 4); };

  const int i = qw * 32 + lane;  // this thread's row of every Q-row product, and its state row
  float dt_next = 0.f;           // the raw step of this thread's row, one chunk ahead

  // ---- per-step vectors of chunk c: step_i, the running sum S_i of step * A (block
  // scan), the chunk's range of S and the split decay factors (smem: Sv, stepv, bv)
  float step = 0.f, Si = 0.f, Slast = 0.f, ai = 0.f;
  bool split = true;
  auto scan = [&](int c) {
    const int64_t t0 = (int64_t)c * Q;
    const float dt_raw = dt_next;
    dt_next = (t0 + Q + i < L) ? __bfloat162float(p.dt[((int64_t)b * L + t0 + Q + i) * p.H + h]) : 0.f;
    step = 0.f;
    if (t0 + i < L) {
      const float v = dt_raw + biash;
      step = p.softplus ? (v > 20.f ? v : log1pf(expf(v))) : v;
    }
    float incl = step * Ah;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    __syncthreads();  // the previous chunk's readers of Sv, stepv, bv and red are done
    if (hf == 0 && lane == 31) red[qw] = incl;  // both warps of a quarter hold the same sums
    __syncthreads();
    for (int w = 0; w < qw; ++w) incl += red[w];
    Si = incl;
    float mn = Si, mx = Si;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    if (hf == 0 && lane == 0) {
      red[4 + qw] = mn;
      red[8 + qw] = mx;
    }
    if (hf == 0) {
      Sv[i] = Si;
      stepv[i] = step;
    }
    __syncthreads();
    mn = fminf(fminf(red[4], red[5]), fminf(red[6], red[7]));
    mx = fmaxf(fmaxf(red[8], red[9]), fmaxf(red[10], red[11]));
    Slast = Sv[Q - 1];
    // both factors within e^(+-80) (inside fp32) when the range of S is at most 160
    split = (mx - mn) <= 160.f;
    const float Sref = 0.5f * (mn + mx);
    ai = ex2f((Si - Sref) * kLog2e);
    if (hf == 0) bv[i] = ex2f((Sref - Si) * kLog2e) * step;
  };
  // ---- the state entering a chunk (sum of its two accumulators): its bf16 copy (hi, lo)
  // for C h_prev, then h <- exp(S_last) h into the first accumulator, zeros into the
  // second.  Needs no input of the chunk, so it runs while the chunk's copies land.
  auto state_copy = [&]() {
    const float dl = ex2f(Slast * kLog2e);
#pragma unroll 1
    for (int nb = 0; nb < NP / 128; ++nb) {
      const int n = nb * 128 + i;
      const int c0 = hf * HP;
      const uint32_t ta = lane_t + Sm::T_H + nb * 2 * PB + c0;
      uint32_t ra[HP], rb[HP];
      tmem_ld16x2(ta, ta + PB, ra, rb);
      float v[HP];
#pragma unroll
      for (int j = 0; j < HP; ++j) v[j] = __uint_as_float(ra[j]) + __uint_as_float(rb[j]);
#pragma unroll
      for (int cb = 0; cb < HP / 8; ++cb) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split2(v[cb * 8 + 2 * e], v[cb * 8 + 2 * e + 1], hi[e], lo[e]);
        const uint32_t off = cm(n, (c0 >> 3) + cb, NP);
        *reinterpret_cast<uint4*>(smem + Sm::H_OFF + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(smem + Sm::H_OFF + NP * PB * 2 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
#pragma unroll
      for (int j = 0; j < HP; ++j) {
        ra[j] = __float_as_uint(v[j] * dl);
        rb[j] = 0u;
      }
      tmem_st16u(ta, ra);
      tmem_st16u(ta + PB, rb);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  };

  uint32_t cur = 0;  // phase parity of the chunk whose products are in hand
  // ---- a chunk's inputs (barrier phase par), then G = C B^T into the columns of G (free
  // once the previous chunk's M X is done).  Every wait is decided by all threads
  // together, so that they leave the loop at the same point; false: the wait ran out.
  auto start_g = [&](uint32_t par) -> bool {
    cur = par;
    if (!__syncthreads_and(mbar_wait(bar_in, par))) return false;
    in_flight = false;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < kN; ++k)
        mma(tmem + Sm::T_G, dC + off16(kmaj(k)), dB + off16(kmaj(k)), ID_G, k > 0);
      mma_commit(bar_g);
    }
    issued |= 1;
    return true;
  };

  bool first = true;
#pragma unroll 1
  for (;;) {
    // ---- the next item
    __syncthreads();  // every thread has read the previous item
    if (tid == 0) *item_s = p.counter ? atomicAdd(p.counter, 1) : (first ? (int)blockIdx.x : p.items);
    __syncthreads();
    const int k = *item_s;
    first = false;
    if (k >= p.items) break;
    const int part = k / p.units, u = k - part * p.units;
    // batch row fastest: the items in hand at one time spread over every batch row, so
    // that they do not all read the same C, B tile from L2 at once
    b = u % p.batch;
    const int hb = u / p.batch;
    h = hb / (P / PB);
    pc = (hb % (P / PB)) * PB;
    g = h / p.hpg;
    Ah = p.A[h];
    Dh = p.D ? p.D[h] : 0.f;
    biash = p.dt_bias ? p.dt_bias[h] : 0.f;
    const int c_begin = (int)((int64_t)nch * part / p.nsplit), c_end = (int)((int64_t)nch * (part + 1) / p.nsplit);

    // the first chunk's copies and per-step vectors
    load_chunk(c_begin, gc & 1);
    {
      const int64_t t = (int64_t)c_begin * Q + i;
      dt_next = (t < L) ? __bfloat162float(p.dt[((int64_t)b * L + t) * p.H + h]) : 0.f;
    }
    scan(c_begin);
    // the entering state: h_{-1} or zeros (part 0), else what part - 1 left in the carry
    const float* src = nullptr;
    int64_t src_n = 0;  // the stride of a channel in src
    if (part > 0) {
      const int* f = p.flags + (size_t)(part - 1) * p.units + u;
      bool ready = true;
      if (tid == 0) {
        ready = ld_acquire(f) != 0;
        if (!ready) {
          const uint64_t w0 = gtimer();
          for (long long it = 0; it < (1ll << 30) && !ready; ++it) {
            __nanosleep(256);
            ready = ld_acquire(f) != 0;
            if (!ready && gtimer() - w0 > kWaitNs) break;
          }
        }
      }
      if (!__syncthreads_and(ready)) { ok = false; break; }
      (void)ld_acquire(f);  // every thread acquires the part's release before its reads
      src = p.carry + ((size_t)(part - 1) * p.units + u) * PB * N;
      src_n = N;
    } else if (p.state_in) {
      src = p.state + (((int64_t)b * p.H + h) * P + pc) * N;
      src_n = N;
    }
    // into the state's first accumulator, zeros into the second; lane n = state n,
    // columns of PB channels
#pragma unroll 1
    for (int nb = 0; nb < NP / 128; ++nb) {
      const int n = nb * 128 + i;
      const int c0 = hf * HP;
      uint32_t v[HP], zero[HP];
#pragma unroll
      for (int j = 0; j < HP; ++j) {
        v[j] = __float_as_uint((src && n < N) ? src[(int64_t)(c0 + j) * src_n + n] : 0.f);
        zero[j] = 0u;
      }
      tmem_st16u(lane_t + Sm::T_H + nb * 2 * PB + c0, v);
      tmem_st16u(lane_t + Sm::T_H + nb * 2 * PB + PB + c0, zero);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    state_copy();
    if (!start_g(gc & 1)) { ok = false; break; }

#pragma unroll 1
  for (int c = c_begin; ok && c < c_end; ++c, ++gc) {
    const uint32_t par = gc & 1;
    const int64_t t0 = (int64_t)c * Q;
    const bool valid = t0 + i < L;

    // ---- Xw_j = exp(S_last - S_j) step_j x_j (hi, lo) for this thread's half of the
    // channels; x_i kept for D x_i; z_i fetched
    uint32_t xr[HP / 2];
    uint4 zv[HP / 8];
#pragma unroll
    for (int q = 0; q < HP / 8; ++q) zv[q] = make_uint4(0, 0, 0, 0);
    const int64_t row = (((int64_t)b * L + t0 + i) * p.H + h) * P + pc + hf * HP;  // first channel of the half
    if (p.z && valid) {
#pragma unroll
      for (int q = 0; q < HP / 8; ++q) zv[q] = __ldg(reinterpret_cast<const uint4*>(p.z + row) + q);
    }
    {
      const float wj = ex2f((Slast - Si) * kLog2e) * step;
#pragma unroll
      for (int ch = 0; ch < HP / 8; ++ch) {
        const int cb = hf * (HP / 8) + ch;  // block of 8 channels
        // row i of x: 64 bytes, its 16-byte pieces permuted by bits 1-2 of the row
        const uint4 v = *reinterpret_cast<const uint4*>(smem + Sm::X_OFF + i * 64 + ((cb ^ ((i >> 1) & 3)) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xr[ch * 4 + e] = w[e];
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
          split2(f.x * wj, f.y * wj, hi[e], lo[e]);
        }
        *reinterpret_cast<uint4*>(smem + Sm::W_OFF + cm(i, cb, Q)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(smem + Sm::W_OFF + Q * PB * 2 + cm(i, cb, Q)) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    // ---- Yo = C h_prev (hi + lo); h += B^T Xw (hi + lo)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // C h_prev (K = n)
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < kN; ++k) mma(tmem + Sm::T_YO, dC + off16(kmaj(k)), dH + off16(k * 256), ID_O, k > 0);
      mma_commit(bar_s);
    } else if (tid == 32) {  // per 128 state rows, B^T Xw (K = j)
      tc_fence_after();
      for (int k = 0; k < Q / 16; ++k)
        for (int nb = 0; nb < NP / 128; ++nb)
          mma(tmem + Sm::T_H + nb * 2 * PB, dBt + off16(nb * 2 * kAtom + k * 16 * 128), dW + off16(k * 256), ID_S,
              true);
      mma_commit(bar_s);
    }
    issued |= 2;

    // ---- M[i][j] = G[i][j] exp(S_i - S_j) step_j (j <= i) as a pair of bf16 (hi, lo),
    // written over G in tensor memory: per K step of 16 columns of M, 8 columns of packed
    // hi values, then 8 of lo values (a column block of G becomes exactly the two K steps
    // of M it holds, so each warp overwrites only what it has just read)
    // each warp waits for G on its own (its rows of M need nothing else) and the CTA
    // decides at the next barrier, so that the warps whose threads issue C h_prev and
    // B^T Xw (their issue waits while the tensor pipe is busy) hold back no other warp
    const bool g_ok = __all_sync(0xffffffffu, mbar_wait(bar_g, par));
    if (g_ok) issued &= ~1;
    tc_fence_after();
#pragma unroll 1
    for (int J = hf; g_ok && J < Q / 32; J += 2) {  // the two warps of a quarter take alternate blocks
      const int j0 = J * 32;
      uint32_t mv[32];  // [hi 0-7 | lo 0-7 | hi 8-15 | lo 8-15] of the block's 16 pairs
      if (J <= qw) {  // warp-uniform: blocks right of the diagonal block are zero
        float gv[32];
        tmem_ld32(lane_t + Sm::T_G + j0, gv);
        float m[32];
        if (split) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 b4 = *reinterpret_cast<const float4*>(bv + j0 + 4 * q);
            m[4 * q + 0] = gv[4 * q + 0] * (ai * b4.x);
            m[4 * q + 1] = gv[4 * q + 1] * (ai * b4.y);
            m[4 * q + 2] = gv[4 * q + 2] * (ai * b4.z);
            m[4 * q + 3] = gv[4 * q + 3] * (ai * b4.w);
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) m[jj] = gv[jj] * ex2f((Si - Sv[j0 + jj]) * kLog2e) * stepv[j0 + jj];
        }
        if (J == qw) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) m[jj] = (j0 + jj <= i) ? m[jj] : 0.f;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e)
          split2(m[2 * e], m[2 * e + 1], mv[(e >> 3) * 16 + (e & 7)], mv[(e >> 3) * 16 + 8 + (e & 7)]);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) mv[e] = 0u;
      }
      tmem_st32u(lane_t + Sm::T_G + j0, mv);
    }
    // ---- the first M X accumulator starts from exp(S_i) C h_prev (C h_hi + C h_lo), in
    // the place of C h_hi; the second starts from zero in the place of C h_lo
    if (!__syncthreads_and(g_ok && mbar_wait(bar_s, par))) { ok = false; break; }
    issued &= ~2;
    tc_fence_after();
    {
      const float ei = ex2f(Si * kLog2e);
      const uint32_t ta = lane_t + Sm::T_YO + hf * HP;
      uint32_t ra[HP], rb[HP];
      tmem_ld16x2(ta, ta + PB, ra, rb);
#pragma unroll
      for (int j = 0; j < HP; ++j) ra[j] = __float_as_uint(ei * (__uint_as_float(ra[j]) + __uint_as_float(rb[j])));
      tmem_st16u(ta, ra);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    // ---- Yd = M X: M_hi X onto exp(S) C h_prev, M_lo X beside it; A from tensor memory
    tc_fence_before();
    __syncthreads();
    if (tid == 0 || tid == 32) {
      tc_fence_after();
      const uint32_t part = tid >> 5;
#pragma unroll
      for (int k = 0; k < Q / 16; ++k)
        mma_ta(tmem + Sm::T_YO + part * PB, tmem + Sm::T_G + k * 16 + part * 8, dX + off16(k * 16 * 64), ID_Y,
               part == 0 || k > 0);
      mma_commit(bar_y);
    }
    issued |= 4;
    if (!__syncthreads_and(mbar_wait(bar_y, par))) { ok = false; break; }
    issued &= ~4;
    tc_fence_after();
    // the tiles are consumed: fetch the next chunk's inputs, and while they land form
    // the next chunk's per-step vectors and state copy; then issue the next chunk's G,
    // which runs while this chunk's outputs are formed
    if (c + 1 < c_end) {
      load_chunk(c + 1, (gc + 1) & 1);
      scan(c + 1);
      state_copy();
      if (!start_g((gc + 1) & 1)) { ok = false; break; }
    }

    // ---- y = exp(S_i) Yo + Yd + D x (the two accumulators); out = y silu(z).  The
    // tensor-memory loads are warp-wide (.sync.aligned): every lane takes them, only
    // valid rows store.
    {
      float yd[HP];
      {
        uint32_t ra[HP], rb[HP];
        tmem_ld16x2(lane_t + Sm::T_YO + hf * HP, lane_t + Sm::T_YO + PB + hf * HP, ra, rb);
#pragma unroll
        for (int j = 0; j < HP; ++j) yd[j] = __uint_as_float(ra[j]) + __uint_as_float(rb[j]);
      }
      {
        constexpr int c0 = 0;
#pragma unroll
        for (int q = 0; q < HP / 8; ++q) {
          uint32_t o[4];
          const uint4 zq = p.z ? zv[q] : make_uint4(0, 0, 0, 0);
          const uint32_t zw[4] = {zq.x, zq.y, zq.z, zq.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = q * 8 + 2 * e;
            const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xr[j / 2]));
            float y0 = fmaf(Dh, xf.x, yd[j]);
            float y1 = fmaf(Dh, xf.y, yd[j + 1]);
            if (p.z) {
              const float2 zf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zw[e]));
              y0 *= __fdividef(zf.x, 1.f + ex2f(-zf.x * kLog2e));
              y1 *= __fdividef(zf.y, 1.f + ex2f(-zf.y * kLog2e));
            }
            o[e] = pack2(y0, y1);
          }
          if (valid) reinterpret_cast<uint4*>(p.out + row + c0)[q] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
    tc_fence_before();
  }
    if (!ok) break;

    // ---- the leaving state (the sum of its two accumulators; lane n, columns of PB
    // channels): into the carry of part + 1, or the final state[b, h, pc + j, n]
    const bool to_carry = part + 1 < p.nsplit;
    if (to_carry || p.state) {
      float* dst = to_carry ? p.carry + ((size_t)part * p.units + u) * PB * N
                            : p.state + (((int64_t)b * p.H + h) * P + pc) * N;
#pragma unroll 1
      for (int nb = 0; nb < NP / 128; ++nb) {
        const int n = nb * 128 + i;
        const int c0 = hf * HP;
        uint32_t ra[HP], rb[HP];
        tmem_ld16x2(lane_t + Sm::T_H + nb * 2 * PB + c0, lane_t + Sm::T_H + nb * 2 * PB + PB + c0, ra, rb);
        if (n < N)
#pragma unroll
          for (int j = 0; j < HP; ++j) dst[(int64_t)(c0 + j) * N + n] = __uint_as_float(ra[j]) + __uint_as_float(rb[j]);
      }
    }
    if (to_carry) {
      __syncthreads();  // every thread's carry stores come before the release
      if (tid == 0 && !(part == 0 && u == p.hold_unit)) {
        __threadfence();
        st_release(p.flags + (size_t)part * p.units + u, 1);
      }
    }
  }
  if (!ok && tid == 0) atomicExch(p.status, 1);

  // after a wait that ran out, let the tensor copy and the products still in flight
  // finish (each wait bounded) before the shared and tensor memory are released
  if (!ok && tid == 0) {  // the products outstanding belong to one chunk (parity cur)
    if (in_flight) mbar_wait(bar_in, in_par);
    if (issued & 1) mbar_wait(bar_g, cur);
    if (issued & 2) mbar_wait(bar_s, cur);
    if (issued & 4) mbar_wait(bar_y, cur);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Sm::TCOLS) : "memory");
}

}  // namespace ssd
