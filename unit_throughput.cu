// Throughput of the B300 units the selective scan's state update runs on, per SM and
// clock: MUFU ex2 (f32, f16x2, bf16x2), FP32 fma (scalar and f32x2 pairs), and ex2
// overlapped with f32x2 fma.  The arithmetic roofline of bench.py is derived from it.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o unit_throughput unit_throughput.cu
//   ./unit_throughput
//
// Each thread runs 8 independent chains for ITERS iterations; 2 CTAs of 512 threads
// per SM (32 warps); cycles are taken with clock64 on the SM itself, so the result is
// independent of the clock frequency.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#define ITERS 4096
__device__ __forceinline__ float ex2ftz(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0,%1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ unsigned ex2h2(unsigned x) {
  unsigned y;
  asm volatile("ex2.approx.f16x2 %0,%1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ unsigned ex2bf2(unsigned x) {
  unsigned y;
  asm volatile("ex2.approx.ftz.bf16x2 %0,%1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ float ffma(float a, float b, float c) {
  float y;
  asm volatile("fma.rn.f32 %0,%1,%2,%3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long A = *(unsigned long long*)&a, B = *(unsigned long long*)&b, C = *(unsigned long long*)&c, Y;
  asm volatile("fma.rn.f32x2 %0,%1,%2,%3;" : "=l"(Y) : "l"(A), "l"(B), "l"(C));
  return *(float2*)&Y;
}

template <int MODE>
__global__ void probe(float* out, long long* cyc, float seed) {
  float v[8];
  unsigned u[8];
  float2 w[8];
  for (int i = 0; i < 8; i++) {
    v[i] = seed * (i + 1) * 1e-3f - 0.5f;
    u[i] = 0x3c003c00u + i;
    w[i] = make_float2(v[i], v[i] + 1.f);
  }
  const float2 m = make_float2(0.999f, 0.998f), c2 = make_float2(1e-3f, 2e-3f);
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < ITERS; it++) {
#pragma unroll
    for (int i = 0; i < 8; i++) {
      if (MODE == 0) v[i] = ex2ftz(v[i]);
      if (MODE == 1) u[i] = ex2h2(u[i]);
      if (MODE == 2) u[i] = ex2bf2(u[i]);
      if (MODE == 3) v[i] = ffma(v[i], 0.999f, 1e-3f);
      if (MODE == 4) w[i] = ffma2(w[i], m, c2);
      if (MODE == 5) {
        v[i] = ex2ftz(v[i]);
        w[i] = ffma2(w[i], m, c2);
        w[i] = ffma2(w[i], m, c2);
      }
    }
  }
  const long long t1 = clock64();
  float s = 0;
  for (int i = 0; i < 8; i++) s += v[i] + __uint_as_float(u[i]) + w[i].x + w[i].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const int threads = 512, blocks = sms * 2;
  float* out;
  long long* cyc;
  cudaMalloc(&out, sizeof(float) * threads * blocks);
  cudaMalloc(&cyc, 8 * blocks);
  const char* names[] = {"ex2.approx.ftz.f32", "ex2.approx.f16x2", "ex2.approx.ftz.bf16x2",
                         "fma.rn.f32", "fma.rn.f32x2", "ex2.f32 + 2 fma.f32x2"};
  const double mufu[] = {1, 1, 1, 0, 0, 1}, fma_lanes[] = {0, 0, 0, 1, 2, 4};
  void (*ks[])(float*, long long*, float) = {probe<0>, probe<1>, probe<2>, probe<3>, probe<4>, probe<5>};
  long long* h = new long long[blocks];
  for (int m = 0; m < 6; m++) {
    ks[m]<<<blocks, threads>>>(out, cyc, 1.f);
    ks[m]<<<blocks, threads>>>(out, cyc, 1.f);
    cudaDeviceSynchronize();
    cudaMemcpy(h, cyc, 8 * blocks, cudaMemcpyDeviceToHost);
    double mx = 0;
    for (int b = 0; b < blocks; b++) mx = h[b] > mx ? h[b] : mx;
    const double ops = 2.0 * threads * 8.0 * ITERS;  // per SM: 2 CTAs x threads x chains x iters
    printf("%-24s per SM per clock: %6.1f MUFU instructions, %6.1f FMA lanes  (%s)\n", names[m],
           ops * mufu[m] / mx, ops * fma_lanes[m] / mx, cudaGetErrorString(cudaGetLastError()));
  }
  delete[] h;
  return 0;
}
