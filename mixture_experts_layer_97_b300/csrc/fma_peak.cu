// fma_peak.cu -- microbenchmark of the GPU's fp32 FMA throughput on the CUDA
// cores, the roofline denominator of the gate projection (the route kernel
// evaluates every logit as an fp32 FMA chain). Built as its own small library
// (libmoe_fma_peak.so) for the benchmark; the MoE library does not use it.
//
// Each thread runs CHAINS independent FMA chains for `iters` steps, either as
// scalar fma.rn.f32 or as packed fma.rn.f32x2 (two chains per instruction,
// the form the route kernel issues). The values stay in a bounded range
// (a <- a * m + c with m < 1), so no chain reaches inf or a denormal. The sum
// of every thread's chains is written out so the work cannot be elided.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kChains = 16;

__global__ void __launch_bounds__(256) fma_peak_scalar_kernel(float* __restrict__ out, int iters) {
  float a[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j) a[j] = 1.0f + 1e-3f * static_cast<float>((threadIdx.x + j) & 63);
  const float m = 0.999f, c = 1e-3f;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
#pragma unroll
      for (int j = 0; j < kChains; ++j) a[j] = fmaf(a[j], m, c);
    }
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) s += a[j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void __launch_bounds__(256) fma_peak_packed_kernel(float* __restrict__ out, int iters) {
  unsigned long long a[kChains / 2];
#pragma unroll
  for (int j = 0; j < kChains / 2; ++j) {
    const float lo = 1.0f + 1e-3f * static_cast<float>((threadIdx.x + 2 * j) & 63);
    const float hi = 1.0f + 1e-3f * static_cast<float>((threadIdx.x + 2 * j + 1) & 63);
    asm("mov.b64 %0, {%1, %2};" : "=l"(a[j]) : "f"(lo), "f"(hi));
  }
  unsigned long long m, c;
  asm("mov.b64 %0, {%1, %1};" : "=l"(m) : "f"(0.999f));
  asm("mov.b64 %0, {%1, %1};" : "=l"(c) : "f"(1e-3f));
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
#pragma unroll
      for (int j = 0; j < kChains / 2; ++j) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(a[j]) : "l"(m), "l"(c));
    }
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kChains / 2; ++j) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a[j]));
    s += lo + hi;
  }
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

extern "C" {

// FLOPs one launch performs: 2 per FMA.
double moe_fma_peak_flops(int blocks, int threads, int iters) {
  return 2.0 * kChains * 8.0 * static_cast<double>(iters) * blocks * threads;
}

// Launch the scalar (packed = 0) or f32x2 (packed = 1) kernel on `stream`;
// out holds blocks * threads floats. Returns 0, or the CUDA error code.
int moe_fma_peak_launch(float* out, int blocks, int threads, int iters, int packed, void* stream) {
  if (out == nullptr || blocks < 1 || threads < 32 || threads > 256 || iters < 1) return cudaErrorInvalidValue;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (packed)
    fma_peak_packed_kernel<<<blocks, threads, 0, st>>>(out, iters);
  else
    fma_peak_scalar_kernel<<<blocks, threads, 0, st>>>(out, iters);
  return static_cast<int>(cudaGetLastError());
}

}  // extern "C"
