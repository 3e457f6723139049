// ffn_simt.cuh -- fp32 grouped GEMM with fused activation on CUDA cores.
//
// The fp32 layer keeps every value in fp32 (tf32 tensor cores would not hold
// a 1e-4 relative error), so its expert FFN runs as a classic shared-memory
// tiled SIMT GEMM: 64 x 64 output tile per CTA, K slices of 16, 4 x 4
// outputs per thread. Same tile schedule as the tensor-core path.
//   EPI_SWIGLU: out = silu(A B0^T) * (A B1^T)   ("MoE混合专家模型计算原理与推理部署实战解析" s3.1)
//   EPI_GELU:   out = gelu_tanh(A B0^T)
//   EPI_PLAIN:  out = A B0^T
#pragma once
#include "schedule.cuh"

namespace moe {

enum { EPI_PLAIN = 0, EPI_SWIGLU = 1, EPI_GELU = 2 };

constexpr int kSimtBM = 64, kSimtBN = 64, kSimtBK = 16;

__device__ __forceinline__ float silu_f(float v) { return v / (1.f + expf(-v)); }
__device__ __forceinline__ float gelu_tanh_f(float v) {
  return 0.5f * v * (1.f + tanhf(0.7978845608028654f * (v + 0.044715f * v * v * v)));
}

template <int EPI>
__global__ void __launch_bounds__(256) grouped_gemm_simt_kernel(const float* __restrict__ A,
                                                                const int32_t* __restrict__ offsets, int N,
                                                                int rows_total, const float* __restrict__ B0,
                                                                const float* __restrict__ B1, int K, int Nout,
                                                                float* __restrict__ out, int ldo) {
  constexpr bool TWO = (EPI == EPI_SWIGLU);
  __shared__ int s_off[257], s_pre[257], s_bad;
  __shared__ float As[kSimtBK][kSimtBM + 4];
  __shared__ float Bs[kSimtBK][kSimtBN + 4];
  __shared__ float Bs2[TWO ? kSimtBK : 1][kSimtBN + 4];

  if (threadIdx.x < 32) build_tile_prefix(offsets, N, rows_total, kSimtBM, s_off, s_pre, &s_bad);
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) record_error(MOE_ERR_CORRUPT);
    return;
  }
  if (static_cast<int>(blockIdx.x) >= s_pre[N]) return;
  const TileInfo ti = decode_tile(blockIdx.x, s_off, s_pre, N, 1, kSimtBM);
  const int n0 = blockIdx.y * kSimtBN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;

  float acc[4][4], acc2[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = acc2[i][j] = 0.f;

  const float* Bbase0 = B0 + static_cast<int64_t>(ti.e) * Nout * K;
  const float* Bbase1 = TWO ? B1 + static_cast<int64_t>(ti.e) * Nout * K : nullptr;
  for (int kb = 0; kb < K; kb += kSimtBK) {
    for (int i = threadIdx.x; i < kSimtBM * kSimtBK; i += 256) {
      const int r = i / kSimtBK, kk = i % kSimtBK;
      const int gk = kb + kk;
      As[kk][r] = (r < ti.rows && gk < K) ? A[static_cast<int64_t>(ti.row0 + r) * K + gk] : 0.f;
      const int c = n0 + r;   // kSimtBN == kSimtBM
      Bs[kk][r] = (c < Nout && gk < K) ? Bbase0[static_cast<int64_t>(c) * K + gk] : 0.f;
      if (TWO) Bs2[kk][r] = (c < Nout && gk < K) ? Bbase1[static_cast<int64_t>(c) * K + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kSimtBK; ++kk) {
      float a[4], b[4], b2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b[j] = Bs[kk][tx + 16 * j];
        if (TWO) b2[j] = Bs2[kk][tx + 16 * j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if (TWO) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty + 16 * i;
    if (r >= ti.rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + tx + 16 * j;
      if (c >= Nout) continue;
      float v = acc[i][j];
      if (EPI == EPI_SWIGLU) v = silu_f(v) * acc2[i][j];
      if (EPI == EPI_GELU) v = gelu_tanh_f(v);
      out[static_cast<int64_t>(ti.row0 + r) * ldo + c] = v;
    }
  }
}

}  // namespace moe
