// route.cuh -- K1: fused gate projection + top-k + renormalised gate weights.
//
// "MoE显存与计算开销四阶段手算指南" sections 2.1-2.2 and
// "MoE混合专家模型计算原理与推理部署实战解析" sections 2.1, 2.2, 2.4:
//   s[t,n] = sum_i x[t,i] W_g[i,n] (+ b[n])  in fp32 (the gate is kept in fp32)
//   the k largest s (ties -> lower expert id), in descending order
//   w_j = softmax(s)_{e_j} / sum_j' softmax(s)_{e_j'}
// The full softmax denominator cancels in the renormalisation, so the kernel
// evaluates w_j = exp(s_j - s_max) / sum_j' exp(s_j' - s_max) over the k
// selected scores only (identical in exact arithmetic).
//
// One CTA owns 64 tokens and all N experts (N padded to NP = 16*EPT). The
// 64 x NP logit tile is accumulated in registers (4 tokens x EPT experts per
// thread) from 32-wide K slices of x and W_g staged in shared memory, then
// written to shared memory where one warp per token runs k rounds of a
// warp-wide argmax. Logits never reach global memory.
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kRouteTokens = 64;
constexpr int kRouteBK = 32;
constexpr int kRouteThreads = 256;

template <int EPT>
constexpr size_t route_smem_bytes() {
  constexpr int NP = 16 * EPT;
  constexpr size_t tiles = sizeof(float) * (kRouteBK * kRouteTokens + kRouteBK * NP);
  constexpr size_t logits = sizeof(float) * kRouteTokens * (NP + 1);
  return tiles > logits ? tiles : logits;
}

template <typename TX>
__device__ __forceinline__ void route_load_x8(const TX* p, float* v);

template <>
__device__ __forceinline__ void route_load_x8<__nv_bfloat16>(const __nv_bfloat16* p, float* v) {
  uint4 q = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
  v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
}

template <>
__device__ __forceinline__ void route_load_x8<float>(const float* p, float* v) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }

// EPT: experts per thread (NP = 16*EPT >= N). TX: element type of x.
template <int EPT, typename TX>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const TX* __restrict__ x, const float* __restrict__ wg,
                                                              const float* __restrict__ bias, int T, int d, int N,
                                                              int k, int32_t* __restrict__ topk_idx,
                                                              float* __restrict__ topk_w) {
  constexpr int NP = 16 * EPT;
  constexpr int NPR = NP < 32 ? 32 : NP;  // register slots per token for the argmax
  constexpr int SLOTS = NPR / 32;
  extern __shared__ __align__(16) float rsm[];
  float* xs = rsm;                              // [BK][64] (transposed x tile)
  float* ws = rsm + kRouteBK * kRouteTokens;    // [BK][NP]
  float* lg = rsm;                              // [64][NP+1] after the K loop

  const int tid = threadIdx.x;
  const int tx = tid & 15;   // expert group: experts tx + 16*j
  const int ty = tid >> 4;   // token group: tokens 4*ty .. 4*ty+3
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kRouteTokens;

  float acc[4][EPT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < EPT; ++j) acc[i][j] = 0.f;

  // x tile loader mapping: token = tid % 64, 8 consecutive k from kq*8.
  const int ltok = tid & 63;
  const int lkq = tid >> 6;  // 0..3
  const bool vec_ok = (d % 8) == 0;

  for (int kb = 0; kb < d; kb += kRouteBK) {
    {  // x slice -> xs[k][token]
      const int64_t t = t0 + ltok;
      const int kk0 = kb + lkq * 8;
      float v[8];
      if (t < T && vec_ok && kk0 + 8 <= d) {
        route_load_x8<TX>(x + t * d + kk0, v);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = (t < T && kk0 + i < d) ? to_f32(x[t * d + kk0 + i]) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[(lkq * 8 + i) * kRouteTokens + ltok] = v[i];
    }
    // W_g slice -> ws[k][n]
    for (int idx = tid; idx < kRouteBK * NP; idx += kRouteThreads) {
      const int kk = idx / NP, n = idx % NP;
      const int gk = kb + kk;
      ws[idx] = (gk < d && n < N) ? wg[static_cast<int64_t>(gk) * N + n] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kRouteBK; ++kk) {
      const float4 xv = *reinterpret_cast<const float4*>(&xs[kk * kRouteTokens + ty * 4]);
      float wv[EPT];
#pragma unroll
      for (int j = 0; j < EPT; ++j) wv[j] = ws[kk * NP + tx + 16 * j];
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        acc[0][j] = fmaf(xv.x, wv[j], acc[0][j]);
        acc[1][j] = fmaf(xv.y, wv[j], acc[1][j]);
        acc[2][j] = fmaf(xv.z, wv[j], acc[2][j]);
        acc[3][j] = fmaf(xv.w, wv[j], acc[3][j]);
      }
    }
    __syncthreads();
  }

  // logits (+ bias) -> lg[token][n]; padded experts get -inf
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int n = tx + 16 * j;
    const float b = (bias != nullptr && n < N) ? bias[n] : 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) lg[(ty * 4 + i) * (NP + 1) + n] = (n < N) ? acc[i][j] + b : -INFINITY;
  }
  __syncthreads();

  // top-k: one warp per token, k rounds of warp argmax (ties -> lower id)
  const int warp = tid >> 5, lane = tid & 31;
  for (int tl = warp; tl < kRouteTokens; tl += kRouteThreads / 32) {
    const int64_t t = t0 + tl;
    if (t >= T) break;
    float v[SLOTS];
    bool taken[SLOTS];
#pragma unroll
    for (int m = 0; m < SLOTS; ++m) {
      const int n = lane + 32 * m;
      v[m] = (n < NP) ? lg[tl * (NP + 1) + n] : -INFINITY;
      taken[m] = (n >= N);
    }
    float sel_v[SLOTS];
    int sel_i[SLOTS];
#pragma unroll
    for (int m = 0; m < SLOTS; ++m) { sel_v[m] = -INFINITY; sel_i[m] = 0; }
    float top = 0.f;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
#pragma unroll
      for (int m = 0; m < SLOTS; ++m) {
        const int n = lane + 32 * m;
        if (!taken[m] && (v[m] > bv || (v[m] == bv && n < bi))) { bv = v[m]; bi = n; }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (j == 0) top = bv;
#pragma unroll
      for (int m = 0; m < SLOTS; ++m) {
        if (bi == lane + 32 * m) taken[m] = true;
        if ((j & 31) == lane && (j >> 5) == m) { sel_v[m] = bv; sel_i[m] = bi; }
      }
    }
    float part = 0.f;
    float ex[SLOTS];
#pragma unroll
    for (int m = 0; m < SLOTS; ++m) {
      const int j = lane + 32 * m;
      ex[m] = (j < k) ? expf(sel_v[m] - top) : 0.f;
      part += ex[m];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    const float inv = 1.f / part;
#pragma unroll
    for (int m = 0; m < SLOTS; ++m) {
      const int j = lane + 32 * m;
      if (j < k) {
        topk_idx[t * k + j] = sel_i[m];
        topk_w[t * k + j] = ex[m] * inv;
      }
    }
  }
}

}  // namespace moe
