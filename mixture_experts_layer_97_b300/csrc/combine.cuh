// combine.cuh -- K4: weighted un-permute back to token order.
//
// "MoE显存与计算开销四阶段手算指南" section 2.4 and
// "MoE混合专家模型计算原理与推理部署实战解析" sections 2.2 and 5.1 step 5:
//   out[t,:] = sum_{j<k} w[t,j] * y_perm[inv_perm[t*k+j], :]
// (an assignment dropped by an expert capacity, inv_perm = -2, adds nothing)
// A flat grid of warps over (token, group of 16-byte column chunks): each
// lane accumulates its chunks of the k gathered rows in fp32 in j order and
// writes them once. No zero-fill and no atomics, so the result is bitwise
// reproducible.
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kCombineThreads = 256;

template <typename T>
struct Vec8;  // 8 bf16 (16 B) or 4 fp32 (16 B) per chunk

template <>
struct Vec8<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ static void load_acc(const void* p, float w, float* acc) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    acc[0] = fmaf(w, bf16_lo(q.x), acc[0]); acc[1] = fmaf(w, bf16_hi(q.x), acc[1]);
    acc[2] = fmaf(w, bf16_lo(q.y), acc[2]); acc[3] = fmaf(w, bf16_hi(q.y), acc[3]);
    acc[4] = fmaf(w, bf16_lo(q.z), acc[4]); acc[5] = fmaf(w, bf16_hi(q.z), acc[5]);
    acc[6] = fmaf(w, bf16_lo(q.w), acc[6]); acc[7] = fmaf(w, bf16_hi(q.w), acc[7]);
  }
  __device__ static void store(void* p, const float* acc) {
    uint4 q;
    q.x = pack_bf16x2(acc[0], acc[1]); q.y = pack_bf16x2(acc[2], acc[3]);
    q.z = pack_bf16x2(acc[4], acc[5]); q.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(p) = q;
  }
};

template <>
struct Vec8<float> {
  static constexpr int kElems = 4;
  __device__ static void load_acc(const void* p, float w, float* acc) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    acc[0] = fmaf(w, q.x, acc[0]); acc[1] = fmaf(w, q.y, acc[1]);
    acc[2] = fmaf(w, q.z, acc[2]); acc[3] = fmaf(w, q.w, acc[3]);
  }
  __device__ static void store(void* p, const float* acc) {
    *reinterpret_cast<float4*>(p) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  }
};

// Warp w owns token t = w / G and a group of 32*CPT 16-byte chunks of the
// output row, lane strided (each load instruction covers 512 contiguous
// bytes). The token's k (row, weight) pairs are loaded once per warp.
template <int CPT>
__host__ __device__ inline int combine_groups(int nchunk) { return (nchunk + 32 * CPT - 1) / (32 * CPT); }

// KMAX > 0: k <= KMAX, and the k (row, weight) pairs and then all k rows'
// chunks are loaded before any is summed, so a lane has k * CPT row loads in
// flight; KMAX = 0: any k, live slots found by a warp ballot and summed one
// row after the other (the expert-choice path, where k is the number of
// experts and most slots are empty).
template <typename T, int CPT, int KMAX>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const T* __restrict__ y_perm,
                                                                  const int32_t* __restrict__ inv_perm,
                                                                  const float* __restrict__ topk_w, int64_t T_tok,
                                                                  int d, int k, int64_t A, T* __restrict__ out) {
  constexpr int E = Vec8<T>::kElems;
  const int nchunk = d / E;
  const int G = combine_groups<CPT>(nchunk);
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * kCombineThreads + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= T_tok * G) return;
  const int64_t t = gw / G;
  const int c0 = static_cast<int>(gw % G) * 32 * CPT + lane;
  float acc[CPT][E];
#pragma unroll
  for (int u = 0; u < CPT; ++u)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[u][e] = 0.f;
  if constexpr (KMAX > 0) {
    int64_t row[KMAX];
    float wt[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      row[j] = j < k ? inv_perm[t * k + j] : -2;
      wt[j] = j < k ? topk_w[t * k + j] : 0.f;
    }
    uint4 q[KMAX][CPT];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      const bool live = row[j] >= 0 && row[j] < A;
      if (row[j] != -2 && !live && c0 == 0) record_error(MOE_ERR_CORRUPT);
      const T* yr = y_perm + (live ? row[j] : 0) * d;
#pragma unroll
      for (int u = 0; u < CPT; ++u) {
        const int c = c0 + 32 * u;
        q[j][u] = (live && c < nchunk) ? *reinterpret_cast<const uint4*>(yr + static_cast<int64_t>(c) * E)
                                       : make_uint4(0, 0, 0, 0);
      }
    }
    // sum in j order; a dropped or empty slot (-2) adds nothing
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (!(row[j] >= 0 && row[j] < A)) continue;
#pragma unroll
      for (int u = 0; u < CPT; ++u) Vec8<T>::load_acc(&q[j][u], wt[j], acc[u]);
    }
  } else {
    // many slots, few of them live (expert choice: k = N): each lane reads one
    // slot, a ballot lists the live ones, and the warp sums their rows in slot order
    const bool first_group = (gw % G) == 0;
    for (int j0 = 0; j0 < k; j0 += 32) {
      const int j = j0 + lane;
      const int64_t r = j < k ? inv_perm[t * k + j] : -2;
      const float wj = j < k ? topk_w[t * k + j] : 0.f;
      const bool live = r >= 0 && r < A;
      if (r != -2 && !live && first_group) record_error(MOE_ERR_CORRUPT);
      unsigned m = __ballot_sync(0xffffffffu, live);
      while (m != 0u) {
        const int b = __ffs(m) - 1;
        m &= m - 1u;
        const int64_t row = __shfl_sync(0xffffffffu, r, b);
        const float w = __shfl_sync(0xffffffffu, wj, b);
        const T* yr = y_perm + row * d;
#pragma unroll
        for (int u = 0; u < CPT; ++u) {
          const int c = c0 + 32 * u;
          if (c < nchunk) Vec8<T>::load_acc(yr + static_cast<int64_t>(c) * E, w, acc[u]);
        }
      }
    }
  }
#pragma unroll
  for (int u = 0; u < CPT; ++u) {
    const int c = c0 + 32 * u;
    if (c < nchunk) Vec8<T>::store(out + t * d + static_cast<int64_t>(c) * E, acc[u]);
  }
}

}  // namespace moe
