// expert_choice.cuh -- expert-choice routing: each expert picks its tokens.
//
// "MoE混合专家模型计算原理与推理部署实战解析" section 2.3: instead of every
// token choosing its top experts, every expert chooses its top tokens, so each
// expert processes exactly the same number of tokens and a token may be
// chosen by none. The affinity is the gate probability p[t,e] (the softmax
// over experts of token t's fp32 logits, written by the route kernel); expert
// e takes the C tokens of largest p[t,e], equal values going to the lower
// token id, and weights each by p[t,e].
//
// One CTA per expert. The C-th largest key of the column p[:, e] is found by
// a most-significant-digit radix select over the fp32 bit patterns (p >= 0,
// so the unsigned patterns order like the values): four passes of 8-bit
// digits, each a shared-memory histogram of the keys that still match the
// prefix. A last pass walks the tokens in order with block-wide scans: every
// key above the threshold is taken, and of the keys equal to it the lowest
// token ids, up to C in all. Expert e's rows e*C .. e*C + C - 1 receive its
// tokens in ascending order (the layout the grouped GEMMs take), and the
// per-token tables inv [T,N] (row or -2) and w [T,N] (p or 0) feed the row
// copy and the combine unchanged (as a top-k with k = N). Integer counts
// only: the choice is deterministic.
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kEcThreads = 1024;
constexpr int32_t kNotChosen = -2;

// Exclusive scan of one value per thread over the 1024-thread block, in
// thread order; *total receives the block sum. Contains __syncthreads.
__device__ inline int ec_block_excl_scan(int v, int* s_warp, int* s_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int wv = s_warp[lane];
    int wi = wv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    s_warp[lane] = wi - wv;
    if (lane == 31) *s_total = wi;
  }
  __syncthreads();
  const int r = s_warp[warp] + incl - v;
  __syncthreads();   // s_warp is reused by the next scan
  return r;
}

__global__ void __launch_bounds__(kEcThreads) ec_select_kernel(const float* __restrict__ probs, int64_t T, int N,
                                                               int64_t C, int32_t* __restrict__ perm,
                                                               int32_t* __restrict__ counts,
                                                               int32_t* __restrict__ offsets,
                                                               int32_t* __restrict__ inv, float* __restrict__ w) {
  __shared__ int hist[256];
  __shared__ int s_warp[32];
  __shared__ int s_total;
  __shared__ int s_digit;
  __shared__ long long s_above;
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    counts[e] = static_cast<int32_t>(C);
    offsets[e] = static_cast<int32_t>(e * C);
    if (e == N - 1) offsets[N] = static_cast<int32_t>(N * C);
  }
  // radix select: prefix / mask describe the threshold's digits found so far;
  // `remaining` counts how many of the keys matching the prefix are still to
  // be taken (at the end: how many keys equal to the threshold are taken).
  uint32_t prefix = 0, mask = 0;
  long long remaining = C;
  if (C > 0) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kEcThreads) hist[i] = 0;
      __syncthreads();
      for (int64_t t = tid; t < T; t += kEcThreads) {
        const uint32_t key = __float_as_uint(probs[t * N + e]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      if (warp == 0) {
        // lane L owns digits 255 - 8L down to 248 - 8L: counts from the top
        int c8 = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) c8 += hist[255 - 8 * lane - j];
        int incl = c8;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        const long long above = incl - c8;
        if (above < remaining && remaining <= incl) {
          long long acc = above;
          for (int j = 0; j < 8; ++j) {
            const int b = 255 - 8 * lane - j;
            if (acc + hist[b] >= remaining) {
              s_digit = b;
              s_above = acc;
              break;
            }
            acc += hist[b];
          }
        }
      }
      __syncthreads();
      prefix |= static_cast<uint32_t>(s_digit) << shift;
      mask |= 255u << shift;
      remaining -= s_above;
      __syncthreads();   // hist and s_digit are rewritten by the next pass
    }
  }
  // take the keys above the threshold, and the first `remaining` equal ones
  long long base_eq = 0, base_sel = 0;
  for (int64_t t0 = 0; t0 < T; t0 += kEcThreads) {
    const int64_t t = t0 + tid;
    const bool in = t < T;
    const float p = in ? probs[t * N + e] : 0.f;
    const uint32_t key = __float_as_uint(p);
    const bool gt = C > 0 && in && key > prefix;
    const bool eq = C > 0 && in && key == prefix;
    int tot_eq, tot_sel;
    const int eq_rank = ec_block_excl_scan(eq ? 1 : 0, s_warp, &s_total);
    tot_eq = s_total;
    const bool sel = gt || (eq && base_eq + eq_rank < remaining);
    const int rank = ec_block_excl_scan(sel ? 1 : 0, s_warp, &s_total);
    tot_sel = s_total;
    if (in) {
      int32_t row = kNotChosen;
      if (sel) {
        row = static_cast<int32_t>(e * C + base_sel + rank);
        perm[row] = static_cast<int32_t>(t);
      }
      inv[t * N + e] = row;
      w[t * N + e] = sel ? p : 0.f;
    }
    base_eq += tot_eq;
    base_sel += tot_sel;
  }
}

}  // namespace moe
