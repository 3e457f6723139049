// permute.cuh -- K2: group the T*k token-expert assignments by expert.
//
// "MoE显存与计算开销四阶段手算指南" section 2.3 and
// "MoE混合专家模型计算原理与推理部署实战解析" section 5.1 steps 2-3:
// count per expert, exclusive prefix sum into offsets, then move every
// assignment's input row into one contiguous buffer ordered by expert.
//
// A deterministic stable counting sort by flat index f = t*k + j, in four
// launches:
//   hist    per chunk of whole tokens (at most 2048 assignments): expert
//           histogram (shared-memory integer atomics: counts do not depend
//           on their order)
//   scan    one CTA: counts, offsets, and the rank base of every
//           (chunk, expert) pair
//   rank    per chunk: stable ranks from warp __match_any_sync + popc in flat
//           order -> perm / inv_perm; with an expert capacity ("MoE混合专家模型
//           计算原理与推理部署实战解析" section 4.3) ranks >= capacity are
//           dropped (inv_perm = -2) and counted
//   copy    flat grid of warps over (token, 2 KB slice of its row): each warp
//           reads its slice of x once with 128-bit loads and writes it to the
//           token's k rows, so the copy spreads over every SM.
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kPermThreads = 256;
constexpr int kPermMaxChunk = 2048;   // assignments per chunk
constexpr int kPermWarps = kPermThreads / 32;
constexpr int kPermSub = kPermMaxChunk / kPermWarps;  // assignments per warp

__host__ __device__ inline int perm_tokens_per_chunk(int k) {
  const int t = kPermMaxChunk / k;
  return t < 1 ? 1 : t;
}

__global__ void __launch_bounds__(kPermThreads) permute_hist_kernel(const int32_t* __restrict__ topk_idx, int64_t T,
                                                                    int N, int k, int32_t* __restrict__ hist) {
  __shared__ int h[256];
  const int tpc = perm_tokens_per_chunk(k);
  const int64_t c = blockIdx.x;
  const int64_t f0 = c * tpc * k;
  const int64_t f1 = min(T, (c + 1) * static_cast<int64_t>(tpc)) * k;
  for (int n = threadIdx.x; n < N; n += blockDim.x) h[n] = 0;
  __syncthreads();
  for (int64_t f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
    const int e = topk_idx[f];
    if (e < 0 || e >= N) {
      record_error(MOE_ERR_CORRUPT);
      continue;
    }
    atomicAdd(&h[e], 1);
  }
  __syncthreads();
  for (int n = threadIdx.x; n < N; n += blockDim.x) hist[c * N + n] = h[n];
}

// Single CTA of 256 threads; thread n owns expert n. On return hist[c][n]
// holds the number of expert n's assignments in chunks before c (its rank
// base); counts / offsets describe the KEPT rows: min(demand, capacity) per
// expert ("MoE混合专家模型计算原理与推理部署实战解析" section 4.3; capacity =
// INT64_MAX keeps everything). *dropped (optional) is zeroed for the rank pass.
__global__ void __launch_bounds__(256) permute_scan_kernel(int32_t* __restrict__ hist, int n_chunks, int N,
                                                           long long capacity, int32_t* __restrict__ counts,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ dropped) {
  __shared__ int warp_sums[8];
  const int n = threadIdx.x;
  int run = 0;
  if (n < N) {
    for (int c = 0; c < n_chunks; ++c) {
      const int v = hist[static_cast<int64_t>(c) * N + n];
      hist[static_cast<int64_t>(c) * N + n] = run;   // rank base of chunk c within expert n
      run += v;
    }
  }
  const int kept = static_cast<int>(run < capacity ? run : capacity);
  // exclusive scan of the kept counts over experts
  const int lane = n & 31, w = n >> 5;
  int incl = kept;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[w] = incl;
  __syncthreads();
  int wbase = 0;
  for (int i = 0; i < w; ++i) wbase += warp_sums[i];
  if (n < N) {
    counts[n] = kept;
    offsets[n] = wbase + incl - kept;
  }
  if (n == 255) offsets[N] = wbase + incl;   // kept rows (T*k when nothing is dropped or corrupt)
  if (n == 0 && dropped != nullptr) *dropped = 0;
}

// Marker of an assignment dropped by the capacity limit in inv_perm.
constexpr int32_t kDroppedRow = -2;

__global__ void __launch_bounds__(kPermThreads) permute_rank_kernel(const int32_t* __restrict__ topk_idx,
                                                                    const int32_t* __restrict__ base,
                                                                    const int32_t* __restrict__ offsets, int64_t T,
                                                                    int N, int k, long long capacity,
                                                                    int32_t* __restrict__ perm,
                                                                    int32_t* __restrict__ inv_perm,
                                                                    int32_t* __restrict__ dropped) {
  __shared__ int wh[kPermWarps][256];
  const int tpc = perm_tokens_per_chunk(k);
  const int64_t c = blockIdx.x;
  const int64_t tok0 = c * tpc;
  const int ntok = static_cast<int>(min(T, tok0 + static_cast<int64_t>(tpc)) - tok0);
  const int nf = ntok * k;
  const int64_t f0 = tok0 * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;

  for (int i = threadIdx.x; i < kPermWarps * 256; i += blockDim.x) (&wh[0][0])[i] = 0;
  __syncthreads();

  const int s0 = warp * kPermSub;
  const int s1 = min(nf, s0 + kPermSub);
  // pass 1: per-warp histogram over the warp's contiguous sub-range
  for (int g = s0; g < s1; g += 32) {
    const int fl = g + lane;
    int e = (fl < s1) ? topk_idx[f0 + fl] : -1;
    if (e >= N) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (peers & lt_mask) == 0) wh[warp][e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // pass 2: per-expert prefix over warps, starting at the chunk's rank base
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    int run = base[c * N + n];
#pragma unroll
    for (int w = 0; w < kPermWarps; ++w) {
      const int v = wh[w][n];
      wh[w][n] = run;
      run += v;
    }
  }
  __syncthreads();
  // pass 3: stable ranks in flat order; rank >= capacity is dropped
  int n_drop = 0;
  for (int g = s0; g < s1; g += 32) {
    const int fl = g + lane;
    int e = (fl < s1) ? topk_idx[f0 + fl] : -1;
    if (e >= N) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    int rank = -1;
    if (e >= 0) rank = wh[warp][e] + __popc(peers & lt_mask);
    __syncwarp();
    if (e >= 0 && (peers & lt_mask) == 0) wh[warp][e] += __popc(peers);
    __syncwarp();
    if (fl < s1) {
      int row = -1;
      if (e >= 0) {
        if (rank < capacity) {
          row = offsets[e] + rank;
          perm[row] = static_cast<int32_t>((f0 + fl) / k);
        } else {
          row = kDroppedRow;
          ++n_drop;
        }
      }
      inv_perm[f0 + fl] = row;
    }
  }
  if (dropped != nullptr) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) n_drop += __shfl_xor_sync(0xffffffffu, n_drop, off);
    if (lane == 0 && n_drop > 0) atomicAdd(dropped, n_drop);   // integer: order-independent
  }
}

// Row copies x[t] -> x_perm[inv_perm[t*k+j]] for j < k. Warp w owns token
// t = w / G and a group of 32*kCopyUnroll 16-byte chunks of its row, lane
// strided so every load and store instruction covers 512 contiguous bytes.
constexpr int kCopyUnroll = 4;

__host__ __device__ inline int64_t copy_groups(int64_t nv) { return (nv + 32 * kCopyUnroll - 1) / (32 * kCopyUnroll); }

__global__ void __launch_bounds__(256) permute_copy_kernel(const int32_t* __restrict__ inv_perm,
                                                           const uint4* __restrict__ x, int64_t T, int k,
                                                           int64_t A, int64_t nv, uint4* __restrict__ x_perm) {
  const int64_t G = copy_groups(nv);
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= T * G) return;
  const int64_t t = gw / G;
  const int64_t v0 = (gw % G) * 32 * kCopyUnroll + lane;
  uint4 val[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u)
    if (v0 + 32 * u < nv) val[u] = x[t * nv + v0 + 32 * u];
  for (int j = 0; j < k; ++j) {
    const int64_t row = inv_perm[t * k + j];
    if (row < 0 || row >= A) continue;
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (v0 + 32 * u < nv) x_perm[row * nv + v0 + 32 * u] = val[u];
  }
}

}  // namespace moe
