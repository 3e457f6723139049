// permute.cuh -- K2: group the T*k token-expert assignments by expert.
//
// "MoE显存与计算开销四阶段手算指南" section 2.3 and
// "MoE混合专家模型计算原理与推理部署实战解析" section 5.1 steps 2-3:
// count per expert, exclusive prefix sum into offsets, then move every
// assignment's input row into one contiguous buffer ordered by expert.
//
// A deterministic stable counting sort by flat index f = t*k + j. A batch of
// at most one chunk (T*k <= 2048, e.g. decode) takes one launch
// (permute_single_kernel); otherwise four:
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

// One warp's share of the row copy: token t, chunk group gi; row_of(j) gives
// the permuted row of assignment (t, j) (negative or >= A: not copied).
template <typename RowOf>
__device__ __forceinline__ void copy_token_slice(const uint4* __restrict__ x, uint4* __restrict__ x_perm, int64_t t,
                                                 int64_t gi, int k, int64_t A, int64_t nv, int lane, RowOf row_of) {
  const int64_t v0 = gi * 32 * kCopyUnroll + lane;
  uint4 val[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u)
    if (v0 + 32 * u < nv) val[u] = x[t * nv + v0 + 32 * u];
  for (int j = 0; j < k; ++j) {
    const int64_t row = row_of(j);
    if (row < 0 || row >= A) continue;
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (v0 + 32 * u < nv) x_perm[row * nv + v0 + 32 * u] = val[u];
  }
}

// A grouping that fits one chunk (T*k <= 2048 assignments, e.g. a decode
// batch) in one launch instead of four: every CTA computes the per-warp
// histograms of the rank pass, the counts / capacity / offsets of the scan
// pass and the stable ranks (a few thousand assignments at most, so the
// repeated work is cheaper than more launches); CTA 0 writes counts, offsets,
// perm, inv_perm and *dropped, and all CTAs share the row copy (x_perm ==
// nullptr: no copy, one CTA). Same results bit for bit as hist + scan + rank
// + copy; an expert index outside [0, N) records MOE_ERR_CORRUPT (the
// assignment belongs to no expert).
__global__ void __launch_bounds__(kPermThreads) permute_single_kernel(const int32_t* __restrict__ topk_idx, int64_t T,
                                                                      int N, int k, long long capacity,
                                                                      int32_t* __restrict__ counts,
                                                                      int32_t* __restrict__ offsets,
                                                                      int32_t* __restrict__ perm,
                                                                      int32_t* __restrict__ inv_perm,
                                                                      int32_t* __restrict__ dropped,
                                                                      const uint4* __restrict__ x, int64_t nv,
                                                                      uint4* __restrict__ x_perm) {
  __shared__ int wh[kPermWarps][256];
  __shared__ int s_off[256];
  __shared__ int s_idx[kPermMaxChunk];     // the expert indices, then the permuted row of each assignment
  __shared__ int warp_sums[kPermWarps];
  const bool writer = blockIdx.x == 0;
  const int nf = static_cast<int>(T * k);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  // this CTA's first share of the row copy is loaded now: its latency overlaps the ranking below
  const int64_t G = copy_groups(nv);
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kPermWarps;
  const int64_t gw0 = static_cast<int64_t>(blockIdx.x) * kPermWarps + warp;
  uint4 first[kCopyUnroll];
  if (x_perm != nullptr && gw0 < T * G) {
    const int64_t v0 = (gw0 % G) * 32 * kCopyUnroll + lane;
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (v0 + 32 * u < nv) first[u] = x[(gw0 / G) * nv + v0 + 32 * u];
  }
  for (int i = threadIdx.x; i < kPermWarps * 256; i += blockDim.x) (&wh[0][0])[i] = 0;
  for (int f = threadIdx.x; f < nf; f += blockDim.x) {
    int e = topk_idx[f];
    if (e < 0 || e >= N) {
      if (writer) record_error(MOE_ERR_CORRUPT);
      e = -1;                              // belongs to no expert
    }
    s_idx[f] = e;
  }
  __syncthreads();
  const int s0 = warp * kPermSub;
  const int s1 = min(nf, s0 + kPermSub);
  // per-warp histograms over contiguous sub-ranges
  for (int g = s0; g < s1; g += 32) {
    const int fl = g + lane;
    const int e = (fl < s1) ? s_idx[fl] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (peers & lt_mask) == 0) wh[warp][e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // per expert: prefix over warps, the kept count, then the exclusive scan over experts
  const int n = threadIdx.x;
  int run = 0;
  if (n < N) {
#pragma unroll
    for (int w = 0; w < kPermWarps; ++w) {
      const int v = wh[w][n];
      wh[w][n] = run;
      run += v;
    }
  }
  const int kept = n < N ? static_cast<int>(run < capacity ? run : capacity) : 0;
  int incl = kept;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int i = 0; i < warp; ++i) wbase += warp_sums[i];
  if (n < N) {
    s_off[n] = wbase + incl - kept;
    if (writer) {
      counts[n] = kept;
      offsets[n] = wbase + incl - kept;
    }
  }
  if (writer && n == kPermThreads - 1) offsets[N] = wbase + incl;
  __syncthreads();
  // stable ranks in flat order (each warp its own sub-range, so s_idx can take the rows in place);
  // rank >= capacity is dropped
  int n_drop = 0;
  for (int g = s0; g < s1; g += 32) {
    const int fl = g + lane;
    const int e = (fl < s1) ? s_idx[fl] : -1;
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
          row = s_off[e] + rank;
          if (writer) perm[row] = fl / k;
        } else {
          row = kDroppedRow;
          ++n_drop;
        }
      }
      s_idx[fl] = row;
      if (writer) inv_perm[fl] = row;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) n_drop += __shfl_xor_sync(0xffffffffu, n_drop, off);
  __syncthreads();                         // every row known; warp_sums free again
  if (lane == 0) warp_sums[warp] = n_drop;
  __syncthreads();
  if (writer && dropped != nullptr && threadIdx.x == 0) {
    int tot = 0;
    for (int w = 0; w < kPermWarps; ++w) tot += warp_sums[w];
    *dropped = tot;
  }
  if (x_perm == nullptr) return;
  // the row copy, shared by all CTAs: warp gw owns (token gw / G, chunk group gw % G)
  for (int64_t gw = gw0; gw < T * G; gw += nw) {
    const int64_t t = gw / G;
    const int64_t v0 = (gw % G) * 32 * kCopyUnroll + lane;
    uint4 val[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (v0 + 32 * u < nv) val[u] = gw == gw0 ? first[u] : x[t * nv + v0 + 32 * u];
    for (int j = 0; j < k; ++j) {
      const int row = s_idx[t * k + j];
      if (row < 0 || row >= nf) continue;
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u)
        if (v0 + 32 * u < nv) x_perm[row * nv + v0 + 32 * u] = val[u];
    }
  }
}

__global__ void __launch_bounds__(256) permute_copy_kernel(const int32_t* __restrict__ inv_perm,
                                                           const uint4* __restrict__ x, int64_t T, int k,
                                                           int64_t A, int64_t nv, uint4* __restrict__ x_perm) {
  const int64_t G = copy_groups(nv);
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= T * G) return;
  const int64_t t = gw / G;
  copy_token_slice(x, x_perm, t, gw % G, k, A, nv, lane, [&](int j) { return static_cast<int64_t>(inv_perm[t * k + j]); });
}

}  // namespace moe
