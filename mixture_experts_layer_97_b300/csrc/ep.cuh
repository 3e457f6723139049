// ep.cuh -- the two local steps of expert parallelism around the all-to-all
// exchange of token rows.
//
// "MoE混合专家模型计算原理与推理部署实战解析" section 3.3: with the experts
// split over G GPUs by expert id (for example 8 experts over 4 cards, 2 per
// card), every card routes its own tokens and sends each token row to the card
// that holds the chosen expert through an all-to-all; section 6.3 names this
// expert parallelism (EP). Here the experts are contiguous id ranges, so the
// grouping step's x_perm (rows ordered by expert) is already ordered by
// destination card and is the send buffer as it stands.
//
// What a card receives is ordered by (source card g, local expert e, the
// source's row order). The grouped GEMM needs its rows grouped by local
// expert, so:
//   regroup   local row order (e, g, i): offsets_local[e] = rows of the local
//             experts before e; local_src[row] = the received row it takes
//             (recv base of g + rows of g for the local experts before e + i);
//             x_local[row] = recv_x[local_src[row]]
//   ungroup   y_recv[local_src[row]] = y_local[row], back to the received
//             order, which the reverse all-to-all returns to the sources in
//             the order they sent (their x_perm order, so their combine runs
//             unchanged).
// The count table recv_counts[g][e] (G x E int32, G * E <= 256 entries) is
// what the counts exchange delivers. Integer work only: bit-exact.
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kEpThreads = 256;
constexpr int kEpMaxTable = 256;

// Shared tables of one CTA, built from recv_counts:
//   eoff[e]        first local row of local expert e (eoff[E] = total rows)
//   gbase[g]       first received row from source g
//   gpre[g * E + e] rows of source g for the local experts before e
//   epre[e * G + g] rows of local expert e from the sources before g
struct EpTables {
  int eoff[kEpMaxTable + 1];
  int gbase[kEpMaxTable + 1];
  int gpre[kEpMaxTable];
  int epre[kEpMaxTable];
  int bad;
};

__device__ inline void ep_build_tables(const int32_t* __restrict__ recv_counts, int G, int E, int64_t rows,
                                       EpTables& tb) {
  if (threadIdx.x == 0) {
    int bad = 0;
    long long run = 0;
    for (int g = 0; g < G; ++g) {
      tb.gbase[g] = static_cast<int>(run);
      long long r = 0;
      for (int e = 0; e < E; ++e) {
        const int c = recv_counts[g * E + e];
        if (c < 0) bad = 1;
        tb.gpre[g * E + e] = static_cast<int>(r);
        r += c > 0 ? c : 0;
      }
      run += r;
    }
    tb.gbase[G] = static_cast<int>(run);
    long long l = 0;
    for (int e = 0; e < E; ++e) {
      tb.eoff[e] = static_cast<int>(l);
      long long r = 0;
      for (int g = 0; g < G; ++g) {
        tb.epre[e * G + g] = static_cast<int>(r);
        const int c = recv_counts[g * E + e];
        r += c > 0 ? c : 0;
      }
      l += r;
    }
    tb.eoff[E] = static_cast<int>(l);
    if (run != rows) bad = 1;       // the table must account for exactly the received rows
    tb.bad = bad;
  }
  __syncthreads();
}

// One warp per local row: find (e, g, i), write local_src, copy the row with
// 128-bit accesses. Block 0 also writes offsets_local.
__global__ void __launch_bounds__(kEpThreads) ep_regroup_kernel(const int32_t* __restrict__ recv_counts, int G,
                                                                int E, int64_t rows, int64_t nv,
                                                                const uint4* __restrict__ recv_x,
                                                                uint4* __restrict__ x_local,
                                                                int32_t* __restrict__ offsets_local,
                                                                int32_t* __restrict__ local_src) {
  __shared__ EpTables tb;
  ep_build_tables(recv_counts, G, E, rows, tb);
  if (tb.bad) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(MOE_ERR_CORRUPT);
    return;
  }
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets_local[e] = tb.eoff[e];
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kEpThreads / 32);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (kEpThreads / 32) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    // local expert: the last e with eoff[e] <= row (empty experts are skipped)
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tb.eoff[mid] <= row) lo = mid;
      else hi = mid;
    }
    const int e = lo;
    const int p = static_cast<int>(row - tb.eoff[e]);        // position within the expert's rows
    // source: the last g with epre[e * G + g] <= p
    int glo = 0, ghi = G;
    while (ghi - glo > 1) {
      const int mid = (glo + ghi) >> 1;
      if (tb.epre[e * G + mid] <= p) glo = mid;
      else ghi = mid;
    }
    const int g = glo;
    const int64_t src = static_cast<int64_t>(tb.gbase[g]) + tb.gpre[g * E + e] + (p - tb.epre[e * G + g]);
    if (lane == 0) local_src[row] = static_cast<int32_t>(src);
    const uint4* s = recv_x + src * nv;
    uint4* dst = x_local + row * nv;
    for (int64_t v = lane; v < nv; v += 32) dst[v] = s[v];
  }
}

// y_recv[local_src[row]] = y_local[row], one warp per row.
__global__ void __launch_bounds__(kEpThreads) ep_ungroup_kernel(const int32_t* __restrict__ local_src, int64_t rows,
                                                                int64_t nv, const uint4* __restrict__ y_local,
                                                                uint4* __restrict__ y_recv) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kEpThreads / 32);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (kEpThreads / 32) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const int64_t dst = local_src[row];
    if (dst < 0 || dst >= rows) {
      if (lane == 0) record_error(MOE_ERR_CORRUPT);
      continue;
    }
    const uint4* s = y_local + row * nv;
    uint4* d = y_recv + dst * nv;
    for (int64_t v = lane; v < nv; v += 32) d[v] = s[v];
  }
}

}  // namespace moe
