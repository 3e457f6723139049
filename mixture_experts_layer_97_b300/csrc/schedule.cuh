// schedule.cuh -- device-side tile schedule of the grouped GEMMs.
//
// The pages' grouped GEMM takes the concatenated expert inputs and an
// expert_offsets array ("MoE显存与计算开销四阶段手算指南" section 4.3). Every CTA
// rebuilds, from offsets[N+1] alone, the prefix of BM-row tiles over experts,
// so no host synchronisation or extra launch is needed between the permute
// and the GEMM. Tile id order is (expert, n-tile, m-tile) with m fastest:
// CTAs that run at the same time share one weight tile through L2.
#pragma once
#include "common.cuh"

namespace moe {

// Called by all 32 lanes of one warp. Fills s_off[0..N] (a copy of offsets)
// and s_pre[0..N] (prefix of ceil(rows / BM) over experts); *s_bad = 1 when
// offsets are not a monotone partition of a prefix [0, offsets[N]) of the
// rows_total rows (offsets[N] < rows_total when an expert capacity dropped
// assignments).
__device__ inline void build_tile_prefix(const int32_t* __restrict__ offsets, int N, int rows_total, int BM,
                                         int* s_off, int* s_pre, int* s_bad) {
  const int lane = threadIdx.x & 31;
  const int per = (N + 31) / 32;
  const int e0 = min(N, lane * per), e1 = min(N, e0 + per);
  bool bad = false;
  int sum = 0;
  for (int e = e0; e < e1; ++e) {
    const int a = offsets[e], b = offsets[e + 1];
    s_off[e] = a;
    if (a < 0 || b < a || b > rows_total) bad = true;
    else sum += (b - a + BM - 1) / BM;
  }
  if (lane == 0) {
    const int a0 = offsets[0], aN = offsets[N];
    s_off[N] = aN;
    if (a0 != 0 || aN > rows_total) bad = true;
  }
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  int run = incl - sum;
  for (int e = e0; e < e1; ++e) {
    s_pre[e] = run;
    const int a = offsets[e], b = offsets[e + 1];
    if (!(a < 0 || b < a || b > rows_total)) run += (b - a + BM - 1) / BM;
  }
  if (lane == 31) s_pre[N] = incl;
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) *s_bad = bad ? 1 : 0;
}

struct TileInfo {
  int e;      // expert
  int nt;     // output column tile
  int row0;   // first permuted row of the tile
  int rows;   // valid rows in the tile (1..BM)
};

__device__ __forceinline__ TileInfo decode_tile(long long id, const int* s_off, const int* s_pre, int N,
                                                int n_tiles, int BM) {
  int lo = 0, hi = N;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<long long>(s_pre[mid]) * n_tiles <= id) lo = mid;
    else hi = mid;
  }
  const int mte = s_pre[lo + 1] - s_pre[lo];
  const long long local = id - static_cast<long long>(s_pre[lo]) * n_tiles;
  TileInfo ti;
  ti.e = lo;
  ti.nt = static_cast<int>(local / mte);
  const int mt = static_cast<int>(local % mte);
  ti.row0 = s_off[lo] + mt * BM;
  ti.rows = min(BM, s_off[lo + 1] - ti.row0);
  return ti;
}

}  // namespace moe
