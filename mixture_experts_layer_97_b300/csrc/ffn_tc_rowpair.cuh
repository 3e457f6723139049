// ffn_tc_rowpair.cuh -- bf16 grouped GEMM with row tiles on SM pairs.
//
// The product of ffn_tc.cuh ("MoE混合专家模型计算原理与推理部署实战解析"
// sections 3.1-3.2; "MoE显存与计算开销四阶段手算指南" section 4.3: one
// launch over every active expert with expert offsets), computed by clusters
// of two CTAs whose tensor cores run one MMA together (tcgen05 cta_group::2):
// D[256 permuted rows, 256 weight rows], each CTA holding 128 of the rows
// (the MMA's A side) and 128 of the weight rows (half of its B side) in its
// shared memory. Against the single-SM row tiles (128 rows x 256 weight
// rows) every weight tile serves twice the rows, so an expert with many
// rows re-reads its weights from L2 half as often, and each CTA stages 32 KB
// per K step instead of 48 KB.
//
// Output columns per pair tile: SwiGLU 128 hidden units (CTA 0 loads their
// gate rows, CTA 1 their up rows: D columns 0-127 are gate, 128-255 up, and
// each CTA's epilogue forms silu(gate) * up for its 128 rows); GELU and the
// down projection 256 output features (CTA r loads rows [128 r, 128 r + 128)).
//
// Roles (both CTAs): warp 0 TMA producer for the CTA's own shared memory,
// warp 1 TMEM (allocated by both CTAs together, two 256-column accumulators
// so the epilogue of one tile overlaps the main loop of the next) and, in the
// even CTA only, the MMA issuer; warps 2-5 epilogue on the CTA's own TMEM
// (its 128 rows x 256 columns), rows written in place with 16-byte stores.
// Barriers as in ffn_tc_pair.cuh: the even CTA's full barriers count both
// CTAs' bytes, the issuer's commits arrive on both CTAs' empty,
// accumulator-full and drain barriers, both CTAs' epilogue warps arrive on
// the even CTA's accumulator-empty barriers. Tiles (expert, column tile,
// row tile) go round robin over the pairs. Every mbarrier wait is bounded;
// both CTAs meet at cluster barriers after set-up and before TMEM is freed.
#pragma once
#include "ffn_tc_pair.cuh"

namespace moe {

constexpr int kRpBM = 256;                                  // permuted rows per pair tile
constexpr int kRpHalf = 128;                                // rows (and weight rows) per CTA
constexpr int kRpBN = 256;                                  // MMA N: weight rows per pair tile
constexpr int kRpStages = 6;
constexpr int kRpABytes = kRpHalf * kTcBK * 2;              // 16 KB of rows
constexpr int kRpBBytes = kRpHalf * kTcBK * 2;              // 16 KB of weight rows
constexpr int kRpStageBytes = kRpABytes + kRpBBytes;        // 32 KB
constexpr int kRpThreads = 192;
constexpr int kRpTmemCols = 2 * kRpBN;                      // two accumulators
constexpr int kRpNumBars = 2 * kRpStages + 5;               // full, empty, tfull[2], tempty[2], drain
constexpr size_t kRpSmemBytes = 1024 + static_cast<size_t>(kRpStages) * kRpStageBytes + 8 * kRpNumBars + 16 +
                                2 * 257 * sizeof(int) + 16;
static_assert(kRpSmemBytes <= 227 * 1024, "row-pair kernel shared memory");

// Output columns of one pair tile.
template <int EPI>
__host__ __device__ constexpr int rp_tile_cols() { return EPI == EPI_SWIGLU ? kRpBN / 2 : kRpBN; }

template <int EPI>
__global__ void __launch_bounds__(kRpThreads, 1)
    grouped_gemm_tc_rowpair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                                   const __grid_constant__ CUtensorMap tmB1, const int32_t* __restrict__ offsets,
                                   int N, int rows_total, int K, int Nout, __nv_bfloat16* __restrict__ out, int ldo,
                                   unsigned long long timeout_ns) {
  constexpr int S = kRpStages;
  constexpr int HB = rp_tile_cols<EPI>();
  constexpr uint32_t IDESC = idesc_bf16_f32(kRpBM, kRpBN);

  extern __shared__ uint8_t rp_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rp_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_a = smem;                        // S x this CTA's 128 rows
  uint8_t* stage_b = smem + S * kRpABytes;        // S x this CTA's 128 weight rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * kRpStageBytes);
  uint64_t* full_bar = bars;                      // used in the even CTA only
  uint64_t* empty_bar = bars + S;
  uint64_t* tfull_bar = bars + 2 * S;             // [2]
  uint64_t* tempty_bar = bars + 2 * S + 2;        // [2], used in the even CTA only
  uint64_t* drain_bar = bars + 2 * S + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kRpNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* bad_flag = reinterpret_cast<int*>(tmem_slot + 2);
  int* s_off = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_pre = s_off + 257;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&tfull_bar[b]), 1);
      mbar_init(smem_addr(&tempty_bar[b]), 2 * 4);   // four epilogue warps in each CTA
    }
    mbar_init(smem_addr(drain_bar), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    build_tile_prefix(offsets, N, rows_total, kRpBM, s_off, s_pre, bad_flag);
    if (lane == 0) {
      prefetch_tensormap(&tmA);
      prefetch_tensormap(&tmB0);
      if (EPI == EPI_SWIGLU) prefetch_tensormap(&tmB1);
    }
  }
  // both CTAs' barriers are initialised before either signals the other's
  cluster_sync_all();
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), kRpTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const bool bad = *bad_flag != 0;
  if (bad && threadIdx.x == 0 && blockIdx.x == 0) record_error(MOE_ERR_CORRUPT);
  const int n_tiles = Nout / HB;
  const long long total = bad ? 0 : static_cast<long long>(s_pre[N]) * n_tiles;
  const int KB = K / kTcBK;
  const long long cid = blockIdx.x >> 1;          // this pair
  const long long ncl = gridDim.x >> 1;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer: this CTA's 128 rows and 128 weight rows per stage
    int s = 0;
    uint32_t ph = 0;
    long long issued = 0;
    bool ok = true;
    const CUtensorMap* mb = (EPI == EPI_SWIGLU && rank == 1) ? &tmB1 : &tmB0;
    for (long long id = cid; id < total && ok; id += ncl) {
      const TileInfo ti = decode_tile(id, s_off, s_pre, N, n_tiles, kRpBM);
      const int arow = ti.row0 + static_cast<int>(rank) * kRpHalf;
      // SwiGLU: gate rows (CTA 0) or up rows (CTA 1) of the tile's hidden units; else this CTA's half
      const int brow = ti.e * Nout + ti.nt * HB + (EPI == EPI_SWIGLU ? 0 : static_cast<int>(rank) * kRpHalf);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_bounded(smem_addr(&empty_bar[s]), ph ^ 1u, abort_flag, timeout_ns)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_addr_in_cta(smem_addr(&full_bar[s]), 0);
        if (leader) mbar_arrive_expect_tx(smem_addr(&full_bar[s]), 2u * kRpStageBytes);
        tma_load_2d_pair(smem_addr(stage_a + s * kRpABytes), &tmA, fb, kb * kTcBK, arow);
        tma_load_2d_pair(smem_addr(stage_b + s * kRpBBytes), mb, fb, kb * kTcBK, brow);
        ++issued;
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
    if (!ok && leader) {
      // let the copies still in flight (both CTAs') land before the CTAs leave
      const long long first = issued > S ? issued - S : 0;
      for (long long i = first; i < issued; ++i)
        mbar_wait_bounded(smem_addr(&full_bar[i % S]), static_cast<uint32_t>((i / S) & 1), nullptr, timeout_ns);
    }
  } else if (warp == 1 && lane == 0) {
    if (leader) {
      // ---------------- MMA issuer for the pair
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      bool ok = true;
      for (long long id = cid; id < total && ok; id += ncl) {
        if (!mbar_wait_bounded(smem_addr(&tempty_bar[acc]), aph ^ 1u, abort_flag, timeout_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kRpBN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_addr(&full_bar[s]), ph, abort_flag, timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = kmajor_swizzled_desc<kPrRowBytes>(smem_addr(stage_a + s * kRpABytes));
          const uint64_t bd = kmajor_swizzled_desc<kPrRowBytes>(smem_addr(stage_b + s * kRpBBytes));
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk)
            umma_bf16_pair(d_tmem, ad + 2u * kk, bd + 2u * kk, IDESC, (kb | kk) != 0 ? 1u : 0u);
          umma_commit_pair(smem_addr(&empty_bar[s]));
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair(smem_addr(&tfull_bar[acc]));
        acc ^= 1;
        if (acc == 0) aph ^= 1u;
      }
      // every MMA issued has completed before either CTA frees TMEM
      umma_commit_pair(smem_addr(drain_bar));
    }
    mbar_wait_bounded(smem_addr(drain_bar), 0u, nullptr, timeout_ns);
  } else if (warp >= 2) {
    // ---------------- epilogue on this CTA's TMEM: its 128 rows x 256 columns
    const int q = warp & 3;   // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t aph = 0;
    for (long long id = cid; id < total; id += ncl) {
      const TileInfo ti = decode_tile(id, s_off, s_pre, N, n_tiles, kRpBM);
      if (!mbar_wait_bounded(smem_addr(&tfull_bar[acc]), aph, abort_flag, timeout_ns)) break;
      tc_fence_after();
      const int r = static_cast<int>(rank) * kRpHalf + q * 32 + lane;   // row within the pair tile
      const bool valid = r < ti.rows;
      const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * kRpBN) + (static_cast<uint32_t>(q * 32) << 16);
      __nv_bfloat16* orow = out + static_cast<int64_t>(ti.row0 + r) * ldo + static_cast<int64_t>(ti.nt) * HB;
#pragma unroll 1
      for (int c = 0; c < HB; c += 32) {
        uint32_t v[32];
        uint32_t packed[16];
        tmem_ld_32x32(tb + c, v);
        if (EPI == EPI_SWIGLU) {
          uint32_t u[32];
          tmem_ld_32x32(tb + HB + c, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(v[2 * i]), g1 = __uint_as_float(v[2 * i + 1]);
            const float h0 = __fdividef(g0, 1.f + __expf(-g0)) * __uint_as_float(u[2 * i]);
            const float h1 = __fdividef(g1, 1.f + __expf(-g1)) * __uint_as_float(u[2 * i + 1]);
            packed[i] = pack_bf16x2(h0, h1);
          }
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float a0 = __uint_as_float(v[2 * i]), a1 = __uint_as_float(v[2 * i + 1]);
            if (EPI == EPI_GELU) {
              a0 = 0.5f * a0 * (1.f + tanh_fast(0.7978845608028654f * (a0 + 0.044715f * a0 * a0 * a0)));
              a1 = 0.5f * a1 * (1.f + tanh_fast(0.7978845608028654f * (a1 + 0.044715f * a1 * a1 * a1)));
            }
            packed[i] = pack_bf16x2(a0, a1);
          }
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(smem_addr_in_cta(smem_addr(&tempty_bar[acc]), 0));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }

  __syncthreads();
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kRpTmemCols);
}

}  // namespace moe
