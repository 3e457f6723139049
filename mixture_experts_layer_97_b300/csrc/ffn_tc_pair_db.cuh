// ffn_tc_pair_db.cuh -- bf16 grouped GEMM with token tiles on SM pairs and a
// double-buffered accumulator (the GELU up projection and the plain down
// projection).
//
// The product of ffn_tc_swap.cuh and ffn_tc_pair.cuh ("MoE混合专家模型计算原理
// 与推理部署实战解析" sections 3.1-3.2; "MoE显存与计算开销四阶段手算指南"
// section 4.3): D[feature, token] = W[feature, :] . X[token, :]^T per expert,
// computed by clusters of two CTAs whose tensor cores run one MMA together
// (tcgen05 cta_group::2, M = 256: 128 weight rows in each CTA's shared memory)
// over a token tile of up to 256 rows (each CTA holding half of them).
//
// Unlike ffn_tc_pair.cuh, each CTA holds ONE 128-row weight block per tile,
// so a tile's accumulator is 128 lanes x at most 256 columns and TMEM (512
// columns) holds two of them: the MMA issuer starts the next tile in the
// other accumulator while the epilogue warps still drain this one, and the
// tensor pipe and the weight stream do not pause for the epilogue. Per K step
// a CTA stages 16 KB of weights and at most 16 KB of tokens: 32 KB stages,
// six of them.
//
// Features per pair tile: 256 (CTA r: weight rows [128 r, 128 r + 128) of
// the tile). Token tiles are those of the single-SM kernel (at most 256 rows,
// balanced per expert, multiples of 16); CTA r holds tokens
// [r nt / 2, (r + 1) nt / 2) of the tile.
//
// Roles (both CTAs): warp 0 TMA producer for the CTA's own shared memory,
// warp 1 TMEM (allocated by both CTAs together) and, in the even CTA only,
// the MMA issuer; warps 2-9 epilogue on the CTA's own TMEM. Barriers: the even
// CTA's full barriers count the bytes of both CTAs' copies; the issuer's
// commits arrive on the empty, accumulator-full and drain barriers of both
// CTAs; both CTAs' epilogue warps arrive on the even CTA's accumulator-empty
// barrier of the accumulator they drained. Every mbarrier wait is bounded;
// both CTAs meet at cluster barriers after set-up and before TMEM is freed.
#pragma once
#include "ffn_tc_pair.cuh"

namespace moe {

constexpr int kPdStages = 6;
constexpr int kPdRowBytes = kTcBK * 2;                       // 128-byte K rows
constexpr int kPdABytes = kSwFM * kPdRowBytes;              // the CTA's 128-row weight block: 16 KB
constexpr int kPdBRows = kSwMaxNT / 2;                      // token rows per CTA (max)
constexpr int kPdBBytes = kPdBRows * kPdRowBytes;           // 16 KB
constexpr int kPdStageBytes = kPdABytes + kPdBBytes;        // 32 KB
constexpr int kPdAccCols = kSwMaxNT;                        // one accumulator: 256 columns
constexpr int kPdTmemCols = 2 * kPdAccCols;
constexpr int kPdFeatures = 2 * kSwFM;                      // features per pair tile
constexpr int kPdNumBars = 2 * kPdStages + 5;               // full, empty, tfull[2], tempty[2], drain
constexpr size_t kPdSmemBytes = 1024 + static_cast<size_t>(kPdStages) * kPdStageBytes + kSwXposeBytes +
                                8 * kPdNumBars + 16 + 2 * 257 * sizeof(int) + 16;
static_assert(kPdSmemBytes <= 227 * 1024, "double-buffered pair kernel shared memory");

template <int EPI>
__global__ void __launch_bounds__(kSwThreads, 1)
    grouped_gemm_tc_pair_db_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                                   const int32_t* __restrict__ offsets, int N, int rows_total, int K, int Nout,
                                   __nv_bfloat16* __restrict__ out, int ldo, unsigned long long timeout_ns) {
  static_assert(EPI == EPI_GELU || EPI == EPI_PLAIN, "one weight block per CTA: GELU or plain epilogue");
  constexpr int S = kPdStages;
  constexpr int OFP = kPdFeatures;
  // M = 256 (128 rows in each CTA); the N field is filled per tile
  constexpr uint32_t IDESC0 = idesc_bf16_f32(2 * kSwFM, 16) & ~(0x3Fu << 17);

  extern __shared__ uint8_t pd_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pd_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_a = smem;                        // S x this CTA's weight block
  uint8_t* stage_b = smem + S * kPdABytes;        // S x this CTA's token half
  uint8_t* xpose = smem + S * kPdStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(xpose + kSwXposeBytes);
  uint64_t* full_bar = bars;                      // used in the even CTA only
  uint64_t* empty_bar = bars + S;
  uint64_t* tfull_bar = bars + 2 * S;             // [2]
  uint64_t* tempty_bar = tfull_bar + 2;           // [2], used in the even CTA only
  uint64_t* drain_bar = tfull_bar + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kPdNumBars);
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
      mbar_init(smem_addr(&tempty_bar[b]), 2 * kSwEpiWarps);
    }
    mbar_init(smem_addr(drain_bar), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    build_tile_prefix(offsets, N, rows_total, kSwMaxNT, s_off, s_pre, bad_flag);
    if (lane == 0) {
      prefetch_tensormap(&tmW);
      prefetch_tensormap(&tmX);
    }
  }
  // both CTAs' barriers are initialised before either signals the other's
  cluster_sync_all();
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), kPdTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const bool bad = *bad_flag != 0;
  if (bad && threadIdx.x == 0 && blockIdx.x == 0) record_error(MOE_ERR_CORRUPT);
  const int n_ftiles = (Nout + OFP - 1) / OFP;
  const long long total = bad ? 0 : static_cast<long long>(s_pre[N]) * n_ftiles;
  const int KB = K / kTcBK;
  const long long pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (each CTA fills its own shared memory)
    int s = 0;
    uint32_t ph = 0;
    long long issued = 0;
    bool ok = true;
    for (long long id = pair; id < total && ok; id += npairs) {
      const SwTile t = sw_decode(id, s_off, s_pre, N, n_ftiles);
      const int wrow = t.e * Nout + t.fi * OFP + static_cast<int>(rank) * kSwFM;
      const int half = t.nt >> 1;                               // token rows per CTA
      const int r0 = t.row0 + static_cast<int>(rank) * half;
      const int nbox = (half + kSwBox - 1) / kSwBox;
      const uint32_t tx_pair = 2u * (kPdABytes + nbox * kSwBox * kPdRowBytes);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_bounded(smem_addr(&empty_bar[s]), ph ^ 1u, abort_flag, timeout_ns)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_addr_in_cta(smem_addr(&full_bar[s]), 0);
        if (leader) mbar_arrive_expect_tx(smem_addr(&full_bar[s]), tx_pair);
        const uint32_t sa = smem_addr(stage_a + s * kPdABytes);
        const uint32_t sb = smem_addr(stage_b + s * kPdBBytes);
        tma_load_2d_pair(sa, &tmW, fb, kb * kTcBK, wrow);
        for (int b = 0; b < nbox; ++b)
          tma_load_2d_pair(sb + b * kSwBox * kPdRowBytes, &tmX, fb, kb * kTcBK, r0 + b * kSwBox);
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
      // ---------------- MMA issuer for the pair, tiles alternating between the two accumulators
      int s = 0;
      uint32_t ph = 0;
      uint32_t it = 0;
      bool ok = true;
      for (long long id = pair; id < total && ok; id += npairs, ++it) {
        const SwTile t = sw_decode(id, s_off, s_pre, N, n_ftiles);
        const uint32_t idesc = IDESC0 | (static_cast<uint32_t>(t.nt >> 3) << 17);
        const uint32_t b = it & 1u;
        // the accumulator's previous tile (two tiles back) has been drained
        if (!mbar_wait_bounded(smem_addr(&tempty_bar[b]), ((it >> 1) & 1u) ^ 1u, abort_flag, timeout_ns)) break;
        tc_fence_after();
        const uint32_t acc_tmem = tmem_base + b * kPdAccCols;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_addr(&full_bar[s]), ph, abort_flag, timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = kmajor_swizzled_desc<kPdRowBytes>(smem_addr(stage_a + s * kPdABytes));
          const uint64_t bd = kmajor_swizzled_desc<kPdRowBytes>(smem_addr(stage_b + s * kPdBBytes));
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk)
            umma_bf16_pair(acc_tmem, ad + 2u * kk, bd + 2u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          umma_commit_pair(smem_addr(&empty_bar[s]));
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair(smem_addr(&tfull_bar[b]));
      }
      // every MMA issued has completed before either CTA frees TMEM
      umma_commit_pair(smem_addr(drain_bar));
    }
    mbar_wait_bounded(smem_addr(drain_bar), 0u, nullptr, timeout_ns);
  } else if (warp >= 2) {
    // ---------------- epilogue on this CTA's TMEM: its 128 weight rows x all tokens of the tile
    const int q = warp & 3;
    const int hsel = (warp - 2) >> 2;
    uint8_t* xp = xpose + (warp - 2) * (32 * 64);
    const uint32_t xp_s = smem_addr(xp);
    uint32_t it = 0;
    for (long long id = pair; id < total; id += npairs, ++it) {
      const SwTile t = sw_decode(id, s_off, s_pre, N, n_ftiles);
      const uint32_t b = it & 1u;
      if (!mbar_wait_bounded(smem_addr(&tfull_bar[b]), (it >> 1) & 1u, abort_flag, timeout_ns)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + b * kPdAccCols + (static_cast<uint32_t>(q * 32) << 16);
      const int f0 = t.fi * OFP + static_cast<int>(rank) * kSwFM + q * 32;   // feature of lane 0
#pragma unroll 1
      for (int c = 32 * hsel; c < t.nt; c += 64) {
        uint32_t v[32];
        tmem_ld_32x32(tb + c, v);
        tmem_ld_wait();
        if (EPI == EPI_GELU) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float a = __uint_as_float(v[i]);
            v[i] = __float_as_uint(0.5f * a * (1.f + tanh_fast(0.7978845608028654f * (a + 0.044715f * a * a * a))));
          }
        }
        if (f0 < Nout) sw_store_transposed(v, xp, xp_s, lane, c, t.rows, t.row0, f0, out, ldo);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(smem_addr_in_cta(smem_addr(&tempty_bar[b]), 0));
    }
  }

  __syncthreads();
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kPdTmemCols);
}

}  // namespace moe
