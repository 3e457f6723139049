// ffn_tc.cuh -- bf16 grouped GEMM on the 5th-generation tensor cores.
//
// The pages' grouped GEMM ("MoE显存与计算开销四阶段手算指南" section 4.3: one
// launch over every active expert, contiguous inputs, expert offsets;
// "MoE混合专家模型计算原理与推理部署实战解析" sections 3.1-3.2, 5.1 step 4) as a
// persistent, warp-specialised sm_103a kernel:
//
//   warp 0     TMA producer: A tile (128 permuted rows x 64 K) and B tile
//              (BN weight rows x 64 K) per stage, 128-byte swizzle, into an
//              S-stage shared-memory ring guarded by full/empty mbarriers.
//              With GATHER the A rows come straight from the unpermuted
//              tokens x through the permutation (perm[row] = token): each
//              lane of the warp gathers four of the tile's rows per stage
//              (TMA tile::gather4), so no permuted copy of x is needed
//   warp 1     allocates 2*BN TMEM columns (two fp32 accumulators), one
//              thread issues tcgen05.mma (M=128, N=BN, K=16, bf16 -> fp32)
//              and commits stages back to the producer
//   warps 2-5  epilogue: tcgen05.ld the accumulator, apply the activation
//              (SwiGLU: the tile holds gate columns then up columns of the
//              same hidden range; GELU; or none), round to bf16, store rows
//              that belong to the tile's expert
//
// Two accumulators let the epilogue of one tile overlap the main loop of the
// next. Tiles are (expert, n-tile, m-tile) in that nesting; CTAs take them
// round-robin. Every wait is bounded: on timeout the CTA records
// MOE_ERR_TIMEOUT, lets its copies and MMAs in flight land, frees TMEM and
// returns.
#pragma once
#include "ffn_simt.cuh"
#include "schedule.cuh"

namespace moe {

constexpr int kTcBM = 128;
constexpr int kTcBK = 64;   // one 128-byte swizzle row of bf16
constexpr int kTcThreads = 192;

template <int BN>
struct TcCfg {
  static constexpr int kABytes = kTcBM * kTcBK * 2;
  static constexpr int kBBytes = BN * kTcBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStagesRaw = (196 * 1024) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kBarBytes = 8 * (2 * kStages + 5);
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + kBarBytes + 16 +
                                       2 * 257 * sizeof(int) + 16;
};

template <int BN, int EPI, bool GATHER = false>
__global__ void __launch_bounds__(kTcThreads, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1, const int32_t* __restrict__ offsets, int N,
                           int rows_total, int K, int Nout, __nv_bfloat16* __restrict__ out, int ldo,
                           unsigned long long timeout_ns, const int32_t* __restrict__ perm) {
  using C = TcCfg<BN>;
  constexpr int S = C::kStages;
  constexpr int HB = (EPI == EPI_SWIGLU) ? BN / 2 : BN;  // weight rows per TMA box = output columns
  constexpr uint32_t IDESC = idesc_bf16_f32(kTcBM, BN);

  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_a = smem;
  uint8_t* stage_b = smem + S * C::kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::kStageBytes);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + S;
  uint64_t* tfull_bar = bars + 2 * S;
  uint64_t* tempty_bar = bars + 2 * S + 2;
  uint64_t* drain_bar = bars + 2 * S + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* bad_flag = reinterpret_cast<int*>(tmem_slot + 2);
  int* s_off = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_pre = s_off + 257;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&tfull_bar[b]), 1);
      mbar_init(smem_addr(&tempty_bar[b]), 4);
    }
    mbar_init(smem_addr(drain_bar), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    build_tile_prefix(offsets, N, rows_total, kTcBM, s_off, s_pre, bad_flag);
    if (lane == 0) {
      prefetch_tensormap(&tmA);
      prefetch_tensormap(&tmB0);
      if (EPI == EPI_SWIGLU) prefetch_tensormap(&tmB1);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const bool bad = *bad_flag != 0;
  if (bad && threadIdx.x == 0 && blockIdx.x == 0) record_error(MOE_ERR_CORRUPT);
  const int n_tiles = Nout / HB;
  const long long total = bad ? 0 : static_cast<long long>(s_pre[N]) * n_tiles;
  const int KB = K / kTcBK;

  if (warp == 0 && (GATHER || lane == 0)) {
    // ---------------- TMA producer (lane 0 waits and loads the weights; with GATHER every lane
    // also gathers four rows of the A tile)
    int s = 0;
    uint32_t ph = 0;
    long long issued = 0;
    bool ok = true;
    for (long long id = blockIdx.x; id < total && ok; id += gridDim.x) {
      const TileInfo ti = decode_tile(id, s_off, s_pre, N, n_tiles, kTcBM);
      const int brow = ti.e * Nout + ti.nt * HB;
      int4 tok = make_int4(0, 0, 0, 0);
      if constexpr (GATHER) tok = gather_rows4(perm, ti.row0, lane, ti.rows);
      for (int kb = 0; kb < KB; ++kb) {
        bool go = lane != 0 || mbar_wait_bounded(smem_addr(&empty_bar[s]), ph ^ 1u, abort_flag, timeout_ns);
        if constexpr (GATHER) go = __shfl_sync(0xffffffffu, go, 0);
        if (!go) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_addr(&full_bar[s]);
        const uint32_t sa = smem_addr(stage_a + s * C::kABytes);
        const uint32_t sb = smem_addr(stage_b + s * C::kBBytes);
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          if (!GATHER) tma_load_2d(sa, &tmA, fb, kb * kTcBK, ti.row0);
          tma_load_2d(sb, &tmB0, fb, kb * kTcBK, brow);
          if (EPI == EPI_SWIGLU) tma_load_2d(sb + HB * kTcBK * 2, &tmB1, fb, kb * kTcBK, brow);
        }
        if constexpr (GATHER) {
          __syncwarp();
          tma_gather4(sa + lane * (4 * kTcBK * 2), &tmA, fb, kb * kTcBK, tok.x, tok.y, tok.z, tok.w);
        }
        ++issued;
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      // let every copy still in flight land before the CTA exits
      const long long first = issued > S ? issued - S : 0;
      for (long long i = first; i < issued; ++i)
        mbar_wait_bounded(smem_addr(&full_bar[i % S]), static_cast<uint32_t>((i / S) & 1), nullptr, timeout_ns);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    int s = 0;
    uint32_t ph = 0;
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    for (long long id = blockIdx.x; id < total && ok; id += gridDim.x) {
      if (!mbar_wait_bounded(smem_addr(&tempty_bar[acc]), aph ^ 1u, abort_flag, timeout_ns)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_bounded(smem_addr(&full_bar[s]), ph, abort_flag, timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = sw128_kmajor_desc(smem_addr(stage_a + s * C::kABytes));
        const uint64_t bd = sw128_kmajor_desc(smem_addr(stage_b + s * C::kBBytes));
#pragma unroll
        for (int kk = 0; kk < kTcBK / 16; ++kk)
          umma_bf16(d_tmem, ad + 2u * kk, bd + 2u * kk, IDESC, (kb | kk) != 0 ? 1u : 0u);
        umma_commit(smem_addr(&empty_bar[s]));
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
      umma_commit(smem_addr(&tfull_bar[acc]));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    // every MMA this thread issued has completed before TMEM is freed
    umma_commit(smem_addr(drain_bar));
    mbar_wait_bounded(smem_addr(drain_bar), 0u, nullptr, timeout_ns);
  } else if (warp >= 2) {
    // ---------------- epilogue
    const int q = warp & 3;   // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t aph = 0;
    for (long long id = blockIdx.x; id < total; id += gridDim.x) {
      const TileInfo ti = decode_tile(id, s_off, s_pre, N, n_tiles, kTcBM);
      if (!mbar_wait_bounded(smem_addr(&tfull_bar[acc]), aph, abort_flag, timeout_ns)) break;
      tc_fence_after();
      const int r = q * 32 + lane;
      const bool valid = r < ti.rows;
      const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(q * 32) << 16);
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
      if (lane == 0) mbar_arrive(smem_addr(&tempty_bar[acc]));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace moe
