// ffn_tc_swap.cuh -- bf16 grouped GEMM on the tensor cores with the expert's
// tokens as the MMA's N side ("token tiles").
//
// Same product as ffn_tc.cuh ("MoE混合专家模型计算原理与推理部署实战解析"
// sections 3.1-3.2; "MoE显存与计算开销四阶段手算指南" section 4.3), computed
// transposed: D[feature, token] = W[feature, :] . X[token, :]^T.
//
// Tokens: an expert with c rows gets ceil(c / 256) token tiles of equal size
// rounded up to 16 (the MMA's N), so padding is < 16 rows per tile instead of
// < 128: experts with a few hundred rows (the pages' worked example, 8192 x 2
// assignments over 64 experts) waste ~5% of the MMA work instead of ~25%.
//
// Weights: each tile pairs two 128-row weight tiles against the one token tile
// (two M = 128 MMAs per K step sharing the B operand): SwiGLU pairs the gate
// rows and the up rows of the same 128 hidden features, so the epilogue forms
// silu(gate) * up lane by lane; GELU and the down projection pair two
// consecutive 128-row blocks (256 output features). A stage is then 32 KB of
// weights + up to 32 KB of tokens for 2 x 128 x N x 64 MMA work: two thirds of
// the bytes per MMA cycle of the row-tile kernel, in a 3-stage ring. The
// pair of fp32 accumulators fills
// the 512 TMEM columns, so the epilogue of a tile is not overlapped with the
// next tile's main loop (a few percent of a tile's time).
//
// Roles: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 2-9
// epilogue, two per TMEM lane quarter taking alternate 32-token chunks (lane = feature, TMEM column = token; each warp transposes its
// 32 features x 32 tokens through a private XOR-swizzled shared tile and
// stores 64 contiguous bytes per token row). All waits are bounded.
#pragma once
#include "ffn_tc.cuh"

namespace moe {

constexpr int kSwFM = 128;                 // MMA M: weight rows per MMA
constexpr int kSwMaxNT = 256;              // MMA N: token rows per tile (max)
constexpr int kSwBox = 32;                 // token rows per TMA box
constexpr int kSwEpiWarps = 8;             // two warps per TMEM lane quarter
constexpr int kSwThreads = 32 * (2 + kSwEpiWarps);   // TMA, MMA, 8 epilogue warps
constexpr int kSwTmemCols = 2 * kSwMaxNT;               // D0 at column 0, D1 at column 256
constexpr int kSwXposeBytes = kSwEpiWarps * 32 * 64;    // one 32 x 32 bf16 tile per epilogue warp
constexpr int kSwRingBudget = 192 * 1024;

// Ring geometry for a K depth of BK elements per stage (BK = 64: 128-byte
// swizzled rows, 3 stages; BK = 32: 64-byte rows, 6 stages). BK = 64 is the
// one launched: the 64-byte-swizzle variant measured ~45 % slower.
template <int BK>
struct SwCfg {
  static constexpr int kRowBytes = BK * 2;
  static constexpr int kWBytes = kSwFM * kRowBytes;              // one 128-row weight block
  static constexpr int kABytes = 2 * kWBytes;                    // the pair of weight blocks
  static constexpr int kBBytes = kSwMaxNT * kRowBytes;           // token block
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kSwRingBudget / kStageBytes;
  static constexpr int kNumBars = 2 * kStages + 3;
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + kSwXposeBytes +
                                       8 * kNumBars + 16 + 2 * 257 * sizeof(int) + 16;
};

// Output features covered by one tile: SwiGLU 128 (gate/up pair), else 256.
template <int EPI>
__host__ __device__ constexpr int sw_tile_features() { return EPI == EPI_SWIGLU ? kSwFM : 2 * kSwFM; }

struct SwTile {
  int e;      // expert
  int fi;     // feature tile
  int row0;   // first permuted row
  int rows;   // valid token rows (1..256)
  int nt;     // MMA N: rows rounded up to 16
};

// Token tiles of expert e: ntt = ceil(c / 256) tiles of base = roundup16(ceil(c / ntt))
// rows; tile ids ordered (expert, feature tile, token tile).
__device__ __forceinline__ SwTile sw_decode(long long id, const int* s_off, const int* s_pre, int N, int n_ftiles) {
  int lo = 0, hi = N;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<long long>(s_pre[mid]) * n_ftiles <= id) lo = mid;
    else hi = mid;
  }
  const int ntt = s_pre[lo + 1] - s_pre[lo];
  const long long local = id - static_cast<long long>(s_pre[lo]) * n_ftiles;
  const int cnt = s_off[lo + 1] - s_off[lo];
  const int base = ((cnt + ntt - 1) / ntt + 15) & ~15;
  const int ti = static_cast<int>(local % ntt);
  SwTile t;
  t.e = lo;
  t.fi = static_cast<int>(local / ntt);
  t.row0 = s_off[lo] + ti * base;
  t.rows = min(base, cnt - ti * base);
  t.nt = (t.rows + 15) & ~15;
  return t;
}

// Byte offset of element (token j, feature l) in a warp's 32 x 32 bf16
// transpose tile: rows of 64 B, 16-byte chunks XOR-swizzled by (j >> 1) & 3 so
// that both the per-feature writes and the per-token 16-byte reads are free
// of bank conflicts.
__device__ __forceinline__ int sw_xpose_off(int j, int l) {
  return j * 64 + ((((l >> 3) ^ (j >> 1)) & 3) << 4) + ((l & 7) << 1);
}

// v[j] (fp32, token c + j of feature `lane`) -> out[row0 + c + j][fcol + lane],
// through the warp's transpose tile; rows >= rows are not written.
__device__ __forceinline__ void sw_store_transposed(const uint32_t* v, uint8_t* xp, uint32_t xp_s, int lane, int c,
                                                    int rows, int row0, int fcol, __nv_bfloat16* out, int ldo) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    *reinterpret_cast<__nv_bfloat16*>(xp + sw_xpose_off(j, lane)) = __float2bfloat16_rn(__uint_as_float(v[j]));
  __syncwarp();
  const int tok = c + lane;
  if (tok < rows) {
    __nv_bfloat16* dst = out + static_cast<int64_t>(row0 + tok) * ldo + fcol;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      uint4 val;
      const uint32_t a = xp_s + lane * 64 + (((ch ^ (lane >> 1)) & 3) << 4);
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                   : "r"(a));
      reinterpret_cast<uint4*>(dst)[ch] = val;
    }
  }
  __syncwarp();
}

// With GATHER the token rows come straight from the unpermuted tokens x
// through the permutation (perm[row] = token), four rows per lane of warp 0
// per stage (TMA tile::gather4); the map of x then has a box one row high.
template <int EPI, int BK, bool GATHER = false>
__global__ void __launch_bounds__(kSwThreads, 1)
    grouped_gemm_tc_swap_kernel(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                                const __grid_constant__ CUtensorMap tmX, const int32_t* __restrict__ offsets, int N,
                                int rows_total, int K, int Nout, __nv_bfloat16* __restrict__ out, int ldo,
                                unsigned long long timeout_ns, const int32_t* __restrict__ perm) {
  static_assert(!GATHER || BK == 64, "gathered rows are 128-byte swizzled");
  using C = SwCfg<BK>;
  constexpr int S = C::kStages;
  constexpr int OF = sw_tile_features<EPI>();
  constexpr uint32_t IDESC0 = idesc_bf16_f32(kSwFM, 16) & ~(0x3Fu << 17);   // N field filled per tile

  extern __shared__ uint8_t sw_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sw_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_a = smem;                      // S x (W0 block | W1 block)
  uint8_t* stage_b = smem + S * C::kABytes;     // S x token block
  uint8_t* xpose = smem + S * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(xpose + kSwXposeBytes);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + S;
  uint64_t* tfull_bar = bars + 2 * S;
  uint64_t* tempty_bar = tfull_bar + 1;
  uint64_t* drain_bar = tfull_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
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
    mbar_init(smem_addr(tfull_bar), 1);
    mbar_init(smem_addr(tempty_bar), kSwEpiWarps);
    mbar_init(smem_addr(drain_bar), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    build_tile_prefix(offsets, N, rows_total, kSwMaxNT, s_off, s_pre, bad_flag);
    if (lane == 0) {
      prefetch_tensormap(&tmW0);
      prefetch_tensormap(&tmX);
      if (EPI == EPI_SWIGLU) prefetch_tensormap(&tmW1);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kSwTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const bool bad = *bad_flag != 0;
  if (bad && threadIdx.x == 0 && blockIdx.x == 0) record_error(MOE_ERR_CORRUPT);
  const int n_ftiles = (Nout + OF - 1) / OF;
  const long long total = bad ? 0 : static_cast<long long>(s_pre[N]) * n_ftiles;
  const int KB = K / BK;

  if (warp == 0 && (GATHER || lane == 0)) {
    // ---------------- TMA producer (lane 0 waits and loads the weights; with GATHER the lanes
    // gather four token rows each, twice for tiles of more than 128 rows)
    int s = 0;
    uint32_t ph = 0;
    long long issued = 0;
    bool ok = true;
    for (long long id = blockIdx.x; id < total && ok; id += gridDim.x) {
      const SwTile t = sw_decode(id, s_off, s_pre, N, n_ftiles);
      // weight rows of the pair: SwiGLU (gate f0.., up f0..); else (f0.., f0+128..)
      const int w0row = t.e * Nout + t.fi * OF;
      const int w1row = (EPI == EPI_SWIGLU) ? w0row : w0row + kSwFM;
      const int nbox = (t.nt + kSwBox - 1) / kSwBox;
      const int ngat = (t.nt + 3) / 4;
      const uint32_t tx_bytes = C::kABytes + (GATHER ? ngat * 4 * C::kRowBytes : nbox * kSwBox * C::kRowBytes);
      int4 tok0 = make_int4(0, 0, 0, 0), tok1 = tok0;
      if constexpr (GATHER) {
        tok0 = gather_rows4(perm, t.row0, lane, t.rows);
        tok1 = gather_rows4(perm, t.row0, lane + 32, t.rows);
      }
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
          mbar_arrive_expect_tx(fb, tx_bytes);
          tma_load_2d(sa, &tmW0, fb, kb * BK, w0row);
          tma_load_2d(sa + C::kWBytes, (EPI == EPI_SWIGLU) ? &tmW1 : &tmW0, fb, kb * BK, w1row);
          if (!GATHER)
            for (int b = 0; b < nbox; ++b)
              tma_load_2d(sb + b * kSwBox * C::kRowBytes, &tmX, fb, kb * BK, t.row0 + b * kSwBox);
        }
        if constexpr (GATHER) {
          __syncwarp();
          if (lane < ngat)
            tma_gather4(sb + lane * (4 * C::kRowBytes), &tmX, fb, kb * BK, tok0.x, tok0.y, tok0.z, tok0.w);
          if (lane + 32 < ngat)
            tma_gather4(sb + (lane + 32) * (4 * C::kRowBytes), &tmX, fb, kb * BK, tok1.x, tok1.y, tok1.z, tok1.w);
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
    // ---------------- MMA issuer: D0 = W0 . X^T, D1 = W1 . X^T
    int s = 0;
    uint32_t ph = 0;
    uint32_t aph = 0;
    bool ok = true;
    for (long long id = blockIdx.x; id < total && ok; id += gridDim.x) {
      const SwTile t = sw_decode(id, s_off, s_pre, N, n_ftiles);
      const uint32_t idesc = IDESC0 | (static_cast<uint32_t>(t.nt >> 3) << 17);
      if (!mbar_wait_bounded(smem_addr(tempty_bar), aph ^ 1u, abort_flag, timeout_ns)) break;
      tc_fence_after();
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_bounded(smem_addr(&full_bar[s]), ph, abort_flag, timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t a0 = kmajor_swizzled_desc<C::kRowBytes>(smem_addr(stage_a + s * C::kABytes));
        const uint64_t a1 = kmajor_swizzled_desc<C::kRowBytes>(smem_addr(stage_a + s * C::kABytes + C::kWBytes));
        const uint64_t bd = kmajor_swizzled_desc<C::kRowBytes>(smem_addr(stage_b + s * C::kBBytes));
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
          umma_bf16(tmem_base, a0 + 2u * kk, bd + 2u * kk, idesc, acc);
          umma_bf16(tmem_base + kSwMaxNT, a1 + 2u * kk, bd + 2u * kk, idesc, acc);
        }
        umma_commit(smem_addr(&empty_bar[s]));
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
      umma_commit(smem_addr(tfull_bar));
      aph ^= 1u;
    }
    // every MMA this thread issued has completed before TMEM is freed
    umma_commit(smem_addr(drain_bar));
    mbar_wait_bounded(smem_addr(drain_bar), 0u, nullptr, timeout_ns);
  } else if (warp >= 2) {
    // ---------------- epilogue: two warps per lane quarter, alternate 32-token chunks
    const int q = warp & 3;   // TMEM lane quarter: features 32q .. 32q+31 of each weight block
    const int half = (warp - 2) >> 2;
    uint8_t* xp = xpose + (warp - 2) * (32 * 64);
    const uint32_t xp_s = smem_addr(xp);
    uint32_t aph = 0;
    for (long long id = blockIdx.x; id < total; id += gridDim.x) {
      const SwTile t = sw_decode(id, s_off, s_pre, N, n_ftiles);
      if (!mbar_wait_bounded(smem_addr(tfull_bar), aph, abort_flag, timeout_ns)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int f0 = t.fi * OF + q * 32;                 // feature of lane 0, first block
#pragma unroll 1
      for (int c = 32 * half; c < t.nt; c += 64) {
        uint32_t v[32];
        tmem_ld_32x32(tb + c, v);
        if (EPI == EPI_SWIGLU) {
          uint32_t u[32];
          tmem_ld_32x32(tb + kSwMaxNT + c, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float g = __uint_as_float(v[i]);
            v[i] = __float_as_uint(__fdividef(g, 1.f + __expf(-g)) * __uint_as_float(u[i]));
          }
          if (f0 < Nout) sw_store_transposed(v, xp, xp_s, lane, c, t.rows, t.row0, f0, out, ldo);
        } else {
          tmem_ld_wait();
          if (EPI == EPI_GELU) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float a = __uint_as_float(v[i]);
              v[i] = __float_as_uint(0.5f * a * (1.f + tanh_fast(0.7978845608028654f * (a + 0.044715f * a * a * a))));
            }
          }
          if (f0 < Nout) sw_store_transposed(v, xp, xp_s, lane, c, t.rows, t.row0, f0, out, ldo);
          tmem_ld_32x32(tb + kSwMaxNT + c, v);
          tmem_ld_wait();
          if (EPI == EPI_GELU) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float a = __uint_as_float(v[i]);
              v[i] = __float_as_uint(0.5f * a * (1.f + tanh_fast(0.7978845608028654f * (a + 0.044715f * a * a * a))));
            }
          }
          if (f0 + kSwFM < Nout) sw_store_transposed(v, xp, xp_s, lane, c, t.rows, t.row0, f0 + kSwFM, out, ldo);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(tempty_bar));
      aph ^= 1u;
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kSwTmemCols);
  }
}

}  // namespace moe
