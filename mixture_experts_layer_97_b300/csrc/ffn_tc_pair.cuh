// ffn_tc_pair.cuh -- bf16 grouped GEMM with token tiles on SM pairs.
//
// The product of ffn_tc_swap.cuh ("MoE混合专家模型计算原理与推理部署实战解析"
// sections 3.1-3.2; "MoE显存与计算开销四阶段手算指南" section 4.3), computed
// by clusters of two CTAs whose tensor cores run one MMA together
// (tcgen05 cta_group::2): D[256 weight rows, N tokens] with each CTA holding
// 128 of the weight rows and HALF of the N token rows in its shared memory.
// Each CTA still pairs two weight blocks (two MMAs per K step share the
// token operand), so per K step a CTA stages 32 KB of weights but only 8-16
// KB of tokens: 48 KB stages, four of them, where the single-SM token kernel
// fits three 64 KB stages. The deeper ring keeps more weight bytes in flight
// per SM; the token half read by each SM also halves the L2 -> SM traffic
// for the tokens.
//
// Features per pair tile: SwiGLU 256 hidden units (CTA r: gate and up rows
// of units [128 r, 128 r + 128) of the tile), GELU and the down projection
// 512 output features (CTA r: rows [256 r, 256 r + 256) as two 128-row
// blocks). Token tiles are those of the single-SM kernel (at most 256 rows,
// balanced per expert, multiples of 16); CTA r holds tokens
// [r nt / 2, (r + 1) nt / 2) of the tile.
//
// With GATHER (the first GEMM of the layer) the token rows come straight from
// the unpermuted tokens x through the permutation (perm[row] = token): lanes
// of warp 0 gather four rows each per stage (TMA tile::gather4).
//
// Tiles are handed out dynamically: the even CTA's producer takes the next
// tile id from a global counter (zeroed before the launch) whenever it starts
// a tile, and passes it through a small queue (kPrQueue slots on mbarriers)
// to its own MMA issuer and epilogue warps and, through distributed shared
// memory, to the odd CTA's producer and epilogue warps; id -1 ends the loop.
// Tile ids keep the (expert, feature tile, token tile) order, so the token
// tiles of one weight tile still run at the same time on neighbouring pairs,
// while tiles of unequal size no longer pile up on some pairs (on the worked
// example's routing a static round robin gives the busiest pair 23 % more
// work than the average in the down projection).
//
// Roles (both CTAs): warp 0 TMA producer for the CTA's own shared memory,
// warp 1 TMEM (allocated by both CTAs together) and, in the even CTA only,
// the MMA issuer; warps 2-9 epilogue on the CTA's own TMEM (its 128 weight
// rows x all N tokens). Barriers: the even CTA's full barriers count the
// bytes of both CTAs' copies; the MMA issuer's commits arrive on the empty,
// accumulator-full and drain barriers of both CTAs; both CTAs' epilogue
// warps arrive on the even CTA's accumulator-empty barrier. Every mbarrier
// wait is bounded; both CTAs meet at cluster barriers after set-up and
// before TMEM is freed, so neither leaves while the other can still touch
// its shared memory or tensor memory.
#pragma once
#include "ffn_tc_swap.cuh"

namespace moe {

constexpr int kPrStages = 4;
constexpr int kPrRowBytes = kTcBK * 2;                       // 128-byte K rows
constexpr int kPrWBytes = kSwFM * kPrRowBytes;              // one 128-row weight block: 16 KB
constexpr int kPrABytes = 2 * kPrWBytes;                    // the CTA's pair of weight blocks
constexpr int kPrBRows = kSwMaxNT / 2;                      // token rows per CTA (max)
constexpr int kPrBBytes = kPrBRows * kPrRowBytes;           // 16 KB
constexpr int kPrStageBytes = kPrABytes + kPrBBytes;        // 48 KB
constexpr int kPrQueue = 4;                                 // tile ids in flight between the roles
constexpr int kPrNumBars = 2 * kPrStages + 3 + 2 * kPrQueue;
// consumers of a queue slot: the MMA issuer, the odd CTA's producer, 8 epilogue warps per CTA
constexpr int kPrQueueConsumers = 2 + 2 * kSwEpiWarps;
constexpr size_t kPrSmemBytes = 1024 + static_cast<size_t>(kPrStages) * kPrStageBytes + kSwXposeBytes +
                                8 * kPrNumBars + 16 + 2 * 257 * sizeof(int) + kPrQueue * sizeof(int) + 16;
static_assert(kPrSmemBytes <= 227 * 1024, "pair kernel shared memory");

// Output features of one pair tile and of each CTA's half.
template <int EPI>
__host__ __device__ constexpr int pr_tile_features() { return EPI == EPI_SWIGLU ? 2 * kSwFM : 4 * kSwFM; }

// ---------------------------------------------------------------- pair PTX
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (both CTAs' TMEM at d_tmem) (+)= A (both CTAs' shared memory at a_desc) *
// B (both CTAs' halves at b_desc)^T; issued by one thread of the even CTA.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at this offset in both CTAs when the MMAs
// issued so far have completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  const uint16_t both = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"(both)
      : "memory");
}

// TMA into this CTA's shared memory, completion counted on the even CTA's
// mbarrier (bar_cluster: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int x,
                                                 int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

template <int EPI, bool GATHER = false>
__global__ void __launch_bounds__(kSwThreads, 1)
    grouped_gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                                const __grid_constant__ CUtensorMap tmX, const int32_t* __restrict__ offsets, int N,
                                int rows_total, int K, int Nout, __nv_bfloat16* __restrict__ out, int ldo,
                                unsigned long long timeout_ns, const int32_t* __restrict__ perm,
                                int* __restrict__ tile_counter) {
  constexpr int S = kPrStages;
  constexpr int OFP = pr_tile_features<EPI>();      // features per pair tile
  constexpr int OFC = OFP / 2;                      // features of this CTA
  // M = 256 (128 rows in each CTA); the N field is filled per tile
  constexpr uint32_t IDESC0 = idesc_bf16_f32(2 * kSwFM, 16) & ~(0x3Fu << 17);

  extern __shared__ uint8_t pr_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pr_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_a = smem;                        // S x (W0 block | W1 block)
  uint8_t* stage_b = smem + S * kPrABytes;        // S x this CTA's token half
  uint8_t* xpose = smem + S * kPrStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(xpose + kSwXposeBytes);
  uint64_t* full_bar = bars;                      // used in the even CTA only
  uint64_t* empty_bar = bars + S;
  uint64_t* tfull_bar = bars + 2 * S;
  uint64_t* tempty_bar = tfull_bar + 1;           // used in the even CTA only
  uint64_t* drain_bar = tfull_bar + 2;
  uint64_t* tq_full = tfull_bar + 3;              // [kPrQueue], both CTAs
  uint64_t* tq_empty = tq_full + kPrQueue;        // [kPrQueue], used in the even CTA only
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kPrNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* bad_flag = reinterpret_cast<int*>(tmem_slot + 2);
  int* s_off = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_pre = s_off + 257;
  volatile int* tq = s_pre + 257;                 // [kPrQueue] tile ids

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), 1);
    }
    mbar_init(smem_addr(tfull_bar), 1);
    mbar_init(smem_addr(tempty_bar), 2 * kSwEpiWarps);
    mbar_init(smem_addr(drain_bar), 1);
    for (int q = 0; q < kPrQueue; ++q) {
      mbar_init(smem_addr(&tq_full[q]), 1);
      mbar_init(smem_addr(&tq_empty[q]), kPrQueueConsumers);
    }
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
  // both CTAs' barriers are initialised before either signals the other's
  cluster_sync_all();
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), kSwTmemCols);
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
  // the tile queue: slot q % kPrQueue; a consumer takes use q at parity (q / kPrQueue) & 1
  auto q_slot = [](uint32_t q) { return q % kPrQueue; };
  auto q_par = [](uint32_t q) { return (q / kPrQueue) & 1u; };
  // Next tile id for use q, in every role's loop (lane 0 of the calling warp
  // answers, the warp gets the id): the even CTA's producer fetches it and
  // publishes it to both CTAs; every other role reads it from its own queue
  // and releases the slot on the even CTA. -1: no more tiles (or gave up).
  auto next_tile = [&](uint32_t q, bool fetcher, bool warp_wide) -> long long {
    long long id = -1;
    if (lane == 0) {
      const uint32_t sl = q_slot(q);
      if (fetcher) {
        if (mbar_wait_bounded(smem_addr(&tq_empty[sl]), q_par(q) ^ 1u, abort_flag, timeout_ns)) {
          const long long v = atomicAdd(tile_counter, 1);
          id = v < total ? v : -1;
        }
        tq[sl] = static_cast<int>(id);
        st_cluster_s32(smem_addr_in_cta(smem_addr(const_cast<int*>(&tq[sl])), 1), static_cast<int>(id));
        mbar_arrive(smem_addr(&tq_full[sl]));
        mbar_arrive_remote(smem_addr_in_cta(smem_addr(&tq_full[sl]), 1));
      } else {
        if (mbar_wait_bounded<true>(smem_addr(&tq_full[sl]), q_par(q), abort_flag, timeout_ns)) id = tq[sl];
        mbar_arrive_remote(smem_addr_in_cta(smem_addr(&tq_empty[sl]), 0));
      }
    }
    return warp_wide ? __shfl_sync(0xffffffffu, id, 0) : id;
  };

  if (warp == 0 && (GATHER || lane == 0)) {
    // ---------------- TMA producer (each CTA fills its own shared memory; lane 0 takes the tile ids,
    // waits and loads the weights, and with GATHER the first lanes gather four token rows each)
    int s = 0;
    uint32_t ph = 0;
    long long issued = 0;
    bool ok = true;
    for (uint32_t qi = 0; ok; ++qi) {
      const long long id = next_tile(qi, leader, GATHER);
      if (id < 0) break;
      const SwTile t = sw_decode(id, s_off, s_pre, N, n_ftiles);
      const int w0row = t.e * Nout + t.fi * OFP + static_cast<int>(rank) * OFC;
      const int w1row = (EPI == EPI_SWIGLU) ? w0row : w0row + kSwFM;
      const int half = t.nt >> 1;                               // token rows per CTA
      const int r0 = t.row0 + static_cast<int>(rank) * half;
      const int nbox = (half + kSwBox - 1) / kSwBox;
      const int ngat = (half + 3) / 4;                          // gathers of four rows (GATHER)
      const uint32_t tx_pair =
          2u * (kPrABytes + (GATHER ? ngat * 4 * kPrRowBytes : nbox * kSwBox * kPrRowBytes));
      int4 tok = make_int4(0, 0, 0, 0);
      if constexpr (GATHER) {
        // this CTA's valid rows of the tile: [rank * half, rank * half + half) clipped to t.rows
        const int valid = min(half, max(0, t.rows - static_cast<int>(rank) * half));
        tok = valid > 0 ? gather_rows4(perm, r0, lane, valid) : gather_rows4(perm, t.row0, 0, 1);
      }
      for (int kb = 0; kb < KB; ++kb) {
        bool go = lane != 0 || mbar_wait_bounded(smem_addr(&empty_bar[s]), ph ^ 1u, abort_flag, timeout_ns);
        if constexpr (GATHER) go = __shfl_sync(0xffffffffu, go, 0);
        if (!go) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_addr_in_cta(smem_addr(&full_bar[s]), 0);
        const uint32_t sa = smem_addr(stage_a + s * kPrABytes);
        const uint32_t sb = smem_addr(stage_b + s * kPrBBytes);
        if (lane == 0) {
          if (leader) mbar_arrive_expect_tx(smem_addr(&full_bar[s]), tx_pair);
          tma_load_2d_pair(sa, &tmW0, fb, kb * kTcBK, w0row);
          tma_load_2d_pair(sa + kPrWBytes, (EPI == EPI_SWIGLU) ? &tmW1 : &tmW0, fb, kb * kTcBK, w1row);
          if (!GATHER)
            for (int b = 0; b < nbox; ++b)
              tma_load_2d_pair(sb + b * kSwBox * kPrRowBytes, &tmX, fb, kb * kTcBK, r0 + b * kSwBox);
        }
        if constexpr (GATHER) {
          __syncwarp();
          if (lane < ngat)
            tma_gather4_pair(sb + lane * (4 * kPrRowBytes), &tmX, fb, kb * kTcBK, tok.x, tok.y, tok.z, tok.w);
        }
        ++issued;
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
    if (!ok && leader && lane == 0) {
      // let the copies still in flight (both CTAs') land before the CTAs leave
      const long long first = issued > S ? issued - S : 0;
      for (long long i = first; i < issued; ++i)
        mbar_wait_bounded(smem_addr(&full_bar[i % S]), static_cast<uint32_t>((i / S) & 1), nullptr, timeout_ns);
    }
  } else if (warp == 1 && lane == 0) {
    if (leader) {
      // ---------------- MMA issuer for the pair: D0 = W0 . X^T, D1 = W1 . X^T
      int s = 0;
      uint32_t ph = 0;
      uint32_t aph = 0;
      bool ok = true;
      for (uint32_t qi = 0; ok; ++qi) {
        const long long id = next_tile(qi, false, false);
        if (id < 0) break;
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
          const uint64_t a0 = kmajor_swizzled_desc<kPrRowBytes>(smem_addr(stage_a + s * kPrABytes));
          const uint64_t a1 = kmajor_swizzled_desc<kPrRowBytes>(smem_addr(stage_a + s * kPrABytes + kPrWBytes));
          const uint64_t bd = kmajor_swizzled_desc<kPrRowBytes>(smem_addr(stage_b + s * kPrBBytes));
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk) {
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            umma_bf16_pair(tmem_base, a0 + 2u * kk, bd + 2u * kk, idesc, acc);
            umma_bf16_pair(tmem_base + kSwMaxNT, a1 + 2u * kk, bd + 2u * kk, idesc, acc);
          }
          umma_commit_pair(smem_addr(&empty_bar[s]));
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair(smem_addr(tfull_bar));
        aph ^= 1u;
      }
      // every MMA issued has completed before either CTA frees TMEM
      umma_commit_pair(smem_addr(drain_bar));
    }
    mbar_wait_bounded(smem_addr(drain_bar), 0u, nullptr, timeout_ns);
  } else if (warp >= 2) {
    // ---------------- epilogue on this CTA's TMEM: its 128 weight rows x all tokens
    const int q = warp & 3;
    const int hsel = (warp - 2) >> 2;
    uint8_t* xp = xpose + (warp - 2) * (32 * 64);
    const uint32_t xp_s = smem_addr(xp);
    const uint32_t tempty_leader = smem_addr_in_cta(smem_addr(tempty_bar), 0);
    uint32_t aph = 0;
    for (uint32_t qi = 0;; ++qi) {
      const long long id = next_tile(qi, false, true);
      if (id < 0) break;
      const SwTile t = sw_decode(id, s_off, s_pre, N, n_ftiles);
      if (!mbar_wait_bounded(smem_addr(tfull_bar), aph, abort_flag, timeout_ns)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int f0 = t.fi * OFP + static_cast<int>(rank) * OFC + q * 32;   // feature of lane 0, first block
#pragma unroll 1
      for (int c = 32 * hsel; c < t.nt; c += 64) {
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
      if (lane == 0) mbar_arrive_remote(tempty_leader);
      aph ^= 1u;
    }
  }

  __syncthreads();
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kSwTmemCols);
}

}  // namespace moe
