// route.cuh -- K1: fused gate projection + top-k + renormalised gate weights.
//
// "MoE显存与计算开销四阶段手算指南" sections 2.1-2.2 and
// "MoE混合专家模型计算原理与推理部署实战解析" sections 2.1, 2.2, 2.4:
//   s[t,n] = sum_i x[t,i] W_g[i,n] (+ b[n])  in fp32 (the gate is kept in fp32)
//   the k largest s (ties -> lower expert id), in descending order
//   w_j = softmax(s)_{e_j} / sum_j' softmax(s)_{e_j'}
// The full softmax denominator cancels in the renormalisation, so the kernel
// evaluates w_j = exp(s_j - s_max) / sum_j' exp(s_j' - s_max) over the k
// selected scores only (identical in exact arithmetic).
//
// Expert bias, two modes: added to the logits before the softmax (so it moves
// both the choice and the weights), or -- the auxiliary-loss-free balancing
// of "MoE混合专家模型计算原理与推理部署实战解析" section 4.4 -- added only to the
// scores that choose the experts, the weights then coming from the softmax of
// the unbiased logits. Either way the choosing score is the fp32 sum
// logit + b.
//
// Routing statistics (optional): each CTA writes, for its tokens, the sum of
// the full softmax p[t,n] per expert, the number of assignments per expert,
// and the sum of the top-1 probabilities, in a fixed order;
// route_stats_kernel reduces the per-CTA rows into the load statistics of
// section 4.2 of the same page (fraction routed f, mean probability P,
// N * sum f P) plus the activation entropy and mean top-1 probability of
// "这不是“参数越多越强”的简单故事" sections 3.1 and 4.4. No float atomics: the
// statistics are reproducible bit for bit.
//
// Gate probabilities (optional, for expert-choice routing): probs_out [T,N]
// receives the full softmax p[t,:] in fp32; with topk_idx == null the top-k
// step is skipped.
//
// Each logit is the sequential FMA chain over i = 0..d-1 in index order (one
// thread owns it from start to end), then one fp32 bias add: the plainest fp32
// evaluation, so the top-k decision is reproducible bit for bit.
//
// One CTA owns TM tokens and all N experts (padded to NP = EG*EPT). K slices
// of 32 columns of x (raw dtype) and W_g (fp32) stream through a cp.async ring
// of STAGES buffers. Thread (ty, tx) accumulates TPT tokens x EPT experts in
// registers; the TM x NP logit tile then goes to shared memory, where one warp
// per token runs k rounds of a warp-wide argmax. Logits never reach HBM.
// TM is picked per launch (64, 32 or 8 tokens) so that small batches still
// spread over many SMs.
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kRouteBK = 32;
constexpr int kRouteThreads = 256;

template <int EG, int EPT, int TPT, typename TX, int THR = kRouteThreads>
struct RouteCfg {
  static constexpr int NP = EG * EPT;
  static constexpr int TG = THR / EG;
  static constexpr int TM = TG * TPT;
  static constexpr int XROW = kRouteBK * static_cast<int>(sizeof(TX)) + 16;  // bytes per token row (+pad)
  static constexpr int XBYTES = TM * XROW;                                   // one stage of x
  static constexpr int WBYTES = kRouteBK * NP * 4;                           // one stage of W_g
  // few experts: a slice is computed quickly, so more slices stay in flight (about 48 KB)
  static constexpr int SFEW = 49152 / (XBYTES + WBYTES);
  static constexpr int STAGES = NP >= 128 ? 3 : (NP >= 32 ? 4 : (SFEW < 4 ? 4 : (SFEW > 12 ? 12 : SFEW)));
  static constexpr size_t kPipe = static_cast<size_t>(STAGES) * (XBYTES + WBYTES);
  static constexpr size_t kLogits = sizeof(float) * TM * (NP + 1);
  // per-warp statistics rows [THR / 32][2*NP + 1] after the logit tile
  static constexpr size_t kStats = kLogits + sizeof(float) * (THR / 32) * (2 * NP + 1);
  static constexpr size_t kSmem = kPipe > kStats ? kPipe : kStats;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;   // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
// Two independent fp32 FMA chains in one instruction: d.lo = fma(a.lo, b.lo,
// d.lo), d.hi = fma(a.hi, b.hi, d.hi), each rounded to nearest like fmaf, so
// a logit's chain is the same as with scalar FMAs.
__device__ __forceinline__ void ffma2(unsigned long long& d, unsigned long long a, unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
__device__ __forceinline__ unsigned long long splat2(float v) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ void unpack2(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 8 consecutive K elements of one token, widened to fp32.
__device__ __forceinline__ void load_x8(const __nv_bfloat16* p, float* v) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
  v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
}
__device__ __forceinline__ void load_x8(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// One token's top-k, by one warp: k rounds of a warp-wide argmax over the
// choosing scores v (ties -> lower expert id), then the renormalised weights
// w_j = exp(g_j - g_max) / sum over the chosen of exp(g - g_max), g being the
// softmax logits of the chosen experts (the max-shifted softmax restricted to
// the k chosen). Expert n = lane + 32 m sits in slot m; taken marks experts
// that may not be chosen (out of range). c_acc[m] += 1 for each chosen expert
// of this lane (routing statistics). Writes idx_out[0..k) and w_out[0..k).
template <int SLOTS>
__device__ __forceinline__ void topk_renorm(const float* g, const float* v, bool* taken, int k, int lane,
                                            int32_t* __restrict__ idx_out, float* __restrict__ w_out, float* c_acc) {
  float sel_v[SLOTS];
  int sel_i[SLOTS];
#pragma unroll
  for (int m = 0; m < SLOTS; ++m) { sel_v[m] = -INFINITY; sel_i[m] = 0; }
  float top = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int m = 0; m < SLOTS; ++m) {
      const int n = lane + 32 * m;
      if (!taken[m] && (v[m] > bv || (v[m] == bv && n < bi))) { bv = v[m]; bi = n; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    // the winner's softmax logit (its score unless the bias only chooses)
    float gw = -INFINITY;
#pragma unroll
    for (int m = 0; m < SLOTS; ++m)
      if ((bi >> 5) == m) gw = g[m];
    gw = __shfl_sync(0xffffffffu, gw, bi & 31);
    top = (j == 0) ? gw : fmaxf(top, gw);
#pragma unroll
    for (int m = 0; m < SLOTS; ++m) {
      if (bi == lane + 32 * m) {
        taken[m] = true;
        c_acc[m] += 1.f;
      }
      if ((j & 31) == lane && (j >> 5) == m) { sel_v[m] = gw; sel_i[m] = bi; }
    }
  }
  float part = 0.f;
  float ex[SLOTS];
#pragma unroll
  for (int m = 0; m < SLOTS; ++m) {
    const int j = lane + 32 * m;
    ex[m] = (j < k) ? expf(sel_v[m] - top) : 0.f;
    part += ex[m];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
  const float inv = 1.f / part;
#pragma unroll
  for (int m = 0; m < SLOTS; ++m) {
    const int j = lane + 32 * m;
    if (j < k) {
      idx_out[j] = sel_i[m];
      w_out[j] = ex[m] * inv;
    }
  }
}

// The end of a routing CTA, shared by the route kernels: the TM x NP logit
// tile lg[token][n] (row pitch NP + 1, padded experts -inf) is complete in
// shared memory. One warp per token runs the top-k and the renormalised
// weights; optionally the full softmax for the statistics rows (srow: shared
// scratch of [THR / 32][2 NP + 1] floats, written into stats_part's row of
// this CTA) and for probs_out.
template <int NP, int TM, int THR>
__device__ __forceinline__ void route_select(const float* lg, float* srow, int64_t t0, int T, int N, int k,
                                             const float* __restrict__ bias, int bias_select,
                                             int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                             float* __restrict__ stats_part, float* __restrict__ probs_out) {
  constexpr int NPR = NP < 32 ? 32 : NP;   // register slots per token for the argmax
  constexpr int SLOTS = NPR / 32;
  // top-k: one warp per token, k rounds of warp argmax (ties -> lower id)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool want_stats = stats_part != nullptr;
  float bsel[SLOTS];          // the bias of the choosing score when it only chooses
  float p_acc[SLOTS];         // statistics: sum over this warp's tokens of p[t,n]
  float c_acc[SLOTS];         //             assignments to n
  float top1_acc = 0.f;       //             sum of the top-1 probabilities
#pragma unroll
  for (int m = 0; m < SLOTS; ++m) {
    const int n = lane + 32 * m;
    bsel[m] = (bias != nullptr && bias_select && n < N) ? bias[n] : 0.f;
    p_acc[m] = 0.f;
    c_acc[m] = 0.f;
  }
  for (int tl = warp; tl < TM; tl += THR / 32) {
    const int64_t t = t0 + tl;
    if (t >= T) break;
    float g[SLOTS];           // logits of the softmax
    float v[SLOTS];           // choosing scores
    bool taken[SLOTS];
#pragma unroll
    for (int m = 0; m < SLOTS; ++m) {
      const int n = lane + 32 * m;
      g[m] = (n < NP) ? lg[tl * (NP + 1) + n] : -INFINITY;
      v[m] = (n < N) ? g[m] + bsel[m] : -INFINITY;
      taken[m] = (n >= N);
    }
    if (topk_idx != nullptr)   // top-k choice and its renormalised weights
      topk_renorm<SLOTS>(g, v, taken, k, lane, topk_idx + t * k, topk_w + t * k, c_acc);
    if (want_stats || probs_out != nullptr) {   // full softmax over the N experts
      float gmax = -INFINITY;
#pragma unroll
      for (int m = 0; m < SLOTS; ++m) gmax = fmaxf(gmax, g[m]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, off));
      float e[SLOTS], z = 0.f;
#pragma unroll
      for (int m = 0; m < SLOTS; ++m) {
        e[m] = (lane + 32 * m < N) ? expf(g[m] - gmax) : 0.f;
        z += e[m];
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
      const float iz = 1.f / z;
#pragma unroll
      for (int m = 0; m < SLOTS; ++m) {
        const int n = lane + 32 * m;
        p_acc[m] += e[m] * iz;
        if (probs_out != nullptr && n < N) probs_out[t * N + n] = e[m] * iz;
      }
      top1_acc += iz;         // p of the largest logit is exp(0) / z
    }
  }
  if (!want_stats) return;
  // per-warp rows -> one row per CTA: [N probability sums | N counts | top-1 sum]
  constexpr int SW = 2 * NP + 1;
#pragma unroll
  for (int m = 0; m < SLOTS; ++m) {
    const int n = lane + 32 * m;
    if (n < NP) {
      srow[warp * SW + n] = p_acc[m];
      srow[warp * SW + NP + n] = c_acc[m];
    }
  }
  if (lane == 0) srow[warp * SW + 2 * NP] = top1_acc;
  __syncthreads();
  float* out = stats_part + static_cast<int64_t>(blockIdx.x) * (2 * N + 1);
  for (int n = tid; n < N; n += THR) {
    float ps = 0.f, cs = 0.f;
#pragma unroll
    for (int w = 0; w < THR / 32; ++w) {
      ps += srow[w * SW + n];
      cs += srow[w * SW + NP + n];
    }
    out[n] = ps;
    out[N + n] = cs;
  }
  if (tid == 0) {
    float ts = 0.f;
#pragma unroll
    for (int w = 0; w < THR / 32; ++w) ts += srow[w * SW + 2 * NP];
    out[2 * N] = ts;
  }
}

template <int EG, int EPT, int TPT, typename TX, int THR = kRouteThreads>
__global__ void __launch_bounds__(THR) route_kernel(const TX* __restrict__ x, const float* __restrict__ wg,
                                                              const float* __restrict__ bias, int T, int d, int N,
                                                              int k, int bias_select,
                                                              int32_t* __restrict__ topk_idx,
                                                              float* __restrict__ topk_w,
                                                              float* __restrict__ stats_part,
                                                              float* __restrict__ probs_out) {
  using C = RouteCfg<EG, EPT, TPT, TX, THR>;
  constexpr int NP = C::NP, TM = C::TM, S = C::STAGES;
  constexpr int XCH = kRouteBK * static_cast<int>(sizeof(TX)) / 16;   // 16-byte chunks per token row slice
  extern __shared__ __align__(16) uint8_t route_smem[];
  uint8_t* xs = route_smem;                      // [S][TM][XROW bytes]
  float* ws = reinterpret_cast<float*>(route_smem + S * C::XBYTES);   // [S][BK][NP]
  float* lg = reinterpret_cast<float*>(route_smem);                   // [TM][NP+1] after the K loop

  // Thread (ty, tx) owns tokens ty*TPT + i and experts V*tx + V*EG*m + c
  // (m < EPT/V, c < V, V = min(EPT, 4)): its W_g reads are V-wide vectors and
  // the threads of a warp read consecutive vectors, free of bank conflicts.
  constexpr int V = EPT < 4 ? EPT : 4;
  const int tid = threadIdx.x;
  const int tx = tid % EG;
  const int ty = tid / EG;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * TM;
  const int KB = (d + kRouteBK - 1) / kRouteBK;
  const bool w_vec = (N % 4) == 0;

  auto issue = [&](int kb) {
    const int st = kb % S;
    const int k0 = kb * kRouteBK;
    const uint32_t xb = smem_addr(xs + st * C::XBYTES);
    for (int c = tid; c < TM * XCH; c += THR) {
      const int r = c / XCH, q = c % XCH;
      const int64_t t = t0 + r;
      const int kk = k0 + q * (16 / static_cast<int>(sizeof(TX)));
      const bool ok = (t < T) && (kk < d);
      const TX* src = ok ? x + t * d + kk : x;
      cp_async16(xb + r * C::XROW + q * 16, src, ok);
    }
    const uint32_t wb = smem_addr(ws + st * kRouteBK * NP);
    if (w_vec) {
      for (int c = tid; c < kRouteBK * NP / 4; c += THR) {
        const int kr = c / (NP / 4), n4 = (c % (NP / 4)) * 4;
        const int gk = k0 + kr;
        const bool ok = (gk < d) && (n4 < N);
        const float* src = ok ? wg + static_cast<int64_t>(gk) * N + n4 : wg;
        cp_async16(wb + (kr * NP + n4) * 4, src, ok);
      }
    } else {
      for (int c = tid; c < kRouteBK * NP; c += THR) {
        const int kr = c / NP, n = c % NP;
        const int gk = k0 + kr;
        const bool ok = (gk < d) && (n < N);
        const float* src = ok ? wg + static_cast<int64_t>(gk) * N + n : wg;
        cp_async4(wb + c * 4, src, ok);
      }
    }
  };

  // Accumulators: with two or more experts per thread, pairs of neighbouring
  // experts share one packed register pair and one f32x2 FMA.
  constexpr bool PACKED = EPT >= 2;
  constexpr int EP2 = PACKED ? EPT / 2 : 1;
  float acc[TPT][EPT];
  unsigned long long acc2[TPT][EP2];
#pragma unroll
  for (int i = 0; i < TPT; ++i) {
#pragma unroll
    for (int j = 0; j < EPT; ++j) acc[i][j] = 0.f;
#pragma unroll
    for (int p = 0; p < EP2; ++p) acc2[i][p] = 0ull;
  }

#pragma unroll
  for (int s = 0; s < S - 1; ++s) {
    if (s < KB) issue(s);
    cp_async_commit();
  }
  for (int kb = 0; kb < KB; ++kb) {
    cp_async_wait<S - 2>();
    __syncthreads();
    if (kb + S - 1 < KB) issue(kb + S - 1);
    cp_async_commit();
    const int st = kb % S;
    const uint8_t* xst = xs + st * C::XBYTES;
    const float* wst = ws + st * kRouteBK * NP;
    if constexpr (EPT == 1 && TPT <= 2) {
      // few chains per thread (few experts): the slice's shared loads first, then its FMAs, so their
      // latency is paid once per slice instead of once per step
      float xv[TPT][kRouteBK];
      float wv[kRouteBK][EPT];
#pragma unroll
      for (int i = 0; i < TPT; ++i)
#pragma unroll
        for (int k8 = 0; k8 < kRouteBK; k8 += 8)
          load_x8(reinterpret_cast<const TX*>(xst + (ty * TPT + i) * C::XROW) + k8, xv[i] + k8);
#pragma unroll
      for (int u = 0; u < kRouteBK; ++u)
#pragma unroll
        for (int m = 0; m < EPT; ++m) wv[u][m] = wst[u * NP + V * tx + V * EG * (m / V) + (m % V)];
#pragma unroll
      for (int u = 0; u < kRouteBK; ++u)
#pragma unroll
        for (int i = 0; i < TPT; ++i)
#pragma unroll
          for (int j = 0; j < EPT; ++j) acc[i][j] = fmaf(xv[i][u], wv[u][j], acc[i][j]);
      continue;
    }
#pragma unroll
    for (int k8 = 0; k8 < kRouteBK; k8 += 8) {
      float xv[TPT][8];
#pragma unroll
      for (int i = 0; i < TPT; ++i)
        load_x8(reinterpret_cast<const TX*>(xst + (ty * TPT + i) * C::XROW) + k8, xv[i]);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float* wr = wst + (k8 + u) * NP + V * tx;
        if constexpr (PACKED) {
          unsigned long long wp[EP2];   // (expert 2p, expert 2p + 1) of this thread
#pragma unroll
          for (int m = 0; m < EPT / V; ++m) {
            if constexpr (V == 4) {
              const ulonglong2 q = *reinterpret_cast<const ulonglong2*>(wr + V * EG * m);
              wp[2 * m] = q.x;
              wp[2 * m + 1] = q.y;
            } else {
              wp[m] = *reinterpret_cast<const unsigned long long*>(wr + V * EG * m);
            }
          }
#pragma unroll
          for (int i = 0; i < TPT; ++i) {
            const unsigned long long xx = splat2(xv[i][u]);
#pragma unroll
            for (int p = 0; p < EP2; ++p) ffma2(acc2[i][p], xx, wp[p]);
          }
        } else {
          float wv[EPT];
#pragma unroll
          for (int m = 0; m < EPT; ++m) wv[m] = wr[EG * m];
#pragma unroll
          for (int i = 0; i < TPT; ++i)
#pragma unroll
            for (int j = 0; j < EPT; ++j) acc[i][j] = fmaf(xv[i][u], wv[j], acc[i][j]);
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  if constexpr (PACKED) {
#pragma unroll
    for (int i = 0; i < TPT; ++i)
#pragma unroll
      for (int p = 0; p < EP2; ++p) unpack2(acc2[i][p], acc[i][2 * p], acc[i][2 * p + 1]);
  }

  // logits (+ bias, unless it only chooses) -> lg[token][n]; padded experts get -inf
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int n = V * tx + V * EG * (j / V) + (j % V);
    const float b = (bias != nullptr && !bias_select && n < N) ? bias[n] : 0.f;
#pragma unroll
    for (int i = 0; i < TPT; ++i) lg[(ty * TPT + i) * (NP + 1) + n] = (n < N) ? acc[i][j] + b : -INFINITY;
  }
  __syncthreads();

  route_select<NP, TM, THR>(lg, reinterpret_cast<float*>(route_smem + C::kLogits), t0, T, N, k, bias, bias_select,
                            topk_idx, topk_w, stats_part, probs_out);
}

// Small batches (decode): each logit chain is d sequential FMAs, so the time
// floor is d FMA latencies whatever the parallelism, and the batch is too
// small to fill the GPU with chains. This kernel trims the per-step work of a
// chain: one CTA holds TC tokens and all N experts (N = NP); its TC x rows
// (contiguous in memory) arrive in shared memory by one bulk copy, and W_g
// streams through a ring of S slices of BK whole rows (each slice contiguous
// in memory, one bulk copy) on mbarriers, every copy issued by one thread, so
// the chains' threads issue no copies. Each thread owns the chains of two
// neighbouring experts (thread (t, p) = (tid / (NP/2), tid % (NP/2)), experts
// 2p and 2p + 1): a step is one 8-byte shared load of W_g[i, 2p..2p+1], one
// widened x value (eight per 16-byte broadcast load) and two independent
// FMAs. Same arithmetic as route_kernel (each chain over i in index order,
// one fp32 bias add), so the routing is identical bit for bit; statistics and
// probability outputs are route_kernel's. Needs N = NP and d a multiple of
// BK. Every wait on a copy is bounded: on a timeout the CTA records
// MOE_ERR_TIMEOUT, lets its copies in flight land and writes nothing.
template <int NP>
struct RouteSmallCfg {
  static constexpr int BK = 64;
  static constexpr int WBYTES = BK * NP * 4;
  static constexpr int SFIT = (96 * 1024) / WBYTES;
  static constexpr int STAGES = SFIT < 3 ? 3 : (SFIT > 8 ? 8 : SFIT);
  // shared memory for TC tokens of d values of es bytes: ring, x rows, barriers
  static size_t smem(int TC, int d, int es) {
    return static_cast<size_t>(STAGES) * WBYTES + static_cast<size_t>(TC) * d * es + 8 * (STAGES + 1);
  }
};

template <int NP, int TC, typename TX>
__global__ void __launch_bounds__(TC * NP / 2) route_small_kernel(const TX* __restrict__ x,
                                                                  const float* __restrict__ wg,
                                                                  const float* __restrict__ bias, int T, int d,
                                                                  int N, int k, int bias_select,
                                                                  int32_t* __restrict__ topk_idx,
                                                                  float* __restrict__ topk_w,
                                                                  unsigned long long timeout_ns) {
  using C = RouteSmallCfg<NP>;
  constexpr int NPH = NP / 2;                     // threads per token
  constexpr int THR = TC * NPH, BK = C::BK, S = C::STAGES;
  constexpr int SLOTS = NP / 32;
  static_assert(NP % 64 == 0 && THR / 32 >= TC, "one warp per token for the top-k");
  extern __shared__ __align__(16) uint8_t rs_smem[];
  float* ws = reinterpret_cast<float*>(rs_smem);                                  // [S][BK][NP]
  TX* xs = reinterpret_cast<TX*>(rs_smem + static_cast<size_t>(S) * C::WBYTES);  // [TC][d]
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xs) +
                                               static_cast<size_t>(TC) * d * sizeof(TX));   // full[S], x
  const int tid = threadIdx.x;
  const int tl = tid / NPH, n = 2 * (tid % NPH);  // experts n, n + 1
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * TC;
  const int KB = d / BK;
  const int rows = static_cast<int>(min(static_cast<int64_t>(TC), static_cast<int64_t>(T) - t0));

  if (tid == 0) {
    for (int s = 0; s <= S; ++s) mbar_init(smem_addr(&bars[s]), 1);
    fence_barrier_init();
  }
  __syncthreads();
  int issued = 0;
  if (tid == 0) {
    // rows past T are never copied: their chains compute garbage nobody reads
    const uint32_t xb = static_cast<uint32_t>(rows) * d * sizeof(TX);
    mbar_arrive_expect_tx(smem_addr(&bars[S]), xb);
    bulk_load(smem_addr(xs), x + t0 * d, xb, smem_addr(&bars[S]));
    for (; issued < S - 1 && issued < KB; ++issued) {
      mbar_arrive_expect_tx(smem_addr(&bars[issued]), C::WBYTES);
      bulk_load(smem_addr(ws + issued * BK * NP), wg + static_cast<int64_t>(issued) * BK * NP, C::WBYTES,
                smem_addr(&bars[issued]));
    }
  }
  bool ok = mbar_wait_bounded(smem_addr(&bars[S]), 0u, nullptr, timeout_ns);

  float acc0 = 0.f, acc1 = 0.f;
  const TX* xr = xs + static_cast<int64_t>(tl) * d;
  int kb = 0;
  for (; kb < KB; ++kb) {
    ok = ok && mbar_wait_bounded(smem_addr(&bars[kb % S]), static_cast<uint32_t>((kb / S) & 1), nullptr, timeout_ns);
    // uniform decision; every thread is done with slice kb - 1, so its slot may be refilled
    if (__syncthreads_or(!ok)) break;
    if (tid == 0 && issued < KB) {
      const int s = issued % S;
      mbar_arrive_expect_tx(smem_addr(&bars[s]), C::WBYTES);
      bulk_load(smem_addr(ws + s * BK * NP), wg + static_cast<int64_t>(issued) * BK * NP, C::WBYTES,
                smem_addr(&bars[s]));
      ++issued;
    }
    const float2* wcol = reinterpret_cast<const float2*>(ws + (kb % S) * BK * NP + n);
    const TX* xk = xr + kb * BK;
#pragma unroll
    for (int g8 = 0; g8 < BK; g8 += 8) {
      float xv[8];
      load_x8(xk + g8, xv);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float2 w2 = wcol[(g8 + u) * NPH];
        acc0 = fmaf(xv[u], w2.x, acc0);
        acc1 = fmaf(xv[u], w2.y, acc1);
      }
    }
  }
  if (kb < KB) {
    // gave up: let every copy in flight land before the CTA exits, write nothing
    if (tid == 0) {
      for (int i = kb; i < issued; ++i)
        mbar_wait_bounded(smem_addr(&bars[i % S]), static_cast<uint32_t>((i / S) & 1), nullptr, timeout_ns);
    }
    return;
  }
  __syncthreads();

  // logits (+ bias, unless it only chooses) -> lg[token][n]
  float* lg = reinterpret_cast<float*>(rs_smem);                                  // [TC][NP + 1]
  const bool add_bias = bias != nullptr && !bias_select;
  lg[tl * (NP + 1) + n] = acc0 + (add_bias ? bias[n] : 0.f);
  lg[tl * (NP + 1) + n + 1] = acc1 + (add_bias ? bias[n + 1] : 0.f);
  __syncthreads();

  const int warp = tid >> 5, lane = tid & 31;
  if (warp >= rows) return;
  const int64_t t = t0 + warp;
  float g[SLOTS], v[SLOTS], c_acc[SLOTS];
  bool taken[SLOTS];
#pragma unroll
  for (int m = 0; m < SLOTS; ++m) {
    const int e = lane + 32 * m;
    const float bs = (bias != nullptr && bias_select) ? bias[e] : 0.f;
    g[m] = lg[warp * (NP + 1) + e];
    v[m] = g[m] + bs;
    taken[m] = false;
    c_acc[m] = 0.f;
  }
  topk_renorm<SLOTS>(g, v, taken, k, lane, topk_idx + t * k, topk_w + t * k, c_acc);
}

// Load statistics from the route kernel's per-CTA rows (one CTA, 256 threads,
// thread n owns expert n; sums in CTA order, in fp64). out layout:
//   out[0, N)    f[n] = assignments to n / (T k)
//   out[N, 2N)   P[n] = mean over tokens of p[t,n]
//   out[2N]      N * sum_n f[n] P[n]        (1 for a uniform load)
//   out[2N + 1]  -sum_{f > 0} f log2 f      (activation entropy, bits)
//   out[2N + 2]  mean top-1 probability
// An empty batch gives zeros.
__global__ void __launch_bounds__(256) route_stats_kernel(const float* __restrict__ part, int64_t n_rows,
                                                          int64_t T, int N, int k, float* __restrict__ out) {
  __shared__ double red_b[256], red_e[256];
  const int n = threadIdx.x;
  const int64_t W = 2 * N + 1;
  double bal = 0.0, ent = 0.0;
  if (n < N) {
    double ps = 0.0, cs = 0.0;
    for (int64_t c = 0; c < n_rows; ++c) {
      ps += part[c * W + n];
      cs += part[c * W + N + n];
    }
    const double f = T > 0 ? cs / (static_cast<double>(T) * k) : 0.0;
    const double P = T > 0 ? ps / static_cast<double>(T) : 0.0;
    out[n] = static_cast<float>(f);
    out[N + n] = static_cast<float>(P);
    bal = f * P;
    ent = f > 0.0 ? -f * log2(f) : 0.0;
  }
  red_b[n] = bal;
  red_e[n] = ent;
  __syncthreads();
  for (int h = 128; h > 0; h >>= 1) {
    if (n < h) {
      red_b[n] += red_b[n + h];
      red_e[n] += red_e[n + h];
    }
    __syncthreads();
  }
  if (n == 0) {
    double ts = 0.0;
    for (int64_t c = 0; c < n_rows; ++c) ts += part[c * W + 2 * N];
    out[2 * N] = static_cast<float>(static_cast<double>(N) * red_b[0]);
    out[2 * N + 1] = static_cast<float>(red_e[0]);
    out[2 * N + 2] = T > 0 ? static_cast<float>(ts / static_cast<double>(T)) : 0.f;
  }
}

}  // namespace moe
