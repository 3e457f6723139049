// moe_b300.cu -- the C ABI of libmoe_b300.so (declared in include/moe.h).
//
// Host side of every entry point: validate arguments before launching,
// carve the caller's workspace, build TMA tensor maps, pick kernel variants
// and launch on the caller's stream. No allocation, no synchronisation
// (except moe_get_error), no CPU fallback.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "combine.cuh"
#include "common.cuh"
#include "ep.cuh"
#include "expert_choice.cuh"
#include "ffn_simt.cuh"
#include "ffn_tc.cuh"
#include "ffn_tc_swap.cuh"
#include "ffn_tc_pair.cuh"
#include "ffn_tc_rowpair.cuh"
#include "permute.cuh"
#include "route.cuh"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;   // 2 s per bounded device wait
constexpr int kMaxDevices = 64;
constexpr int kAutoTokenTileMinRowsPerExpert = 64;  // auto tiling: token tiles from this many rows per expert
constexpr int kAutoTokenTileMinK = 4096;            // ... and this reduction length

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t esize(const moe_shape* s) { return s->dtype == MOE_F32 ? 4 : 2; }
int64_t n_assign(const moe_shape* s) { return s->T * s->k; }

// Bump allocator over the caller's workspace (base == nullptr: size only).
struct Carve {
  uint8_t* base;
  size_t used = 0;
  explicit Carve(void* p) : base(static_cast<uint8_t*>(p)) {}
  template <typename T>
  T* take(size_t bytes) {
    T* r = base ? reinterpret_cast<T*>(base + used) : nullptr;
    used += align_up(bytes);
    return r;
  }
};

int64_t perm_chunks(const moe_shape* s) {
  const int tpc = perm_tokens_per_chunk(s->k);
  return (s->T + tpc - 1) / tpc;
}

size_t permute_ws(const moe_shape* s) { return align_up(sizeof(int32_t) * perm_chunks(s) * s->N); }
// The grouped FFN's workspace: h [A, F], then the SM-pair GEMM's tile counter.
size_t ffn_h_bytes(const moe_shape* s) { return align_up(esize(s) * static_cast<size_t>(n_assign(s)) * s->d_ff); }
size_t ffn_ws(const moe_shape* s) { return ffn_h_bytes(s) + kAlign; }
// Statistics rows of one route launch: at most one per 4 tokens, 2N + 1 floats each.
size_t route_stats_ws(const moe_shape* s) {
  return align_up(sizeof(float) * static_cast<size_t>((s->T + 3) / 4) * (2 * static_cast<size_t>(s->N) + 1));
}

constexpr long long kNoCapacity = 0x7fffffffffffffffLL;

// Options of one forward beyond the plain layer.
struct FwdOpts {
  int bias_select = 0;                 // the expert bias only chooses
  long long capacity = kNoCapacity;    // rows an expert keeps
  int32_t* dropped = nullptr;          // device [1]: dropped assignments
  float* load_stats = nullptr;         // device [2N + 3]: routing statistics
  int tiling = -1;                     // grouped-GEMM tiling of this call; -1: the process-wide setting
};

struct FwdBufs {
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  void* x_perm;
  void* y_perm;
  void* perm_ws;
  void* ffn_ws;
  void* stats_ws;
  void* x_dev;     // hostio only
  void* out_dev;   // hostio only
  size_t total;
};

FwdBufs carve_forward(const moe_shape* s, void* ws, bool hostio) {
  Carve c(ws);
  FwdBufs b{};
  const size_t A = static_cast<size_t>(n_assign(s));
  const size_t es = esize(s);
  b.topk_idx = c.take<int32_t>(sizeof(int32_t) * A);
  b.topk_w = c.take<float>(sizeof(float) * A);
  b.counts = c.take<int32_t>(sizeof(int32_t) * s->N);
  b.offsets = c.take<int32_t>(sizeof(int32_t) * (s->N + 1));
  b.perm = c.take<int32_t>(sizeof(int32_t) * A);
  b.inv_perm = c.take<int32_t>(sizeof(int32_t) * A);
  b.x_perm = c.take<uint8_t>(es * A * s->d);
  b.y_perm = c.take<uint8_t>(es * A * s->d);
  b.perm_ws = c.take<uint8_t>(permute_ws(s));
  b.ffn_ws = c.take<uint8_t>(ffn_ws(s));
  b.stats_ws = c.take<uint8_t>(route_stats_ws(s));
  if (hostio) {
    b.x_dev = c.take<uint8_t>(es * static_cast<size_t>(s->T) * s->d);
    b.out_dev = c.take<uint8_t>(es * static_cast<size_t>(s->T) * s->d);
  }
  b.total = c.used;
  return b;
}

moe_status shape_status(const moe_shape* s) {
  if (s == nullptr) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->d < 1 || s->N < 1 || s->k < 1 || s->d_ff < 1 || s->k > s->N) return MOE_ERR_INVALID_ARG;
  if (s->act != MOE_SWIGLU && s->act != MOE_GELU_TANH) return MOE_ERR_INVALID_ARG;
  if (s->dtype != MOE_F32 && s->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (s->N > 256) return MOE_ERR_UNSUPPORTED;
  if (s->T * static_cast<int64_t>(s->k) >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  const int64_t big = static_cast<int64_t>(s->N) * (s->d > s->d_ff ? s->d : s->d_ff);
  if (big >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  if (s->dtype == MOE_BF16) {
    if (s->d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (s->d_ff % (s->act == MOE_SWIGLU ? 64 : 128) != 0) return MOE_ERR_UNSUPPORTED;
  } else {
    if (s->d % 4 != 0) return MOE_ERR_UNSUPPORTED;
    if (s->d_ff > 65535 * 64 || s->d > 65535 * 64) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

bool ptr_ok(const void* p, bool needed) { return needed ? (p != nullptr && aligned16(p)) : (p == nullptr || aligned16(p)); }

// SM count of the current device, looked up once per device. Host threads may
// race on the first lookup: each slot is an atomic, and every racer stores the
// same value.
int num_sms() {
  static std::atomic<int> cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= kMaxDevices) return 148;
  int n = cache[dev].load(std::memory_order_acquire);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev].store(n, std::memory_order_release);
  }
  return n;
}

moe_status launched() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ---------------------------------------------------------------- route
// What one route launch writes besides the top-k; `rows` returns the number
// of per-CTA statistics rows the launch produced.
struct RouteArgs {
  const float* wg;
  const float* bias;
  int bias_select;
  int32_t* idx;
  float* w;
  float* stats_part;   // [grid][2N + 1] or null
  int64_t rows;
  float* probs_out;    // [T, N] or null
};

template <int EG, int EPT, int TPT, typename TX>
moe_status launch_route_cfg(const moe_shape* s, const TX* x, RouteArgs& a, cudaStream_t st) {
  using Cfg = RouteCfg<EG, EPT, TPT, TX>;
  auto kern = route_kernel<EG, EPT, TPT, TX>;
  if (Cfg::kSmem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Cfg::kSmem)) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  const int64_t grid = (s->T + Cfg::TM - 1) / Cfg::TM;
  a.rows = grid;
  kern<<<static_cast<unsigned>(grid), kRouteThreads, Cfg::kSmem, st>>>(
      x, a.wg, a.bias, static_cast<int>(s->T), s->d, s->N, s->k, a.bias_select, a.idx, a.w, a.stats_part,
      a.probs_out);
  return launched();
}

// Experts padded to NP = EG * EPT, the smallest power of two >= max(N, EG);
// tokens per CTA TM = (256 / EG) * TPT.
template <int EG, int TPT, typename TX>
moe_status launch_route_tm(const moe_shape* s, const TX* x, RouteArgs& a, cudaStream_t st) {
  if (s->N <= EG) return launch_route_cfg<EG, 1, TPT, TX>(s, x, a, st);
  if constexpr (EG * 2 <= 256) {
    if (s->N <= EG * 2) return launch_route_cfg<EG, 2, TPT, TX>(s, x, a, st);
  }
  if constexpr (EG * 4 <= 256) {
    if (s->N <= EG * 4) return launch_route_cfg<EG, 4, TPT, TX>(s, x, a, st);
  }
  if constexpr (EG * 8 <= 256) {
    if (s->N <= EG * 8) return launch_route_cfg<EG, 8, TPT, TX>(s, x, a, st);
  }
  if constexpr (EG * 16 <= 256) {
    if (s->N <= EG * 16) return launch_route_cfg<EG, 16, TPT, TX>(s, x, a, st);
  }
  return MOE_ERR_UNSUPPORTED;
}

// Decode-sized batches: one CTA per token with all experts (route_small_kernel).
template <int NP, typename TX>
moe_status launch_route_small(const moe_shape* s, const TX* x, RouteArgs& a, cudaStream_t st) {
  using C = RouteSmallCfg<NP>;
  auto kern = route_small_kernel<NP, 1, TX>;
  const size_t smem = C::smem(1, s->d, static_cast<int>(sizeof(TX)));
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  kern<<<static_cast<unsigned>(s->T), NP / 2, smem, st>>>(x, a.wg, a.bias, static_cast<int>(s->T), s->d, s->N, s->k,
                                                         a.bias_select, a.idx, a.w, kWaitTimeoutNs);
  return launched();
}

// The small-batch kernel applies to top-k routing without statistics or
// probability outputs, 64 or 128 experts (its whole W_g rows are its ring
// slices), d a multiple of its 64-row slices with an x row of at most 48 KB,
// and up to four CTAs per SM (measured: 32 tokens x 3584 x 64 experts 27 us
// against 55 us for route_kernel; 128 tokens the same 27 us).
bool use_route_small(const moe_shape* s, const RouteArgs& a, int64_t sms) {
  if (a.stats_part != nullptr || a.probs_out != nullptr || a.idx == nullptr) return false;
  if (s->N != 64 && s->N != 128) return false;
  if (s->d % 64 != 0 || static_cast<int64_t>(s->d) * esize(s) > 48 * 1024) return false;
  return s->T <= 4 * sms;
}

// Each logit is one thread's sequential chain over d, so parallelism comes
// from tokens x experts: pick the largest token tile that still gives every
// SM a CTA, down to 4 tokens per CTA for decode-sized batches.
template <typename TX>
moe_status launch_route(const moe_shape* s, const TX* x, RouteArgs& a, cudaStream_t st) {
  a.rows = 0;
  if (s->T == 0) return MOE_OK;
  const int64_t sms = num_sms();
  const int64_t T = s->T;
  if (use_route_small(s, a, sms))
    return s->N == 64 ? launch_route_small<64, TX>(s, x, a, st) : launch_route_small<128, TX>(s, x, a, st);
  if (s->N <= 8) {   // 8 expert lanes: few experts are not padded to 16 or 32
    if ((T + 127) / 128 >= sms) return launch_route_tm<8, 4, TX>(s, x, a, st);   // 128 tokens/CTA
    if ((T + 63) / 64 >= sms) return launch_route_tm<8, 2, TX>(s, x, a, st);     // 64 tokens/CTA
    return launch_route_tm<8, 1, TX>(s, x, a, st);                                // 32 tokens/CTA
  }
  // Large batches: seven tokens per thread (more independent chains per thread hide more latency
  // than more warps do) in tiles that give each SM one CTA: 56 tokens x up to 64 experts, or 112
  // tokens x up to 128 experts (8192 x 64: 154 vs 168 us at 64 tokens per CTA; 16384 x 128: 227 vs
  // 252 us; 512-thread CTAs with fewer chains per thread were slower in both, and so were token
  // pairs in the packed FMAs with x widened once per CTA: 164 vs 154 us, 252 vs 229 us)
  if (s->N > 8 && s->N <= 64 && (T + 55) / 56 >= sms * 9 / 10) {
    if (s->N <= 32) return launch_route_cfg<32, 1, 7, TX>(s, x, a, st);                 // 56 tokens/CTA
    return launch_route_cfg<32, 2, 7, TX>(s, x, a, st);
  }
  if (s->N > 64 && s->N <= 128 && (T + 111) / 112 >= sms * 9 / 10)
    return launch_route_cfg<16, 8, 7, TX>(s, x, a, st);                                  // 112 tokens/CTA
  // 64 tokens per CTA already at 3/4 of an SM each: measured faster than 32 tokens on every SM
  // (8192 tokens, 64 experts: 166 vs 184 us), the 16 chains per thread hiding more FMA latency
  if ((T + 63) / 64 >= sms * 3 / 4) return launch_route_tm<16, 4, TX>(s, x, a, st);   // 64 tokens/CTA
  if ((T + 31) / 32 >= sms) return launch_route_tm<16, 2, TX>(s, x, a, st);       // 32 tokens/CTA
  if ((T + 7) / 8 >= sms / 2) return launch_route_tm<32, 1, TX>(s, x, a, st);     // 8 tokens/CTA
  return launch_route_tm<64, 1, TX>(s, x, a, st);                                 // 4 tokens/CTA
}

// Route, then (when load_stats is given) reduce the statistics rows that the
// route kernel left in stats_ws.
moe_status route_impl(const moe_shape* s, const void* x, const float* wg, const float* bias, int32_t* idx, float* w,
                      cudaStream_t st, int bias_select = 0, float* load_stats = nullptr, void* stats_ws = nullptr) {
  RouteArgs a{wg, bias, bias_select, idx, w, load_stats ? static_cast<float*>(stats_ws) : nullptr, 0, nullptr};
  moe_status r = s->dtype == MOE_BF16
                     ? launch_route<__nv_bfloat16>(s, static_cast<const __nv_bfloat16*>(x), a, st)
                     : launch_route<float>(s, static_cast<const float*>(x), a, st);
  if (r != MOE_OK || load_stats == nullptr) return r;
  route_stats_kernel<<<1, 256, 0, st>>>(a.stats_part, a.rows, s->T, s->N, s->k, load_stats);
  return launched();
}

// ---------------------------------------------------------------- permute
// x_perm[inv[t*k + j]] = x[t] for every j < k whose row is in [0, A).
moe_status launch_row_copy(const moe_shape* s, const int32_t* inv, const void* x, int k, int64_t A, void* x_perm,
                           cudaStream_t st) {
  if (s->T == 0) return MOE_OK;
  const int64_t nv = static_cast<int64_t>(s->d) * esize(s) / 16;
  const int64_t warps = s->T * copy_groups(nv);
  permute_copy_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, st>>>(
      inv, static_cast<const uint4*>(x), s->T, k, A, nv, static_cast<uint4*>(x_perm));
  return launched();
}


// x_perm == nullptr: counts, offsets, perm and inv_perm only (the grouped GEMM
// then gathers the token rows of x through perm itself).
moe_status permute_impl(const moe_shape* s, const int32_t* idx, const void* x, int32_t* counts, int32_t* offsets,
                        int32_t* perm, int32_t* inv_perm, void* x_perm, void* ws, cudaStream_t st,
                        long long capacity = kNoCapacity, int32_t* dropped = nullptr) {
  const int64_t C = perm_chunks(s);
  if (C == 1) {   // one chunk of whole tokens (T*k <= 2048): grouping and row copy in one launch
    const int64_t nv = static_cast<int64_t>(s->d) * esize(s) / 16;
    const int64_t copy_warps = x_perm != nullptr ? s->T * copy_groups(nv) : 0;
    const int64_t grid = copy_warps > 0 ? (copy_warps + kPermWarps - 1) / kPermWarps : 1;
    permute_single_kernel<<<static_cast<unsigned>(grid), kPermThreads, 0, st>>>(
        idx, s->T, s->N, s->k, capacity, counts, offsets, perm, inv_perm, dropped, static_cast<const uint4*>(x), nv,
        static_cast<uint4*>(x_perm));
    return launched();
  }
  int32_t* hist = static_cast<int32_t*>(ws);
  if (C > 0) {
    permute_hist_kernel<<<static_cast<unsigned>(C), kPermThreads, 0, st>>>(idx, s->T, s->N, s->k, hist);
    if (launched() != MOE_OK) return MOE_ERR_CUDA;
  }
  permute_scan_kernel<<<1, 256, 0, st>>>(hist, static_cast<int>(C), s->N, capacity, counts, offsets, dropped);
  if (launched() != MOE_OK) return MOE_ERR_CUDA;
  if (C > 0) {
    permute_rank_kernel<<<static_cast<unsigned>(C), kPermThreads, 0, st>>>(idx, hist, offsets, s->T, s->N, s->k,
                                                                            capacity, perm, inv_perm, dropped);
    if (launched() != MOE_OK) return MOE_ERR_CUDA;
    if (x_perm == nullptr) return MOE_OK;
    return launch_row_copy(s, inv_perm, x, s->k, n_assign(s), x_perm, st);
  }
  return MOE_OK;
}

// Rows an expert keeps under a capacity factor: ceil(cf * T * k / N) ("MoE混合专家
// 模型计算原理与推理部署实战解析" section 4.3, total counted in assignments).
long long capacity_rows(const moe_shape* s, double capacity_factor) {
  const double c = std::ceil(capacity_factor * static_cast<double>(s->T) * static_cast<double>(s->k) /
                             static_cast<double>(s->N));
  return c >= 2147483647.0 ? kNoCapacity : static_cast<long long>(c);
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, resolved once per process (std::call_once:
// safe when several host threads make their first call together).
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Tiling of the bf16 grouped GEMMs (moe_set_ffn_tiling), process wide; a
// moe_forward_ex call can override it for itself (moe_options.use_tiling).
std::atomic<int> g_ffn_tiling{MOE_TILING_AUTO};

bool tiling_valid(int mode) {
  return mode == MOE_TILING_AUTO || mode == MOE_TILING_ROWS || mode == MOE_TILING_TOKENS || mode == MOE_TILING_PAIRS ||
         mode == MOE_TILING_ROW_PAIRS;
}

// bf16 matrix [rows, cols] row-major; box = box_rows x box_cols columns with the
// swizzle whose span is one box row (box_cols * 2 bytes: 128 or 64).
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
              uint32_t box_cols = kTcBK) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = box_cols * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Where a grouped GEMM's token rows come from: the permuted rows a[A, K]
// (perm == nullptr), or rows of the unpermuted a[a_rows, K] gathered through
// perm (row -> token) by the kernel's loads.
struct RowSource {
  const void* a;
  const int32_t* perm;
  int64_t a_rows;
};

// The tensor map of a GEMM's token operand: box_rows-row boxes of permuted
// rows, or one-row boxes of the unpermuted rows for gathering.
bool make_row_map(CUtensorMap* m, const RowSource& src, int64_t A, int K, uint32_t box_rows) {
  if (src.perm != nullptr) return make_map(m, src.a, static_cast<uint64_t>(src.a_rows), static_cast<uint64_t>(K), 1);
  return make_map(m, src.a, static_cast<uint64_t>(A), static_cast<uint64_t>(K), box_rows);
}

// One grouped GEMM on the tensor cores: out[rows, Nout-slices] for every expert.
template <int BN, int EPI>
moe_status launch_tc(const moe_shape* s, const RowSource& src, int K, const void* b0, const void* b1, int Nout,
                     const int32_t* offsets, void* out, int ldo, cudaStream_t st) {
  using Cfg = TcCfg<BN>;
  constexpr int HB = (EPI == EPI_SWIGLU) ? BN / 2 : BN;
  const int64_t A = n_assign(s);
  CUtensorMap ma, mb0, mb1;
  if (!make_row_map(&ma, src, A, K, kTcBM)) return MOE_ERR_CUDA;
  const uint64_t brows = static_cast<uint64_t>(s->N) * Nout;
  if (!make_map(&mb0, b0, brows, static_cast<uint64_t>(K), HB)) return MOE_ERR_CUDA;
  if (EPI == EPI_SWIGLU) {
    if (!make_map(&mb1, b1, brows, static_cast<uint64_t>(K), HB)) return MOE_ERR_CUDA;
  } else {
    mb1 = mb0;
  }
  auto kern = src.perm != nullptr ? grouped_gemm_tc_kernel<BN, EPI, true> : grouped_gemm_tc_kernel<BN, EPI, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Cfg::kSmemBytes)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  const int64_t n_tiles = Nout / HB;
  const int64_t upper = ((A + kTcBM - 1) / kTcBM + s->N) * n_tiles;
  const int grid = static_cast<int>(upper < num_sms() ? upper : num_sms());
  kern<<<grid, kTcThreads, Cfg::kSmemBytes, st>>>(ma, mb0, mb1, offsets, s->N, static_cast<int>(A), K, Nout,
                                                  static_cast<__nv_bfloat16*>(out), ldo, kWaitTimeoutNs, src.perm);
  return launched();
}

// The same grouped GEMM with weights as the MMA's M side and the tokens of
// an expert as its N side (balanced token tiles, multiples of 16).
template <int EPI, int BK>
moe_status launch_tc_swap_bk(const moe_shape* s, const RowSource& src, int K, const void* w0, const void* w1,
                             int Nout, const int32_t* offsets, void* out, int ldo, cudaStream_t st) {
  using Cfg = SwCfg<BK>;
  constexpr int OF = sw_tile_features<EPI>();
  const int64_t A = n_assign(s);
  CUtensorMap mx, mw0, mw1;
  if (src.perm != nullptr) {
    if (!make_row_map(&mx, src, A, K, kSwBox)) return MOE_ERR_CUDA;
  } else if (!make_map(&mx, src.a, static_cast<uint64_t>(A), static_cast<uint64_t>(K), kSwBox, BK)) {
    return MOE_ERR_CUDA;
  }
  const uint64_t wrows = static_cast<uint64_t>(s->N) * Nout;
  if (!make_map(&mw0, w0, wrows, static_cast<uint64_t>(K), kSwFM, BK)) return MOE_ERR_CUDA;
  if (EPI == EPI_SWIGLU) {
    if (!make_map(&mw1, w1, wrows, static_cast<uint64_t>(K), kSwFM, BK)) return MOE_ERR_CUDA;
  } else {
    mw1 = mw0;
  }
  auto kern = src.perm != nullptr ? grouped_gemm_tc_swap_kernel<EPI, BK, true>
                                  : grouped_gemm_tc_swap_kernel<EPI, BK, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Cfg::kSmemBytes)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  const int64_t n_ftiles = (Nout + OF - 1) / OF;
  const int64_t upper = ((A + kSwMaxNT - 1) / kSwMaxNT + s->N) * n_ftiles;
  const int grid = static_cast<int>(upper < num_sms() ? upper : num_sms());
  kern<<<grid, kSwThreads, Cfg::kSmemBytes, st>>>(mw0, mw1, mx, offsets, s->N, static_cast<int>(A), K, Nout,
                                                  static_cast<__nv_bfloat16*>(out), ldo, kWaitTimeoutNs, src.perm);
  return launched();
}

// The token-tile grouped GEMM on SM pairs: clusters of two CTAs sharing
// each MMA (tcgen05 cta_group::2).
// tile_counter: a device int the kernel hands out tiles from; zeroed here, on
// the stream, before the launch.
template <int EPI>
moe_status launch_tc_pair(const moe_shape* s, const RowSource& src, int K, const void* w0, const void* w1, int Nout,
                          const int32_t* offsets, void* out, int ldo, cudaStream_t st, int* tile_counter) {
  constexpr int OFP = pr_tile_features<EPI>();
  const int64_t A = n_assign(s);
  CUtensorMap mx, mw0, mw1;
  if (!make_row_map(&mx, src, A, K, kSwBox)) return MOE_ERR_CUDA;
  const uint64_t wrows = static_cast<uint64_t>(s->N) * Nout;
  if (!make_map(&mw0, w0, wrows, static_cast<uint64_t>(K), kSwFM, kTcBK)) return MOE_ERR_CUDA;
  if (EPI == EPI_SWIGLU) {
    if (!make_map(&mw1, w1, wrows, static_cast<uint64_t>(K), kSwFM, kTcBK)) return MOE_ERR_CUDA;
  } else {
    mw1 = mw0;
  }
  auto kern = src.perm != nullptr ? grouped_gemm_tc_pair_kernel<EPI, true> : grouped_gemm_tc_pair_kernel<EPI, false>;
  if (cudaMemsetAsync(tile_counter, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kPrSmemBytes)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  const int64_t n_ftiles = (Nout + OFP - 1) / OFP;
  const int64_t pairs_needed = ((A + kSwMaxNT - 1) / kSwMaxNT + s->N) * n_ftiles;
  const int64_t max_pairs = num_sms() / 2;
  const int64_t pairs = pairs_needed < max_pairs ? pairs_needed : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kSwThreads, 1, 1);
  cfg.dynamicSmemBytes = kPrSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, mw0, mw1, mx, offsets, s->N, static_cast<int>(A), K, Nout,
                         static_cast<__nv_bfloat16*>(out), ldo, kWaitTimeoutNs, src.perm, tile_counter) != cudaSuccess)
    return MOE_ERR_CUDA;
  return launched();
}

// Row tiles on SM pairs: clusters of two CTAs sharing each MMA (256 permuted
// rows x 256 weight rows per tile, 128 of each in each CTA).
template <int EPI>
moe_status launch_tc_rowpair(const moe_shape* s, const void* a, int K, const void* b0, const void* b1, int Nout,
                             const int32_t* offsets, void* out, int ldo, cudaStream_t st) {
  constexpr int HB = rp_tile_cols<EPI>();
  const int64_t A = n_assign(s);
  CUtensorMap ma, mb0, mb1;
  if (!make_map(&ma, a, static_cast<uint64_t>(A), static_cast<uint64_t>(K), kRpHalf)) return MOE_ERR_CUDA;
  const uint64_t brows = static_cast<uint64_t>(s->N) * Nout;
  if (!make_map(&mb0, b0, brows, static_cast<uint64_t>(K), kRpHalf)) return MOE_ERR_CUDA;
  if (EPI == EPI_SWIGLU) {
    if (!make_map(&mb1, b1, brows, static_cast<uint64_t>(K), kRpHalf)) return MOE_ERR_CUDA;
  } else {
    mb1 = mb0;
  }
  auto kern = grouped_gemm_tc_rowpair_kernel<EPI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kRpSmemBytes)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  const int64_t n_tiles = Nout / HB;
  const int64_t pairs_needed = ((A + kRpBM - 1) / kRpBM + s->N) * n_tiles;
  const int64_t max_pairs = num_sms() / 2;
  const int64_t pairs = pairs_needed < max_pairs ? pairs_needed : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kRpThreads, 1, 1);
  cfg.dynamicSmemBytes = kRpSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, ma, mb0, mb1, offsets, s->N, static_cast<int>(A), K, Nout,
                         static_cast<__nv_bfloat16*>(out), ldo, kWaitTimeoutNs) != cudaSuccess)
    return MOE_ERR_CUDA;
  return launched();
}

template <int EPI>
moe_status launch_tc_swap(const moe_shape* s, const RowSource& src, int K, const void* w0, const void* w1, int Nout,
                          const int32_t* offsets, void* out, int ldo, cudaStream_t st, int mode, int* tile_counter) {
  // auto and "pairs" run token tiles on SM pairs, "tokens" on single SMs
  if (mode == MOE_TILING_TOKENS)
    return launch_tc_swap_bk<EPI, kTcBK>(s, src, K, w0, w1, Nout, offsets, out, ldo, st);
  return launch_tc_pair<EPI>(s, src, K, w0, w1, Nout, offsets, out, ldo, st, tile_counter);
}

// K is the reduction length of the GEMM in question (d for the first, F for
// the second). Token tiles pad less but keep one accumulator pair in TMEM, so
// their epilogue is not overlapped with the next tile: they pay off when an
// expert holds enough rows to fill tiles and K is long enough to hide it.
bool use_token_tiles(const moe_shape* s, int K, int mode) {
  if (mode == MOE_TILING_TOKENS || mode == MOE_TILING_PAIRS) return true;
  if (mode == MOE_TILING_ROWS || mode == MOE_TILING_ROW_PAIRS) return false;
  return n_assign(s) >= static_cast<int64_t>(kAutoTokenTileMinRowsPerExpert) * s->N && K >= kAutoTokenTileMinK;
}

// Row tiles on SM pairs (MOE_TILING_ROW_PAIRS only), where their output
// columns divide the GEMM's and its rows are the permuted copy. Auto does not
// take them: on the skewed batch they are within 1-2 % of row tiles (581 + 374
// against 589 + 379 us per launch), with a capacity of 1.25 on the same batch
// 6 % slower (most experts then hold few rows, and a 256-row tile of them is
// mostly padding), on decode 8 % slower.
bool use_row_pairs(int mode, int cols, int tile_cols, bool permuted) {
  return mode == MOE_TILING_ROW_PAIRS && permuted && cols % tile_cols == 0;
}

template <int EPI>
moe_status launch_simt(const moe_shape* s, const void* a, int K, const void* b0, const void* b1, int Nout,
                       const int32_t* offsets, void* out, int ldo, cudaStream_t st) {
  const int64_t A = n_assign(s);
  dim3 grid(static_cast<unsigned>((A + kSimtBM - 1) / kSimtBM + s->N),
            static_cast<unsigned>((Nout + kSimtBN - 1) / kSimtBN));
  grouped_gemm_simt_kernel<EPI><<<grid, 256, 0, st>>>(static_cast<const float*>(a), offsets, s->N,
                                                      static_cast<int>(A), static_cast<const float*>(b0),
                                                      static_cast<const float*>(b1), K, Nout,
                                                      static_cast<float*>(out), ldo);
  return launched();
}

// The grouped FFN: h = act(x W_1^T) per expert (the first GEMM), y = h W_2^T
// (the second). src gives the first GEMM's token rows: the permuted rows
// x_perm [A, d], or (bf16 only) the tokens x gathered through perm.
// tiling: a moe_tiling value for this call, or -1 for the process-wide setting
// (moe_set_ffn_tiling), read once per call so both GEMMs see the same mode.
moe_status ffn_impl(const moe_shape* s, const RowSource& src, const int32_t* offsets, const void* w_gate,
                    const void* w_up, const void* w_down, void* y_perm, void* ws, cudaStream_t st,
                    int tiling = -1) {
  if (n_assign(s) == 0) return MOE_OK;
  const int d = s->d, F = s->d_ff;
  const int mode = tiling >= 0 ? tiling : g_ffn_tiling.load(std::memory_order_relaxed);
  void* h = ws;
  const RowSource hs{h, nullptr, 0};
  int* ctr = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + ffn_h_bytes(s));
  moe_status r;
  if (s->dtype == MOE_BF16) {
    const bool rp1 = use_row_pairs(mode, F, s->act == MOE_SWIGLU ? rp_tile_cols<EPI_SWIGLU>() : rp_tile_cols<EPI_GELU>(),
                                   src.perm == nullptr);
    const bool rp2 = use_row_pairs(mode, d, rp_tile_cols<EPI_PLAIN>(), true);
    if (rp1)
      r = (s->act == MOE_SWIGLU) ? launch_tc_rowpair<EPI_SWIGLU>(s, src.a, d, w_gate, w_up, F, offsets, h, F, st)
                                 : launch_tc_rowpair<EPI_GELU>(s, src.a, d, w_gate, nullptr, F, offsets, h, F, st);
    else if (use_token_tiles(s, d, mode))
      r = (s->act == MOE_SWIGLU)
              ? launch_tc_swap<EPI_SWIGLU>(s, src, d, w_gate, w_up, F, offsets, h, F, st, mode, ctr)
              : launch_tc_swap<EPI_GELU>(s, src, d, w_gate, nullptr, F, offsets, h, F, st, mode, ctr);
    else if (s->act == MOE_SWIGLU)
      r = (F % 128 == 0) ? launch_tc<256, EPI_SWIGLU>(s, src, d, w_gate, w_up, F, offsets, h, F, st)
                         : launch_tc<128, EPI_SWIGLU>(s, src, d, w_gate, w_up, F, offsets, h, F, st);
    else
      r = (F % 256 == 0) ? launch_tc<256, EPI_GELU>(s, src, d, w_gate, nullptr, F, offsets, h, F, st)
                         : launch_tc<128, EPI_GELU>(s, src, d, w_gate, nullptr, F, offsets, h, F, st);
    if (r != MOE_OK) return r;
    if (rp2) return launch_tc_rowpair<EPI_PLAIN>(s, h, F, w_down, nullptr, d, offsets, y_perm, d, st);
    if (use_token_tiles(s, F, mode))
      return launch_tc_swap<EPI_PLAIN>(s, hs, F, w_down, nullptr, d, offsets, y_perm, d, st, mode, ctr);
    return (d % 256 == 0) ? launch_tc<256, EPI_PLAIN>(s, hs, F, w_down, nullptr, d, offsets, y_perm, d, st)
                          : launch_tc<128, EPI_PLAIN>(s, hs, F, w_down, nullptr, d, offsets, y_perm, d, st);
  }
  if (src.perm != nullptr) return MOE_ERR_UNSUPPORTED;    // fp32: the rows are always permuted first
  r = (s->act == MOE_SWIGLU) ? launch_simt<EPI_SWIGLU>(s, src.a, d, w_gate, w_up, F, offsets, h, F, st)
                             : launch_simt<EPI_GELU>(s, src.a, d, w_gate, nullptr, F, offsets, h, F, st);
  if (r != MOE_OK) return r;
  return launch_simt<EPI_PLAIN>(s, h, F, w_down, nullptr, d, offsets, y_perm, d, st);
}

// ---------------------------------------------------------------- combine
moe_status combine_impl(const moe_shape* s, const void* y_perm, const int32_t* inv_perm, const float* topk_w,
                        void* out, cudaStream_t st) {
  if (s->T == 0) return MOE_OK;
  constexpr int CPT = 2;
  const int nchunk = s->d / (s->dtype == MOE_BF16 ? 8 : 4);
  const int64_t warps = s->T * combine_groups<CPT>(nchunk);
  const int64_t grid = (warps + kCombineThreads / 32 - 1) / (kCombineThreads / 32);
  auto go = [&](auto kmax) {
    constexpr int KMAX = decltype(kmax)::value;
    if (s->dtype == MOE_BF16)
      combine_kernel<__nv_bfloat16, CPT, KMAX><<<static_cast<unsigned>(grid), kCombineThreads, 0, st>>>(
          static_cast<const __nv_bfloat16*>(y_perm), inv_perm, topk_w, s->T, s->d, s->k, n_assign(s),
          static_cast<__nv_bfloat16*>(out));
    else
      combine_kernel<float, CPT, KMAX><<<static_cast<unsigned>(grid), kCombineThreads, 0, st>>>(
          static_cast<const float*>(y_perm), inv_perm, topk_w, s->T, s->d, s->k, n_assign(s),
          static_cast<float*>(out));
    return launched();
  };
  if (s->k <= 2) return go(std::integral_constant<int, 2>{});
  if (s->k <= 4) return go(std::integral_constant<int, 4>{});
  if (s->k <= 8) return go(std::integral_constant<int, 8>{});
  return go(std::integral_constant<int, 0>{});
}

moe_status forward_impl(const moe_shape* s, const void* x, const float* wg, const float* bias, const void* w_gate,
                        const void* w_up, const void* w_down, void* out, int32_t* topk_idx, float* topk_w,
                        int32_t* counts, const FwdBufs& b, cudaStream_t st, const FwdOpts& o = FwdOpts{}) {
  int32_t* idx = topk_idx ? topk_idx : b.topk_idx;
  float* w = topk_w ? topk_w : b.topk_w;
  int32_t* cnt = counts ? counts : b.counts;
  moe_status r = route_impl(s, x, wg, bias, idx, w, st, o.bias_select, o.load_stats, b.stats_ws);
  if (r != MOE_OK) return r;
  // the grouping writes the permuted copy x_perm, which the first grouped GEMM
  // reads in whole tiles: measured faster than gathering the rows of x in the
  // GEMM (moe_grouped_ffn_gather), whose per-row loads slow the weight stream
  r = permute_impl(s, idx, x, cnt, b.offsets, b.perm, b.inv_perm, b.x_perm, b.perm_ws, st, o.capacity, o.dropped);
  if (r != MOE_OK) return r;
  r = ffn_impl(s, RowSource{b.x_perm, nullptr, 0}, b.offsets, w_gate, w_up, w_down, b.y_perm, b.ffn_ws, st,
               o.tiling);
  if (r != MOE_OK) return r;
  return combine_impl(s, b.y_perm, b.inv_perm, w, out, st);
}

// ---------------------------------------------------------------- expert choice
// Shapes of the expert-choice path: C tokens per expert, N*C rows; every
// token has N (row, weight) slots, so the row copy and the combine run as a
// top-k with k = N.
moe_status ec_shape_status(const moe_shape* s, int64_t C) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  if (C < 0 || C > s->T) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(s->N) * C >= (int64_t(1) << 31) || s->T * s->N >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_shape ec_ffn_shape(const moe_shape* s, int64_t C) {
  moe_shape f = *s;
  f.T = static_cast<int64_t>(s->N) * C;
  f.k = 1;
  return f;
}

moe_shape ec_slot_shape(const moe_shape* s) {
  moe_shape c = *s;
  c.k = s->N;
  return c;
}

struct EcBufs {
  float* probs;
  int32_t* inv;
  float* w;
  int32_t* perm;
  int32_t* counts;
  int32_t* offsets;
  void* x_perm;
  void* y_perm;
  void* ffn_ws;
  size_t total;
};

EcBufs carve_ec(const moe_shape* s, int64_t C, void* ws) {
  Carve c(ws);
  EcBufs b{};
  const size_t TN = static_cast<size_t>(s->T) * s->N;
  const size_t rows = static_cast<size_t>(s->N) * C;
  const moe_shape f = ec_ffn_shape(s, C);
  b.probs = c.take<float>(sizeof(float) * TN);
  b.inv = c.take<int32_t>(sizeof(int32_t) * TN);
  b.w = c.take<float>(sizeof(float) * TN);
  b.perm = c.take<int32_t>(sizeof(int32_t) * rows);
  b.counts = c.take<int32_t>(sizeof(int32_t) * s->N);
  b.offsets = c.take<int32_t>(sizeof(int32_t) * (s->N + 1));
  b.x_perm = c.take<uint8_t>(esize(s) * rows * s->d);
  b.y_perm = c.take<uint8_t>(esize(s) * rows * s->d);
  b.ffn_ws = c.take<uint8_t>(ffn_ws(&f));
  b.total = c.used;
  return b;
}

moe_status ec_route_impl(const moe_shape* s, int64_t C, const void* x, const float* wg, const float* bias,
                         float* probs, int32_t* perm, int32_t* counts, int32_t* offsets, int32_t* inv, float* w,
                         cudaStream_t st) {
  RouteArgs a{wg, bias, 0, nullptr, nullptr, nullptr, 0, probs};
  moe_status r = s->dtype == MOE_BF16
                     ? launch_route<__nv_bfloat16>(s, static_cast<const __nv_bfloat16*>(x), a, st)
                     : launch_route<float>(s, static_cast<const float*>(x), a, st);
  if (r != MOE_OK) return r;
  ec_select_kernel<<<static_cast<unsigned>(s->N), kEcThreads, 0, st>>>(probs, s->T, s->N, C, perm, counts, offsets,
                                                                       inv, w);
  return launched();
}

moe_status ec_forward_impl(const moe_shape* s, int64_t C, const void* x, const float* wg, const float* bias,
                           const void* w_gate, const void* w_up, const void* w_down, void* out, const EcBufs& b,
                           cudaStream_t st) {
  moe_status r = ec_route_impl(s, C, x, wg, bias, b.probs, b.perm, b.counts, b.offsets, b.inv, b.w, st);
  if (r != MOE_OK) return r;
  const moe_shape slots = ec_slot_shape(s);
  const moe_shape f = ec_ffn_shape(s, C);
  r = launch_row_copy(s, b.inv, x, s->N, f.T, b.x_perm, st);
  if (r != MOE_OK) return r;
  r = ffn_impl(&f, RowSource{b.x_perm, nullptr, 0}, b.offsets, w_gate, w_up, w_down, b.y_perm, b.ffn_ws, st);
  if (r != MOE_OK) return r;
  return combine_impl(&slots, b.y_perm, b.inv, b.w, out, st);
}

bool weights_ok(const moe_shape* s, const void* w_gate, const void* w_up, const void* w_down) {
  if (!ptr_ok(w_gate, true) || !ptr_ok(w_down, true)) return false;
  if (s->act == MOE_SWIGLU) return ptr_ok(w_up, true);
  return w_up == nullptr;
}

// ---------------------------------------------------------------- expert parallelism
moe_status ep_args_status(int32_t G, int32_t E, int64_t rows, int32_t d, int32_t dtype) {
  if (G < 1 || E < 1 || rows < 0 || d < 1) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(G) * E > kEpMaxTable || rows >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  if ((static_cast<int64_t>(d) * (dtype == MOE_F32 ? 4 : 2)) % 16 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

unsigned ep_grid(int64_t rows) {
  const int64_t per = kEpThreads / 32;
  const int64_t want = (rows + per - 1) / per;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  return static_cast<unsigned>(want < 1 ? 1 : (want < cap ? want : cap));
}

__global__ void bounded_wait_selftest_kernel(unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(smem_addr(&bar), 0u, &abort_flag, timeout_ns);   // nothing arrives
  __syncthreads();
}

}  // namespace

extern "C" {

moe_status moe_check_shape(const moe_shape* s) { return shape_status(s); }

size_t moe_permute_workspace_size(const moe_shape* s) { return shape_status(s) == MOE_OK ? permute_ws(s) : 0; }

size_t moe_grouped_ffn_workspace_size(const moe_shape* s) { return shape_status(s) == MOE_OK ? ffn_ws(s) : 0; }

size_t moe_workspace_size(const moe_shape* s) {
  return shape_status(s) == MOE_OK ? carve_forward(s, nullptr, false).total : 0;
}

size_t moe_forward_hostio_workspace_size(const moe_shape* s) {
  return shape_status(s) == MOE_OK ? carve_forward(s, nullptr, true).total : 0;
}

moe_status moe_route(const moe_shape* s, const void* x, const float* w_g, const float* bias, int32_t* topk_idx,
                     float* topk_w, void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  const bool any = s->T > 0;
  if (!ptr_ok(x, any) || !ptr_ok(w_g, true) || !ptr_ok(bias, false) || !ptr_ok(topk_idx, any) ||
      !ptr_ok(topk_w, any))
    return MOE_ERR_INVALID_ARG;
  return route_impl(s, x, w_g, bias, topk_idx, topk_w, static_cast<cudaStream_t>(stream));
}

size_t moe_route_ex_workspace_size(const moe_shape* s) { return shape_status(s) == MOE_OK ? route_stats_ws(s) : 0; }

moe_status moe_route_ex(const moe_shape* s, const void* x, const float* w_g, const float* bias, int32_t bias_mode,
                        int32_t* topk_idx, float* topk_w, float* load_stats, void* ws, size_t ws_bytes,
                        void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  if (bias_mode != MOE_BIAS_LOGITS && bias_mode != MOE_BIAS_SELECT) return MOE_ERR_INVALID_ARG;
  const bool any = s->T > 0;
  const bool stats = load_stats != nullptr;
  if (!ptr_ok(x, any) || !ptr_ok(w_g, true) || !ptr_ok(bias, false) || !ptr_ok(topk_idx, any) ||
      !ptr_ok(topk_w, any) || !ptr_ok(load_stats, false) || !ptr_ok(ws, stats && any))
    return MOE_ERR_INVALID_ARG;
  if (stats && ws_bytes < route_stats_ws(s)) return MOE_ERR_WORKSPACE;
  return route_impl(s, x, w_g, bias, topk_idx, topk_w, static_cast<cudaStream_t>(stream),
                    bias_mode == MOE_BIAS_SELECT ? 1 : 0, load_stats, ws);
}

moe_status moe_permute(const moe_shape* s, const int32_t* topk_idx, const void* x, int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* x_perm, void* ws, size_t ws_bytes,
                       void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  const bool any = s->T > 0;
  // x_perm may be NULL: the indices only (the grouped GEMM can gather the rows itself)
  if (!ptr_ok(topk_idx, any) || !ptr_ok(x, any && x_perm != nullptr) || !ptr_ok(counts, true) ||
      !ptr_ok(offsets, true) || !ptr_ok(perm, any) || !ptr_ok(inv_perm, any) || !ptr_ok(x_perm, false) ||
      !ptr_ok(ws, permute_ws(s) > 0))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < permute_ws(s)) return MOE_ERR_WORKSPACE;
  return permute_impl(s, topk_idx, x, counts, offsets, perm, inv_perm, x_perm, ws, static_cast<cudaStream_t>(stream));
}

moe_status moe_permute_capacity(const moe_shape* s, const int32_t* topk_idx, const void* x, double capacity_factor,
                                int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* x_perm,
                                int32_t* dropped, void* ws, size_t ws_bytes, void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  if (!(capacity_factor >= 0.0)) return MOE_ERR_INVALID_ARG;
  const bool any = s->T > 0;
  // x_perm may be NULL: the indices only (as moe_permute)
  if (!ptr_ok(topk_idx, any) || !ptr_ok(x, any && x_perm != nullptr) || !ptr_ok(counts, true) ||
      !ptr_ok(offsets, true) || !ptr_ok(perm, any) || !ptr_ok(inv_perm, any) || !ptr_ok(x_perm, false) ||
      !ptr_ok(dropped, false) || !ptr_ok(ws, permute_ws(s) > 0))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < permute_ws(s)) return MOE_ERR_WORKSPACE;
  return permute_impl(s, topk_idx, x, counts, offsets, perm, inv_perm, x_perm, ws, static_cast<cudaStream_t>(stream),
                      capacity_rows(s, capacity_factor), dropped);
}

moe_status moe_grouped_ffn(const moe_shape* s, const void* x_perm, const int32_t* offsets, const void* w_gate,
                           const void* w_up, const void* w_down, void* y_perm, void* ws, size_t ws_bytes,
                           void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  const bool any = s->T > 0;
  if (!ptr_ok(x_perm, any) || !ptr_ok(offsets, true) || !weights_ok(s, w_gate, w_up, w_down) ||
      !ptr_ok(y_perm, any) || !ptr_ok(ws, ffn_ws(s) > 0))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ffn_ws(s)) return MOE_ERR_WORKSPACE;
  return ffn_impl(s, RowSource{x_perm, nullptr, 0}, offsets, w_gate, w_up, w_down, y_perm, ws,
                  static_cast<cudaStream_t>(stream));
}

moe_status moe_grouped_ffn_gather(const moe_shape* s, const void* x, const int32_t* perm, const int32_t* offsets,
                                  const void* w_gate, const void* w_up, const void* w_down, void* y_perm, void* ws,
                                  size_t ws_bytes, void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  if (s->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  const bool any = s->T > 0;
  if (!ptr_ok(x, any) || !ptr_ok(perm, any) || !ptr_ok(offsets, true) || !weights_ok(s, w_gate, w_up, w_down) ||
      !ptr_ok(y_perm, any) || !ptr_ok(ws, ffn_ws(s) > 0))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ffn_ws(s)) return MOE_ERR_WORKSPACE;
  return ffn_impl(s, RowSource{x, perm, s->T}, offsets, w_gate, w_up, w_down, y_perm, ws,
                  static_cast<cudaStream_t>(stream));
}

moe_status moe_combine(const moe_shape* s, const void* y_perm, const int32_t* inv_perm, const float* topk_w,
                       void* out, void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  const bool any = s->T > 0;
  if (!ptr_ok(y_perm, any) || !ptr_ok(inv_perm, any) || !ptr_ok(topk_w, any) || !ptr_ok(out, any))
    return MOE_ERR_INVALID_ARG;
  return combine_impl(s, y_perm, inv_perm, topk_w, out, static_cast<cudaStream_t>(stream));
}

moe_status moe_forward(const moe_shape* s, const void* x, const float* w_g, const float* bias, const void* w_gate,
                       const void* w_up, const void* w_down, void* out, int32_t* topk_idx, float* topk_w,
                       int32_t* counts, void* ws, size_t ws_bytes, void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  const bool any = s->T > 0;
  if (!ptr_ok(x, any) || !ptr_ok(w_g, true) || !ptr_ok(bias, false) || !weights_ok(s, w_gate, w_up, w_down) ||
      !ptr_ok(out, any) || !ptr_ok(topk_idx, false) || !ptr_ok(topk_w, false) || !ptr_ok(counts, false) ||
      !ptr_ok(ws, true))
    return MOE_ERR_INVALID_ARG;
  const FwdBufs b = carve_forward(s, ws, false);
  if (ws_bytes < b.total) return MOE_ERR_WORKSPACE;
  return forward_impl(s, x, w_g, bias, w_gate, w_up, w_down, out, topk_idx, topk_w, counts, b,
                      static_cast<cudaStream_t>(stream));
}

moe_status moe_forward_capacity(const moe_shape* s, double capacity_factor, const void* x, const float* w_g,
                                const float* bias, const void* w_gate, const void* w_up, const void* w_down,
                                void* out, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* dropped,
                                void* ws, size_t ws_bytes, void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  if (!(capacity_factor >= 0.0)) return MOE_ERR_INVALID_ARG;
  const bool any = s->T > 0;
  if (!ptr_ok(x, any) || !ptr_ok(w_g, true) || !ptr_ok(bias, false) || !weights_ok(s, w_gate, w_up, w_down) ||
      !ptr_ok(out, any) || !ptr_ok(topk_idx, false) || !ptr_ok(topk_w, false) || !ptr_ok(counts, false) ||
      !ptr_ok(dropped, false) || !ptr_ok(ws, true))
    return MOE_ERR_INVALID_ARG;
  const FwdBufs b = carve_forward(s, ws, false);
  if (ws_bytes < b.total) return MOE_ERR_WORKSPACE;
  FwdOpts o;
  o.capacity = capacity_rows(s, capacity_factor);
  o.dropped = dropped;
  return forward_impl(s, x, w_g, bias, w_gate, w_up, w_down, out, topk_idx, topk_w, counts, b,
                      static_cast<cudaStream_t>(stream), o);
}

moe_status moe_forward_ex(const moe_shape* s, const moe_options* opt, const void* x, const float* w_g,
                          const float* bias, const void* w_gate, const void* w_up, const void* w_down, void* out,
                          int32_t* topk_idx, float* topk_w, int32_t* counts, void* ws, size_t ws_bytes,
                          void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  FwdOpts o;
  if (opt != nullptr) {
    if (opt->bias_mode != MOE_BIAS_LOGITS && opt->bias_mode != MOE_BIAS_SELECT) return MOE_ERR_INVALID_ARG;
    if (opt->use_capacity && !(opt->capacity_factor >= 0.0)) return MOE_ERR_INVALID_ARG;
    if (!ptr_ok(opt->load_stats, false) || !ptr_ok(opt->dropped, false)) return MOE_ERR_INVALID_ARG;
    if (opt->use_tiling && !tiling_valid(opt->ffn_tiling)) return MOE_ERR_INVALID_ARG;
    if (opt->use_tiling) o.tiling = opt->ffn_tiling;
    o.bias_select = opt->bias_mode == MOE_BIAS_SELECT ? 1 : 0;
    if (opt->use_capacity) o.capacity = capacity_rows(s, opt->capacity_factor);
    o.load_stats = opt->load_stats;
    o.dropped = opt->dropped;
  }
  const bool any = s->T > 0;
  if (!ptr_ok(x, any) || !ptr_ok(w_g, true) || !ptr_ok(bias, false) || !weights_ok(s, w_gate, w_up, w_down) ||
      !ptr_ok(out, any) || !ptr_ok(topk_idx, false) || !ptr_ok(topk_w, false) || !ptr_ok(counts, false) ||
      !ptr_ok(ws, true))
    return MOE_ERR_INVALID_ARG;
  const FwdBufs b = carve_forward(s, ws, false);
  if (ws_bytes < b.total) return MOE_ERR_WORKSPACE;
  return forward_impl(s, x, w_g, bias, w_gate, w_up, w_down, out, topk_idx, topk_w, counts, b,
                      static_cast<cudaStream_t>(stream), o);
}

moe_status moe_gather_rows(const moe_shape* s, const int32_t* inv, int32_t slots, int64_t rows, const void* x,
                           void* x_perm, void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  if (slots < 1 || rows < 0 || s->T * static_cast<int64_t>(slots) >= (int64_t(1) << 31)) return MOE_ERR_INVALID_ARG;
  const bool any = s->T > 0;
  if (!ptr_ok(inv, any) || !ptr_ok(x, any) || !ptr_ok(x_perm, any && rows > 0)) return MOE_ERR_INVALID_ARG;
  return launch_row_copy(s, inv, x, slots, rows, x_perm, static_cast<cudaStream_t>(stream));
}

size_t moe_expert_choice_workspace_size(const moe_shape* s, int64_t C) {
  return ec_shape_status(s, C) == MOE_OK ? carve_ec(s, C, nullptr).total : 0;
}

moe_status moe_route_expert_choice(const moe_shape* s, int64_t C, const void* x, const float* w_g, const float* bias,
                                   float* probs, int32_t* perm, int32_t* counts, int32_t* offsets, int32_t* inv,
                                   float* w, void* stream) {
  moe_status st = ec_shape_status(s, C);
  if (st != MOE_OK) return st;
  const bool any = s->T > 0;
  if (!ptr_ok(x, any) || !ptr_ok(w_g, true) || !ptr_ok(bias, false) || !ptr_ok(probs, any) ||
      !ptr_ok(perm, C > 0) || !ptr_ok(counts, true) || !ptr_ok(offsets, true) || !ptr_ok(inv, any) ||
      !ptr_ok(w, any))
    return MOE_ERR_INVALID_ARG;
  return ec_route_impl(s, C, x, w_g, bias, probs, perm, counts, offsets, inv, w, static_cast<cudaStream_t>(stream));
}

moe_status moe_forward_expert_choice(const moe_shape* s, int64_t C, const void* x, const float* w_g,
                                     const float* bias, const void* w_gate, const void* w_up, const void* w_down,
                                     void* out, int32_t* counts, void* ws, size_t ws_bytes, void* stream) {
  moe_status st = ec_shape_status(s, C);
  if (st != MOE_OK) return st;
  const bool any = s->T > 0;
  if (!ptr_ok(x, any) || !ptr_ok(w_g, true) || !ptr_ok(bias, false) || !weights_ok(s, w_gate, w_up, w_down) ||
      !ptr_ok(out, any) || !ptr_ok(counts, false) || !ptr_ok(ws, true))
    return MOE_ERR_INVALID_ARG;
  EcBufs b = carve_ec(s, C, ws);
  if (ws_bytes < b.total) return MOE_ERR_WORKSPACE;
  if (counts != nullptr) b.counts = counts;
  return ec_forward_impl(s, C, x, w_g, bias, w_gate, w_up, w_down, out, b, static_cast<cudaStream_t>(stream));
}

moe_status moe_forward_hostio(const moe_shape* s, const void* x_host, const float* w_g, const float* bias,
                              const void* w_gate, const void* w_up, const void* w_down, void* out_host, void* ws,
                              size_t ws_bytes, void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  const bool any = s->T > 0;
  if ((any && (x_host == nullptr || out_host == nullptr)) || !ptr_ok(w_g, true) || !ptr_ok(bias, false) ||
      !weights_ok(s, w_gate, w_up, w_down) || !ptr_ok(ws, true))
    return MOE_ERR_INVALID_ARG;
  const FwdBufs b = carve_forward(s, ws, true);
  if (ws_bytes < b.total) return MOE_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const size_t bytes = esize(s) * static_cast<size_t>(s->T) * s->d;
  if (any && cudaMemcpyAsync(b.x_dev, x_host, bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess) return MOE_ERR_CUDA;
  st = forward_impl(s, b.x_dev, w_g, bias, w_gate, w_up, w_down, b.out_dev, nullptr, nullptr, nullptr, b, cs);
  if (st != MOE_OK) return st;
  if (any && cudaMemcpyAsync(out_host, b.out_dev, bytes, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// ---------------------------------------------------------------- pipelined host I/O
// Workspace of moe_forward_hostio_pipelined: the forward's buffers, then two
// slots of (x, out) device copies.
struct PipeBufs {
  FwdBufs f;
  void* x_slot[2];
  void* out_slot[2];
  size_t total;
};

PipeBufs carve_pipelined(const moe_shape* s, void* ws) {
  PipeBufs p{};
  p.f = carve_forward(s, ws, false);
  Carve c(ws);
  c.used = p.f.total;
  const size_t io = esize(s) * static_cast<size_t>(s->T) * s->d;
  for (int b = 0; b < 2; ++b) {
    p.x_slot[b] = c.take<uint8_t>(io);
    p.out_slot[b] = c.take<uint8_t>(io);
  }
  p.total = c.used;
  return p;
}

// Per device and slot: x copied in, x no longer read, out written, out copied
// back. Created on first use, kept for the life of the process.
struct PipeEvents {
  cudaEvent_t in_ready[2], in_free[2], out_ready[2], out_free[2];
  bool made = false;
};

PipeEvents* pipe_events() {
  static PipeEvents ev[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  PipeEvents& e = ev[dev];
  if (!e.made) {
    for (int b = 0; b < 2; ++b) {
      cudaEvent_t* all[4] = {&e.in_ready[b], &e.in_free[b], &e.out_ready[b], &e.out_free[b]};
      for (cudaEvent_t* x : all)
        if (cudaEventCreateWithFlags(x, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    }
    e.made = true;
  }
  return &e;
}

size_t moe_forward_hostio_pipelined_workspace_size(const moe_shape* s) {
  return shape_status(s) == MOE_OK ? carve_pipelined(s, nullptr).total : 0;
}

moe_status moe_forward_hostio_pipelined(const moe_shape* s, const void* x_host, const float* w_g, const float* bias,
                                        const void* w_gate, const void* w_up, const void* w_down, void* out_host,
                                        void* ws, size_t ws_bytes, int32_t slot, void* compute_stream,
                                        void* h2d_stream, void* d2h_stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  const bool any = s->T > 0;
  if (slot != 0 && slot != 1) return MOE_ERR_INVALID_ARG;
  if ((any && (x_host == nullptr || out_host == nullptr)) || !ptr_ok(w_g, true) || !ptr_ok(bias, false) ||
      !weights_ok(s, w_gate, w_up, w_down) || !ptr_ok(ws, true))
    return MOE_ERR_INVALID_ARG;
  const PipeBufs p = carve_pipelined(s, ws);
  if (ws_bytes < p.total) return MOE_ERR_WORKSPACE;
  PipeEvents* ev = pipe_events();
  if (ev == nullptr) return MOE_ERR_CUDA;
  cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
  cudaStream_t in = static_cast<cudaStream_t>(h2d_stream);
  cudaStream_t out = static_cast<cudaStream_t>(d2h_stream);
  const size_t bytes = esize(s) * static_cast<size_t>(s->T) * s->d;
  const int b = slot;
  // copy in, once the call two steps back has finished reading this slot's x
  if (cudaStreamWaitEvent(in, ev->in_free[b], 0) != cudaSuccess) return MOE_ERR_CUDA;
  if (any && cudaMemcpyAsync(p.x_slot[b], x_host, bytes, cudaMemcpyHostToDevice, in) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaEventRecord(ev->in_ready[b], in) != cudaSuccess) return MOE_ERR_CUDA;
  // the layer, once x is in and this slot's previous output has been copied out
  if (cudaStreamWaitEvent(cs, ev->in_ready[b], 0) != cudaSuccess ||
      cudaStreamWaitEvent(cs, ev->out_free[b], 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  st = forward_impl(s, p.x_slot[b], w_g, bias, w_gate, w_up, w_down, p.out_slot[b], nullptr, nullptr, nullptr, p.f,
                    cs);
  if (st != MOE_OK) return st;
  if (cudaEventRecord(ev->in_free[b], cs) != cudaSuccess || cudaEventRecord(ev->out_ready[b], cs) != cudaSuccess)
    return MOE_ERR_CUDA;
  // copy out
  if (cudaStreamWaitEvent(out, ev->out_ready[b], 0) != cudaSuccess) return MOE_ERR_CUDA;
  if (any && cudaMemcpyAsync(out_host, p.out_slot[b], bytes, cudaMemcpyDeviceToHost, out) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaEventRecord(ev->out_free[b], out) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

// ---------------------------------------------------------------- permute without a workspace
// Chunk-histogram scratch of moe_permute_noalloc. Host code must not pass this
// name to a kernel (on the host it is only a stand-in for the symbol): the
// device address comes from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) int32_t g_permute_noalloc_scratch[MOE_PERMUTE_NOALLOC_SCRATCH_INTS];

// The current device's address of the scratch array, looked up on the first
// call on that device (with the device current) and cached under a mutex, so
// host threads that make their first calls together are safe. The cache is not
// refreshed after cudaDeviceReset: the library is not usable across a reset.
static void* noalloc_scratch_address() {
  static void* addr[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

moe_status moe_permute_noalloc(const moe_shape* s, const int32_t* topk_idx, const void* x, int32_t* counts,
                               int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* x_perm, void* stream) {
  moe_status st = shape_status(s);
  if (st != MOE_OK) return st;
  const bool any = s->T > 0;
  if (!ptr_ok(topk_idx, any) || !ptr_ok(x, any) || !ptr_ok(counts, true) || !ptr_ok(offsets, true) ||
      !ptr_ok(perm, any) || !ptr_ok(inv_perm, any) || !ptr_ok(x_perm, any))
    return MOE_ERR_INVALID_ARG;
  if (perm_chunks(s) * s->N > MOE_PERMUTE_NOALLOC_SCRATCH_INTS) return MOE_ERR_WORKSPACE;
  void* scratch = noalloc_scratch_address();
  if (scratch == nullptr) return MOE_ERR_CUDA;
  return permute_impl(s, topk_idx, x, counts, offsets, perm, inv_perm, x_perm, scratch,
                      static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- expert parallelism
moe_status moe_ep_regroup(int32_t G, int32_t E, const int32_t* recv_counts, int64_t rows, int32_t d, int32_t dtype,
                          const void* recv_x, void* x_local, int32_t* offsets_local, int32_t* local_src,
                          void* stream) {
  moe_status st = ep_args_status(G, E, rows, d, dtype);
  if (st != MOE_OK) return st;
  const bool any = rows > 0;
  if (!ptr_ok(recv_counts, true) || !ptr_ok(recv_x, any) || !ptr_ok(x_local, any) || !ptr_ok(offsets_local, true) ||
      !ptr_ok(local_src, any))
    return MOE_ERR_INVALID_ARG;
  const int64_t nv = static_cast<int64_t>(d) * (dtype == MOE_F32 ? 4 : 2) / 16;
  ep_regroup_kernel<<<ep_grid(rows), kEpThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      recv_counts, G, E, rows, nv, static_cast<const uint4*>(recv_x), static_cast<uint4*>(x_local), offsets_local,
      local_src);
  return launched();
}

moe_status moe_ep_ungroup(int64_t rows, int32_t d, int32_t dtype, const int32_t* local_src, const void* y_local,
                          void* y_recv, void* stream) {
  moe_status st = ep_args_status(1, 1, rows, d, dtype);
  if (st != MOE_OK) return st;
  if (rows == 0) return MOE_OK;
  if (!ptr_ok(local_src, true) || !ptr_ok(y_local, true) || !ptr_ok(y_recv, true)) return MOE_ERR_INVALID_ARG;
  const int64_t nv = static_cast<int64_t>(d) * (dtype == MOE_F32 ? 4 : 2) / 16;
  ep_ungroup_kernel<<<ep_grid(rows), kEpThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      local_src, rows, nv, static_cast<const uint4*>(y_local), static_cast<uint4*>(y_recv));
  return launched();
}

moe_status moe_set_ffn_tiling(int mode) {
  if (!tiling_valid(mode)) return MOE_ERR_INVALID_ARG;
  g_ffn_tiling.store(mode, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_get_ffn_tiling(void) { return g_ffn_tiling.load(std::memory_order_relaxed); }

moe_status moe_get_error(void* stream) {
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  int* word = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&word), g_error_word) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyAsync(&v, word, sizeof(int), cudaMemcpyDeviceToHost, cs) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(word, 0, sizeof(int), cs) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(cs) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status>(v);
}

moe_status moe_selftest_bounded_wait(int64_t timeout_ns, void* stream) {
  if (timeout_ns < 1000000) timeout_ns = 1000000;
  if (timeout_ns > 2000000000) timeout_ns = 2000000000;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned long long>(timeout_ns));
  return launched();
}

const char* moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_CORRUPT: return "corrupt routing data";
  }
  return "unknown status";
}

int moe_version(void) { return 100; }

}  // extern "C"
