/*
 * moe.h -- C ABI of libmoe_b300.so: the forward pass of one Mixture-of-Experts
 * layer on one NVIDIA B300 (sm_103a).
 *
 * The layer, as the pages define it:
 *   "MoE显存与计算开销四阶段手算指南" section 2 (four stages: gate projection,
 *   routing, grouped expert computation, weighted combine) and
 *   "MoE混合专家模型计算原理与推理部署实战解析" sections 2.1-2.2 (gate, softmax,
 *   top-k, renormalised gates, weighted sum), 3.1 (SwiGLU expert) and 5.1
 *   (count -> prefix sum -> permute -> grouped GEMM -> unpermute + merge).
 *
 * Conventions for every call:
 *   - Tensors are dense, row-major and live in DEVICE memory owned by the
 *     caller; pointers must be 16-byte aligned. The library never allocates
 *     or frees device memory (scratch comes from the caller's workspace) and
 *     never synchronises, except moe_get_error.
 *   - All work is queued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns before it runs.
 *   - Argument errors are detected on the host and return a status before
 *     anything is launched. Launch failures return MOE_ERR_CUDA. Errors found
 *     by the kernels (an expert index out of range, offsets that do not add
 *     up, a device-side wait that ran out) are recorded in a per-device error
 *     word and reported by moe_get_error; outputs are then undefined.
 *   - Shapes: T tokens, d model dim, N experts, k experts per token, F = d_ff
 *     expert hidden dim, A = T*k token-expert assignments.
 *     1 <= k <= N <= 256, T >= 0, T*k < 2^31.
 *     dtype MOE_BF16: activations and expert weights bf16, gate fp32;
 *       needs d % 128 == 0, F % 64 == 0 (SwiGLU) or F % 128 == 0 (GELU).
 *     dtype MOE_F32: everything fp32; needs d % 4 == 0.
 *   - Weights are stored [out, in]: w_gate, w_up [N, F, d]; w_down [N, d, F]
 *     (for the two-matrix GELU FFN w_gate holds W_1 and w_up is NULL).
 *   - Results do not depend on the stream, the launch order or the run:
 *     no floating-point atomics are used anywhere.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, k > N, negative size ... */
    MOE_ERR_UNSUPPORTED = 2,   /* valid but not handled (e.g. d % 128 != 0 in bf16) */
    MOE_ERR_WORKSPACE = 3,     /* ws_bytes smaller than the call needs */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    MOE_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out (kernel returned) */
    MOE_ERR_CORRUPT = 6        /* expert index out of range or inconsistent offsets */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;
typedef enum { MOE_SWIGLU = 0, MOE_GELU_TANH = 1 } moe_act;

typedef struct {
    int64_t T;      /* tokens */
    int32_t d;      /* model dim */
    int32_t N;      /* experts */
    int32_t k;      /* experts per token */
    int32_t d_ff;   /* expert hidden dim F */
    int32_t act;    /* moe_act */
    int32_t dtype;  /* moe_dtype */
} moe_shape;

/*
 * Gate and routing: "MoE显存与计算开销四阶段手算指南" sections 2.1-2.2,
 * "MoE混合专家模型计算原理与推理部署实战解析" sections 2.1, 2.2, 2.4.
 *   s[t,n]   = sum_i x[t,i] * w_g[i,n] (+ bias[n])   fp32, FMA accumulation
 *   topk_idx = the k experts of largest s, descending; equal s -> lower id first
 *   topk_w   = softmax(s) restricted to the k selected and renormalised to sum 1
 * x [T,d] (bf16 or fp32 per dtype), w_g [d,N] fp32, bias [N] fp32 or NULL
 * (added to the logits before the softmax). Outputs topk_idx [T,k] int32,
 * topk_w [T,k] fp32. Needs no workspace.
 */
moe_status moe_route(const moe_shape *s, const void *x, const float *w_g, const float *bias,
                     int32_t *topk_idx, float *topk_w, void *stream);

/*
 * Routing with a choice of bias mode and optional routing statistics.
 * bias_mode MOE_BIAS_LOGITS: as moe_route (bias added to the logits before
 * the softmax). MOE_BIAS_SELECT: the auxiliary-loss-free balancing of
 * "MoE混合专家模型计算原理与推理部署实战解析" section 4.4 -- the experts are
 * chosen by s = logit + bias (fp32 sum) but topk_w is the renormalised softmax
 * of the logits WITHOUT the bias.
 * load_stats (device, MOE_LOAD_STATS_LEN(N) floats, or NULL) receives, with p
 * the softmax that weights the experts (over all N):
 *   [0, N)     f[n] = assignments to expert n / (T*k)
 *   [N, 2N)    P[n] = mean over tokens of p[t,n]
 *   [2N]       N * sum_n f[n] * P[n]   (section 4.2 of the same page: 1 for
 *              a uniform load, up to N when one expert takes everything)
 *   [2N+1]     -sum_{f>0} f log2 f, the activation entropy in bits (maximum
 *              log2 N; "这不是“参数越多越强”的简单故事" sections 3.1, 4.4)
 *   [2N+2]     mean over tokens of max_n p[t,n] (top-1 confidence, same page
 *              section 4.4)
 * all zero for T = 0. Statistics are reduced in a fixed order (reproducible
 * bit for bit). ws: moe_route_ex_workspace_size(s) bytes (may be NULL when
 * load_stats is NULL). Other arguments as moe_route.
 */
typedef enum { MOE_BIAS_LOGITS = 0, MOE_BIAS_SELECT = 1 } moe_bias_mode;
#define MOE_LOAD_STATS_LEN(N) (2 * (N) + 3)
moe_status moe_route_ex(const moe_shape *s, const void *x, const float *w_g, const float *bias,
                        int32_t bias_mode, int32_t *topk_idx, float *topk_w, float *load_stats,
                        void *ws, size_t ws_bytes, void *stream);
size_t moe_route_ex_workspace_size(const moe_shape *s);

/*
 * Grouping by expert: "MoE显存与计算开销四阶段手算指南" section 2.3,
 * "MoE混合专家模型计算原理与推理部署实战解析" section 5.1 steps 2-3.
 *   counts[n]  = number of assignments to expert n (sum = T*k)
 *   offsets    = exclusive prefix sum of counts, offsets[N] = T*k   ([N+1])
 *   rows offsets[n] .. offsets[n+1]-1 hold expert n's assignments in flat
 *   order f = t*k + j (a stable counting sort):
 *   perm[row] = t,  inv_perm[f] = row,  x_perm[row,:] = x[t,:]
 * topk_idx [T,k]; x [T,d]; x_perm [T*k, d] (dtype of x). Bit-exact and
 * deterministic. ws: at least moe_permute_workspace_size(s) bytes.
 * x_perm may be NULL (x is then not read): counts, offsets, perm and
 * inv_perm only, for moe_grouped_ffn_gather, which loads the rows itself.
 * An index outside [0,N) records MOE_ERR_CORRUPT.
 */
moe_status moe_permute(const moe_shape *s, const int32_t *topk_idx, const void *x,
                       int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                       void *x_perm, void *ws, size_t ws_bytes, void *stream);

/*
 * Every active expert's FFN as grouped GEMMs over the permuted rows:
 * "MoE混合专家模型计算原理与推理部署实战解析" section 3.1 (SwiGLU:
 * h = SiLU(x W_gate^T) * (x W_up^T), y = h W_down^T) and section 3.2;
 * "MoE显存与计算开销四阶段手算指南" sections 2.3 and 4.3 (one launch over
 * all experts, inputs contiguous, expert_offsets).
 * For MOE_GELU_TANH: h = gelu_tanh(x W_1^T), y = h W_2^T (w_up = NULL).
 * x_perm [A,d], offsets [N+1] (as from moe_permute / moe_permute_capacity:
 * rows offsets[N] .. A-1 are ignored), y_perm [A,d].
 * bf16: tcgen05 tensor cores, fp32 accumulation in tensor memory, h rounded
 * to bf16; f32: fp32 CUDA-core GEMM. ws: moe_grouped_ffn_workspace_size(s)
 * bytes; on return its first A*F elements (dtype of s) hold h [A, F] in the
 * rows of x_perm (rows past offsets[N] unwritten). Offsets that are not a
 * monotone partition of a prefix
 * [0, offsets[N]) of the A rows record MOE_ERR_CORRUPT and the GEMMs do
 * nothing.
 */
moe_status moe_grouped_ffn(const moe_shape *s, const void *x_perm, const int32_t *offsets,
                           const void *w_gate, const void *w_up, const void *w_down,
                           void *y_perm, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_grouped_ffn with the first GEMM's rows taken from the unpermuted tokens:
 * row r of expert e's block is token perm[r], loaded by the GEMM's TMA
 * through the permutation ("MoE显存与计算开销四阶段手算指南" section 4.3 notes
 * what non-contiguous expert inputs cost; here the rows are gathered by the
 * tile loads, so the contiguous x_perm is never written or read). x [T,d]
 * bf16 and perm [A] as from moe_permute (x_perm may be NULL there); other
 * arguments, the result and the workspace as moe_grouped_ffn. bf16 only
 * (MOE_ERR_UNSUPPORTED for fp32). Bit-identical to moe_grouped_ffn on the
 * copy, and saves the T*k x d x_perm buffer and its copy, but is slower on
 * B300 (worked example: 5.1 ms against 3.7-3.8 ms for the grouped FFN; the
 * per-row gathers slow the weight stream), so moe_forward does not use it.
 */
moe_status moe_grouped_ffn_gather(const moe_shape *s, const void *x, const int32_t *perm,
                                  const int32_t *offsets, const void *w_gate, const void *w_up,
                                  const void *w_down, void *y_perm, void *ws, size_t ws_bytes,
                                  void *stream);

/*
 * Weighted combine back to token order: "MoE显存与计算开销四阶段手算指南"
 * section 2.4, "MoE混合专家模型计算原理与推理部署实战解析" sections 2.2 and 5.1
 * step 5:   out[t,:] = sum_{j<k} topk_w[t,j] * y_perm[inv_perm[t*k+j], :]
 * summed in j order in fp32, written once per row (no zero-fill, no atomics).
 * y_perm [A,d], inv_perm [A], topk_w [T,k] fp32, out [T,d] (dtype).
 */
moe_status moe_combine(const moe_shape *s, const void *y_perm, const int32_t *inv_perm,
                       const float *topk_w, void *out, void *stream);

/*
 * The whole layer, "MoE混合专家模型计算原理与推理部署实战解析" section 6.1
 * steps 1-5: moe_route -> moe_permute -> moe_grouped_ffn -> moe_combine on one
 * stream, intermediates in ws (moe_workspace_size(s) bytes). topk_idx,
 * topk_w and counts may be NULL (then they live in ws) or caller buffers
 * that receive the routing.
 */
moe_status moe_forward(const moe_shape *s, const void *x, const float *w_g, const float *bias,
                       const void *w_gate, const void *w_up, const void *w_down, void *out,
                       int32_t *topk_idx, float *topk_w, int32_t *counts,
                       void *ws, size_t ws_bytes, void *stream);

/*
 * Grouping with an expert capacity: "MoE混合专家模型计算原理与推理部署实战解析"
 * section 4.3 (at inference an expert takes at most
 * capacity_factor * total_tokens / num_experts tokens; the overflow is dropped
 * and only the residual path carries it). Here the capacity is
 * ceil(capacity_factor * T * k / N) assignments per expert; an expert keeps
 * its earliest assignments in flat order t*k + j. Outputs as moe_permute,
 * except: counts / offsets describe the kept rows (offsets[N] <= T*k),
 * inv_perm[f] = -2 for a dropped assignment, and *dropped (optional, int32)
 * receives the number of dropped assignments; x_perm may be NULL as for
 * moe_permute. moe_grouped_ffn, moe_grouped_ffn_gather and moe_combine
 * accept these directly (a dropped assignment adds nothing to
 * the token's output; kept gate weights are not renormalised).
 */
moe_status moe_permute_capacity(const moe_shape *s, const int32_t *topk_idx, const void *x,
                                double capacity_factor, int32_t *counts, int32_t *offsets,
                                int32_t *perm, int32_t *inv_perm, void *x_perm, int32_t *dropped,
                                void *ws, size_t ws_bytes, void *stream);

/* moe_forward with an expert capacity (see moe_permute_capacity); ws as moe_forward. */
moe_status moe_forward_capacity(const moe_shape *s, double capacity_factor, const void *x,
                                const float *w_g, const float *bias, const void *w_gate,
                                const void *w_up, const void *w_down, void *out, int32_t *topk_idx,
                                float *topk_w, int32_t *counts, int32_t *dropped, void *ws,
                                size_t ws_bytes, void *stream);

/*
 * moe_forward with options, all optional and combinable:
 *   bias_mode       moe_bias_mode (see moe_route_ex)
 *   use_capacity    nonzero: expert capacity ceil(capacity_factor * T*k / N)
 *                   as moe_permute_capacity (capacity_factor >= 0)
 *   load_stats      device, MOE_LOAD_STATS_LEN(N) floats, or NULL (see
 *                   moe_route_ex; statistics of the routing, before any drop)
 *   dropped         device int32, or NULL: assignments dropped by the capacity
 *   use_tiling      nonzero: this call's grouped GEMMs use ffn_tiling (a
 *                   moe_tiling value) instead of the process-wide setting of
 *                   moe_set_ffn_tiling, so callers in one process that want
 *                   different tilings do not share a global
 * opt == NULL is the plain moe_forward. ws: moe_workspace_size(s) bytes.
 */
typedef struct {
    int32_t bias_mode;
    int32_t use_capacity;
    double capacity_factor;
    float *load_stats;
    int32_t *dropped;
    int32_t use_tiling;
    int32_t ffn_tiling;
} moe_options;
moe_status moe_forward_ex(const moe_shape *s, const moe_options *opt, const void *x, const float *w_g,
                          const float *bias, const void *w_gate, const void *w_up,
                          const void *w_down, void *out, int32_t *topk_idx, float *topk_w,
                          int32_t *counts, void *ws, size_t ws_bytes, void *stream);

/*
 * Expert-choice routing: "MoE混合专家模型计算原理与推理部署实战解析" section
 * 2.3 (each expert picks its own top tokens: every expert processes the same
 * number, and a token may be picked by none). Readings: the affinity is the
 * gate probability p[t,e] = softmax over the experts of the fp32 logits
 * x w_g (+ bias, added to the logits); expert e takes the C tokens of
 * largest p[t,e] (equal values: lower token id first) and weights each by
 * p[t,e] (no renormalisation). s->k is not used (any valid value).
 * Outputs:
 *   probs   [T,N] fp32   the gate probabilities
 *   perm    [N*C] int32  row -> token; expert e owns rows e*C .. e*C + C - 1,
 *                        its tokens in ascending order
 *   counts  [N]   = C;   offsets [N+1] = e*C
 *   inv     [T,N] int32  row of (t, e), or -2 when e did not pick t
 *   w       [T,N] fp32   p[t,e] when e picked t, else 0
 * Needs 0 <= C <= T. The choice is deterministic (integer radix select).
 */
moe_status moe_route_expert_choice(const moe_shape *s, int64_t C, const void *x, const float *w_g,
                                   const float *bias, float *probs, int32_t *perm, int32_t *counts,
                                   int32_t *offsets, int32_t *inv, float *w, void *stream);

/*
 * The row copy of the grouping step on its own ("MoE混合专家模型计算原理与推理
 * 部署实战解析" section 5.1 step 3): x_perm[inv[t*slots + j]] = x[t] for every
 * t < T and j < slots whose row lies in [0, rows); other entries (-2: not
 * chosen or dropped) are skipped. With the expert-choice tables (slots = N,
 * rows = N*C) it builds the expert-choice x_perm; moe_grouped_ffn then runs
 * on a shape with T = N*C, k = 1, and moe_combine on one with k = N.
 * x [T,d], x_perm [rows, d] (dtype of s).
 */
moe_status moe_gather_rows(const moe_shape *s, const int32_t *inv, int32_t slots, int64_t rows,
                           const void *x, void *x_perm, void *stream);

/*
 * The whole layer with expert-choice routing: moe_route_expert_choice, the
 * row copy x_perm[row] = x[perm[row]], the grouped FFN over the N*C rows
 * (C per expert), and out[t] = sum over the experts e that picked t of
 * p[t,e] * y_e(x_t), summed in expert order (a token picked by no expert
 * gets 0). counts [N] is optional. ws: moe_expert_choice_workspace_size(s, C)
 * bytes.
 */
moe_status moe_forward_expert_choice(const moe_shape *s, int64_t C, const void *x, const float *w_g,
                                     const float *bias, const void *w_gate, const void *w_up,
                                     const void *w_down, void *out, int32_t *counts, void *ws,
                                     size_t ws_bytes, void *stream);
size_t moe_expert_choice_workspace_size(const moe_shape *s, int64_t C);

/*
 * moe_forward with x and out in HOST memory (pinned memory makes the copies
 * asynchronous): copies x into ws, runs the layer, copies out back, all on
 * `stream`. The caller synchronises the stream before reading out_host.
 * ws: moe_forward_hostio_workspace_size(s) bytes.
 */
moe_status moe_forward_hostio(const moe_shape *s, const void *x_host, const float *w_g,
                              const float *bias, const void *w_gate, const void *w_up,
                              const void *w_down, void *out_host, void *ws, size_t ws_bytes,
                              void *stream);

/*
 * moe_forward_hostio for a sequence of batches, with the copies of one batch
 * overlapping the layer of another: three streams (compute_stream for the
 * layer, h2d_stream for the x copies, d2h_stream for the output copies) and
 * two workspace slots, alternated by the caller (slot = 0, 1, 0, 1, ... on
 * consecutive calls, from one host thread). The call only enqueues work:
 *   h2d_stream:     x_host -> slot's x once the call two back stopped reading it
 *   compute_stream: the layer on the slot's x once it is in and the slot's
 *                   previous output has been copied out
 *   d2h_stream:     the slot's out -> out_host
 * out_host holds this batch's output once d2h_stream has passed this call
 * (synchronise it, or an event recorded on it after the call); x_host must
 * stay unchanged until h2d_stream has passed the call. Device inputs
 * (weights, w_g, bias) must not change while calls are in flight. The
 * library creates eight events per device on first use (kept until the
 * process exits); they order the two slots, so one such pipeline runs per
 * device at a time. ws: moe_forward_hostio_pipelined_workspace_size(s) bytes.
 * The pages name no such entry point: it exists so that host<->device copies
 * of consecutive batches hide behind the layer.
 */
moe_status moe_forward_hostio_pipelined(const moe_shape *s, const void *x_host, const float *w_g,
                                        const float *bias, const void *w_gate, const void *w_up,
                                        const void *w_down, void *out_host, void *ws, size_t ws_bytes,
                                        int32_t slot, void *compute_stream, void *h2d_stream,
                                        void *d2h_stream);
size_t moe_forward_hostio_pipelined_workspace_size(const moe_shape *s);

/*
 * moe_permute without a caller workspace. No passage of the pages has a
 * counterpart: this exists for callers that cannot hand the library device
 * scratch memory -- for example a host framework that gives a custom operator
 * only its input and output tensors and no allocator, or latency-critical code
 * that must not call cudaMalloc (it can synchronise the device) in the middle
 * of a forward. Outputs and their meaning are exactly those of moe_permute.
 *
 * The per-chunk expert histogram lives in a fixed array inside the library
 * (MOE_PERMUTE_NOALLOC_SCRATCH_INTS int32 values, 256 KiB, held on every
 * device that loads the library until the process exits). The shape must
 * satisfy ceil(T / max(1, 2048 / k)) * N <= MOE_PERMUTE_NOALLOC_SCRATCH_INTS
 * (for example T up to about 1M tokens at k = 2, N = 64); larger shapes return
 * MOE_ERR_WORKSPACE and launch nothing. The call allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine.
 *
 * The first call on a device looks up that device's address of the array
 * (cudaGetSymbolAddress, with the device current; under a mutex, so first
 * calls from several host threads are safe); make that first call before any
 * stream capture. The cached address is not valid across a device reset
 * (cudaDeviceReset): do not call this after one in the same process. All
 * calls share the one array and it keeps the
 * last call's contents (every entry a call reads is written first by the same
 * call, so nothing needs clearing); calls whose work overlaps on the GPU (two
 * streams at once) race on it and must be serialised by the caller.
 */
#define MOE_PERMUTE_NOALLOC_SCRATCH_INTS 65536
moe_status moe_permute_noalloc(const moe_shape *s, const int32_t *topk_idx, const void *x,
                               int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                               void *x_perm, void *stream);

/*
 * Expert parallelism: "MoE混合专家模型计算原理与推理部署实战解析" section 3.3
 * (experts split over G GPUs by expert id, e.g. 8 experts over 4 cards with
 * 2 each; every card routes its own tokens and an all-to-all carries each
 * token row to the card that holds its expert; the traffic grows with tokens
 * x hidden size) and section 6.3 (EP). Reading: card g holds the contiguous
 * expert range [g*E, (g+1)*E) with E = N / G, so moe_permute's x_perm, ordered
 * by expert, is already ordered by destination card: card g's share is rows
 * offsets[g*E] .. offsets[(g+1)*E] - 1. The exchanges themselves (an
 * all-to-all of the per-expert counts, then of the rows, and back) are the
 * caller's, e.g. NCCL or any other transport; the library does the local
 * steps on either side of them.
 *
 * moe_ep_regroup: the rows a card received, ordered by (source card g, local
 * expert e, the source's row order), regrouped by local expert for
 * moe_grouped_ffn:
 *   recv_counts [G][E] int32 (device): rows card g sent for local expert e;
 *                the table must account for exactly `rows` received rows
 *   recv_x      [rows, d] (dtype): the received rows in that order
 *   x_local     [rows, d]: the same rows ordered (e, g, source order)
 *   offsets_local [E+1]: expert e's rows are offsets_local[e] .. [e+1]-1
 *   local_src   [rows] int32: the received row each local row came from
 * moe_grouped_ffn then runs on a shape with T = rows, k = 1, N = E and the
 * card's E experts' weights.
 * moe_ep_ungroup: y_recv[local_src[i]] = y_local[i] (back to the received
 * order); the reverse all-to-all then returns every row to its source in the
 * order it was sent, i.e. as that source's y_perm, and moe_combine runs on it
 * unchanged.
 * Needs 1 <= G*E <= 256, rows < 2^31, d * element size a multiple of 16
 * bytes. A count table that is negative or does not add up to `rows`, or a
 * local_src entry out of range, records MOE_ERR_CORRUPT (nothing copied).
 * Integer bookkeeping and row copies only: bit-exact.
 */
moe_status moe_ep_regroup(int32_t G, int32_t E, const int32_t *recv_counts, int64_t rows, int32_t d,
                          int32_t dtype, const void *recv_x, void *x_local, int32_t *offsets_local,
                          int32_t *local_src, void *stream);
moe_status moe_ep_ungroup(int64_t rows, int32_t d, int32_t dtype, const int32_t *local_src,
                          const void *y_local, void *y_recv, void *stream);

/*
 * Tiling of the bf16 grouped GEMMs in moe_grouped_ffn / moe_forward (process
 * wide; results agree within the bf16 tolerance, not bit for bit):
 *   MOE_TILING_ROWS    128 permuted rows x 256 weight rows per tile (weights
 *                      are the MMA's N side); an expert's last tile is padded
 *                      up to 128 rows.
 *   MOE_TILING_TOKENS  128 weight rows x up to 256 tokens per tile (tokens are
 *                      the MMA's N side, tiles balanced per expert and rounded
 *                      to 16 rows): little padding when experts hold few rows.
 *   MOE_TILING_PAIRS   token tiles computed by clusters of two SMs sharing each
 *                      MMA (256 weight rows per MMA, each SM holding half of
 *                      the tile's tokens): four 48 KB pipeline stages per SM
 *                      instead of three 64 KB ones.
 *   MOE_TILING_ROW_PAIRS row tiles computed by clusters of two SMs sharing each
 *                      MMA: 256 permuted rows x 256 weight rows per tile, 128
 *                      of each in each SM, so every weight tile serves twice the
 *                      rows of MOE_TILING_ROWS. Used where the tile's output
 *                      columns divide the GEMM's (SwiGLU F % 128, GELU F % 256,
 *                      the down projection d % 256) and the rows are permuted
 *                      (not moe_grouped_ffn_gather); row tiles otherwise.
 *   MOE_TILING_AUTO    per GEMM: token tiles on SM pairs when T*k >= 64*N and
 *                      the GEMM's reduction length (d for the first, F for the
 *                      second) is >= 4096, else row tiles (default).
 * The pages' grouped GEMM ("MoE显存与计算开销四阶段手算指南" section 4.3)
 * fixes no tiling; this only chooses how the same product is blocked.
 */
typedef enum {
    MOE_TILING_AUTO = 0,
    MOE_TILING_ROWS = 1,
    MOE_TILING_TOKENS = 2,
    MOE_TILING_PAIRS = 3,
    MOE_TILING_ROW_PAIRS = 4
} moe_tiling;
moe_status moe_set_ffn_tiling(int mode);
int moe_get_ffn_tiling(void);

/* Workspace sizes in bytes (0 when the shape is invalid or unsupported). */
size_t moe_workspace_size(const moe_shape *s);
size_t moe_forward_hostio_workspace_size(const moe_shape *s);
size_t moe_permute_workspace_size(const moe_shape *s);
size_t moe_grouped_ffn_workspace_size(const moe_shape *s);

/* Host-side shape check: MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED. */
moe_status moe_check_shape(const moe_shape *s);

/*
 * Synchronises `stream`, then returns and clears the current device's error
 * word (MOE_OK if no kernel recorded an error). MOE_ERR_CUDA if the
 * synchronisation itself failed.
 */
moe_status moe_get_error(void *stream);

/*
 * Self-test of the bounded device-side wait used by the pipelined kernels:
 * one CTA waits on a shared-memory barrier that nothing ever completes,
 * gives up after timeout_ns (clamped to [1 ms, 2 s]), records
 * MOE_ERR_TIMEOUT and returns. The context stays usable.
 */
moe_status moe_selftest_bounded_wait(int64_t timeout_ns, void *stream);

const char *moe_status_string(moe_status st);

/* Library version, major*10000 + minor*100 + patch. */
int moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
