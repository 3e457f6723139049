/*
 * moe_oracle.c -- CPU oracle of the MoE layer forward (fp64; fp32 gate).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the package's smoke check and the benchmark's CPU
 * baseline use it. It shares no code, header or table with the CUDA library.
 *
 * It is a plain, slow, obviously correct restatement of what the pages define,
 * in double precision except for the gate logits, which the pages keep in
 * fp32 (see the readings below). Inputs are read exactly as the GPU receives
 * them (fp32 or bf16 values widened to fp64, which is exact). OpenMP only
 * splits independent tokens / rows across host threads.
 *
 * Sources (page titles as printed on the pages):
 *   [P2] "MoE显存与计算开销四阶段手算指南": s2.1 gate projection logits = x @ W_g,
 *        s2.2 softmax then per-token top-k (topk_indices / topk_probs),
 *        s2.3 grouping of tokens per expert (N_i, sum N_i = B*S*k),
 *        s2.4 weighted sum of the k expert outputs back in token order,
 *        s3 the toy forward (stacked per-expert inputs, per-expert Linear).
 *   [P4] "这不是“参数越多越强”的简单故事" (deployment notes): s3.1 / s4.4
 *        expert activation entropy and top-1 confidence as routing health
 *        statistics.
 *   [P3] "MoE混合专家模型计算原理与推理部署实战解析": s2.1 gate, softmax, top-k;
 *        s2.2 renormalisation g_i' = g_i / sum of selected g and the weighted
 *        output; s2.4 gate kept in fp32; s3.1 SwiGLU expert
 *        (gate, up, SiLU(gate)*up, down); s5.1 count -> prefix sum -> permute ->
 *        per-expert GEMM -> unpermute + weighted merge.
 *
 * Readings where the pages are silent or ambiguous, taken here:
 *   - the gate is computed in fp32 ([P3] s2.4 and s7 keep the gate in FP32
 *     and the experts in bf16). Its plainest fp32 evaluation is used: for
 *     each logit the sequential chain s <- fma(x_i, W_g[i,n], s) over
 *     i = 0..d-1 from s = 0, then one fp32 addition of the bias. The top-k
 *     decision is taken on these fp32 values; softmax and renormalisation
 *     then run in fp64 on them. (gate_fp32 = 0 gives exact fp64 logits.)
 *   - top-k is taken on the score s = logit (+ per-expert bias); softmax is
 *     monotone, so this is the pages' top-k over probabilities, without the
 *     false ties that rounded probabilities can create;
 *   - equal scores: the lower expert id wins; the k slots are in descending
 *     score order;
 *   - the bias (when given) is added to the logits before the softmax
 *     (bias_mode 0), or, as the auxiliary-loss-free balancing of [P3] s4.4
 *     describes it, only to the scores that choose the experts
 *     (bias_mode 1): then the gate weights come from the softmax of the
 *     logits without the bias;
 *   - rows of one expert are kept in flat assignment order t*k + j (stable);
 *   - the two-matrix FFN uses the tanh form of GELU; no biases anywhere;
 *   - weights are stored [out, in].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F64 = 0, OR_F32 = 1, OR_BF16 = 2 };
enum { OR_SWIGLU = 0, OR_GELU_TANH = 1 };

/* Read element i of an input array stored as fp64, fp32 or bf16 bits. */
static double rd(const void *p, int dt, int64_t i)
{
    if (dt == OR_F64) return ((const double *)p)[i];
    if (dt == OR_F32) return (double)((const float *)p)[i];
    uint32_t u = ((uint32_t)((const uint16_t *)p)[i]) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * Route: [P2] s2.1-2.2, [P3] s2.1-2.2, s2.4.
 *   g[t,n] = sum_i x[t,i] * W_g[i,n]            in fp32 when gate_fp32 != 0
 *            (sequential FMA chain in index order), else exactly in fp64
 *   s[t,n] = g[t,n] + b[n]   (fp32 addition when gate_fp32; s = g without bias)
 *   bias_mode 0: l = s    the bias is part of the logits
 *   bias_mode 1: l = g    the bias only chooses ([P3] s4.4)
 *   p[t,:] = softmax(l[t,:])
 *   top-k by s (ties -> lower id), in descending order
 *   w[t,j] = p[t,e_j] / sum_j' p[t,e_j']
 *   probs   optional [T,N] copy of p
 *
 * Also returns, per token, how fragile the decision is against rounding
 * (computed from the exact fp64 logits whatever gate_fp32 says):
 *   errb[t,n]  a bound on |fl32(l[t,n]) - l_exact[t,n]| for ANY fp32 summation order:
 *              gamma_{d+2} * (sum_i |x_i W_g[i,n]| + |b_n|), gamma_m = m u/(1-m u),
 *              u = 2^-24 (the classical bound for a sum of d rounded products
 *              plus one rounded bias addition);
 *   cert[t]    min over i < k, j > i (sorted exact order) of
 *              (s_(i) - errb_(i)) - (s_(j) + errb_(j)) on the exact scores.
 *              cert > 0 proves that ANY fp32 evaluation selects the same
 *              experts in the same order as exact arithmetic.
 *   logits     optional [T,N] copy of the scores s (fp32 values when gate_fp32).
 * Returns 0, or -1 on bad arguments.
 * ------------------------------------------------------------------------- */
int oracle_route(int64_t T, int d, int N, int k,
                 const void *x, int x_dt,
                 const void *wg, int wg_dt,
                 const void *bias, int b_dt, int bias_mode, int gate_fp32,
                 int32_t *topk_idx, double *topk_w,
                 double *logits, double *errb, double *cert, double *probs)
{
    if (T < 0 || d < 1 || N < 1 || k < 1 || k > N || bias_mode < 0 || bias_mode > 1) return -1;
    const double u = ldexp(1.0, -24);
    const double gam = (d + 2) * u / (1.0 - (d + 2) * u);
    int bad = 0;

#pragma omp parallel
    {
        double *l = (double *)malloc(sizeof(double) * N);   /* scores: choose the experts */
        double *g = (double *)malloc(sizeof(double) * N);   /* logits of the softmax */
        double *s = (double *)malloc(sizeof(double) * N);
        double *p = (double *)malloc(sizeof(double) * N);
        double *eb = (double *)malloc(sizeof(double) * N);
        double *ex = (double *)malloc(sizeof(double) * N);
        int *taken = (int *)malloc(sizeof(int) * N);
        int *order = (int *)malloc(sizeof(int) * N);
        if (!l || !g || !s || !p || !eb || !ex || !taken || !order) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t t = 0; t < T; ++t) {
                /* gate projection */
                for (int n = 0; n < N; ++n) {
                    double acc = 0.0, aabs = 0.0;
                    float acc32 = 0.0f;
                    for (int i = 0; i < d; ++i) {
                        double xi = rd(x, x_dt, t * d + i), wi = rd(wg, wg_dt, (int64_t)i * N + n);
                        double prod = xi * wi;
                        acc += prod;
                        aabs += fabs(prod);
                        if (gate_fp32) acc32 = fmaf((float)xi, (float)wi, acc32);
                    }
                    double b = bias ? rd(bias, b_dt, n) : 0.0;
                    ex[n] = acc + b;
                    l[n] = gate_fp32 ? (double)(bias ? acc32 + (float)b : acc32) : acc + b;
                    g[n] = bias_mode == 1 ? (gate_fp32 ? (double)acc32 : acc) : l[n];
                    s[n] = aabs + fabs(b);
                    eb[n] = gam * s[n];
                }
                /* softmax over all N experts, with max subtraction */
                double m = g[0];
                for (int n = 1; n < N; ++n) if (g[n] > m) m = g[n];
                double z = 0.0;
                for (int n = 0; n < N; ++n) { p[n] = exp(g[n] - m); z += p[n]; }
                for (int n = 0; n < N; ++n) p[n] /= z;
                if (probs) for (int n = 0; n < N; ++n) probs[t * N + n] = p[n];
                /* full descending order by (l desc, id asc): repeated argmax */
                for (int n = 0; n < N; ++n) taken[n] = 0;
                for (int r = 0; r < N; ++r) {
                    int best = -1;
                    for (int n = 0; n < N; ++n) {
                        if (taken[n]) continue;
                        if (best < 0 || l[n] > l[best]) best = n;   /* strict: lower id kept on ties */
                    }
                    taken[best] = 1;
                    order[r] = best;
                }
                /* renormalise the k selected gate values */
                double sel = 0.0;
                for (int j = 0; j < k; ++j) sel += p[order[j]];
                for (int j = 0; j < k; ++j) {
                    topk_idx[t * k + j] = order[j];
                    topk_w[t * k + j] = p[order[j]] / sel;
                }
                if (logits) for (int n = 0; n < N; ++n) logits[t * N + n] = l[n];
                if (errb) for (int n = 0; n < N; ++n) errb[t * N + n] = eb[n];
                if (cert) {
                    /* order of the exact logits, then the smallest separation */
                    for (int n = 0; n < N; ++n) taken[n] = 0;
                    for (int r = 0; r < N; ++r) {
                        int best = -1;
                        for (int n = 0; n < N; ++n) {
                            if (taken[n]) continue;
                            if (best < 0 || ex[n] > ex[best]) best = n;
                        }
                        taken[best] = 1;
                        order[r] = best;
                    }
                    double c = INFINITY;
                    for (int i = 0; i < k; ++i) {
                        double lo = ex[order[i]] - eb[order[i]];
                        for (int j2 = i + 1; j2 < N; ++j2) {
                            double hi = ex[order[j2]] + eb[order[j2]];
                            if (lo - hi < c) c = lo - hi;
                        }
                    }
                    cert[t] = c;
                }
            }
        }
        free(l); free(g); free(s); free(p); free(eb); free(ex); free(taken); free(order);
    }
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------------------
 * Group assignments by expert: [P2] s2.3, [P3] s5.1 steps 2-3.
 *   counts[n]  = number of (t,j) with e_{t,j} = n      (sum = T*k)
 *   offsets    = exclusive prefix sum of counts, offsets[N] = T*k
 *   rows of expert n are offsets[n] .. offsets[n+1]-1, filled in flat order
 *   f = t*k + j:   perm[row] = t,  inv_perm[f] = row.
 * Returns 0, or -1 if an index is out of [0, N).
 * ------------------------------------------------------------------------- */
int oracle_permute(int64_t T, int N, int k, const int32_t *topk_idx,
                   int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm)
{
    const int64_t A = T * k;
    for (int n = 0; n < N; ++n) counts[n] = 0;
    for (int64_t f = 0; f < A; ++f) {
        int e = topk_idx[f];
        if (e < 0 || e >= N) return -1;
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int n = 0; n < N; ++n) offsets[n + 1] = offsets[n] + counts[n];
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    if (!fill) return -1;
    for (int n = 0; n < N; ++n) fill[n] = offsets[n];
    for (int64_t f = 0; f < A; ++f) {
        int e = topk_idx[f];
        int32_t row = fill[e]++;
        perm[row] = (int32_t)(f / k);
        inv_perm[f] = row;
    }
    free(fill);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Grouping with an expert capacity: [P3] s4.3. At inference an expert takes
 * at most `capacity` assignments; the rest are dropped (the token skips that
 * expert and only the residual path carries it). Readings: capacity counts
 * assignments, capacity = ceil(capacity_factor * T * k / N) (oracle_capacity);
 * an expert keeps its assignments in flat order t*k + j, so the earliest
 * `capacity` are kept; a dropped assignment contributes nothing to the output
 * and the kept gate weights are not renormalised again.
 *   counts[n]  kept assignments of expert n = min(demand, capacity)
 *   offsets    exclusive prefix sum of the kept counts
 *   perm[row] = t for kept rows; inv_perm[f] = row, or -2 when dropped
 * Returns the number of dropped assignments, or -1 on a bad index.
 * ------------------------------------------------------------------------- */
int64_t oracle_capacity(int64_t T, int N, int k, double capacity_factor)
{
    return (int64_t)ceil(capacity_factor * (double)T * (double)k / (double)N);
}

int64_t oracle_permute_capacity(int64_t T, int N, int k, const int32_t *topk_idx, int64_t capacity,
                                int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm)
{
    const int64_t A = T * k;
    int64_t *demand = (int64_t *)calloc((size_t)N, sizeof(int64_t));
    if (!demand) return -1;
    for (int64_t f = 0; f < A; ++f) {
        int e = topk_idx[f];
        if (e < 0 || e >= N) { free(demand); return -1; }
        demand[e] += 1;
    }
    offsets[0] = 0;
    for (int n = 0; n < N; ++n) {
        counts[n] = (int32_t)(demand[n] < capacity ? demand[n] : capacity);
        offsets[n + 1] = offsets[n] + counts[n];
    }
    int64_t dropped = 0;
    for (int n = 0; n < N; ++n) demand[n] = 0;          /* reused: assignments seen so far */
    for (int64_t f = 0; f < A; ++f) {
        int e = topk_idx[f];
        int64_t r = demand[e]++;
        if (r < capacity) {
            int32_t row = offsets[e] + (int32_t)r;
            perm[row] = (int32_t)(f / k);
            inv_perm[f] = row;
        } else {
            inv_perm[f] = -2;
            dropped += 1;
        }
    }
    free(demand);
    return dropped;
}

/* ---------------------------------------------------------------------------
 * Load statistics of one routed batch: [P3] s4.2 (the Switch load-balance
 * quantity) and [P4] "这不是“参数越多越强”的简单故事" s3.1 (expert activation
 * entropy, maximum 4.0 for 16 experts) and s4.4 (monitoring: activation
 * entropy, top-1 routing confidence).
 *   f[n] = (number of assignments to n) / (T*k)          fraction routed to n
 *   P[n] = (1/T) sum_t p[t,n]                            mean gate probability
 *   out3[0] = N * sum_n f[n] * P[n]                      balance quantity (1 when uniform)
 *   out3[1] = -sum_{f[n] > 0} f[n] log2 f[n]             activation entropy, bits (max log2 N)
 *   out3[2] = (1/T) sum_t max_n p[t,n]                   mean top-1 probability
 * p is the softmax whose values weight the experts (probs of oracle_route).
 * Readings: f counts the k assignments of a token each (so sum f = 1 for any
 * k, and uniform routing gives f = 1/N as the page's example needs); the
 * entropy is in bits, as the page's "maximum 4.0 for 16 experts" implies; an
 * empty batch gives all zeros. Returns 0, or -1 on a bad index.
 * ------------------------------------------------------------------------- */
int oracle_load_stats(int64_t T, int N, int k, const double *probs, const int32_t *topk_idx,
                      double *f, double *P, double *out3)
{
    for (int n = 0; n < N; ++n) { f[n] = 0.0; P[n] = 0.0; }
    out3[0] = out3[1] = out3[2] = 0.0;
    if (T == 0) return 0;
    for (int64_t a = 0; a < T * k; ++a) {
        int e = topk_idx[a];
        if (e < 0 || e >= N) return -1;
        f[e] += 1.0;
    }
    for (int n = 0; n < N; ++n) f[n] /= (double)(T * k);
    double conf = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        double mx = probs[t * N];
        for (int n = 0; n < N; ++n) {
            P[n] += probs[t * N + n];
            if (probs[t * N + n] > mx) mx = probs[t * N + n];
        }
        conf += mx;
    }
    double bal = 0.0, ent = 0.0;
    for (int n = 0; n < N; ++n) {
        P[n] /= (double)T;
        bal += f[n] * P[n];
        if (f[n] > 0.0) ent -= f[n] * log2(f[n]);
    }
    out3[0] = (double)N * bal;
    out3[1] = ent;
    out3[2] = conf / (double)T;
    return 0;
}

/* ---------------------------------------------------------------------------
 * Expert-choice routing: [P3] s2.3 (each expert picks its own top tokens, so
 * every expert processes exactly the same number and a token may be picked
 * by no expert). Readings where the page is silent:
 *   - the token-expert affinity is the gate probability p[t,e] = softmax over
 *     the experts of token t's logits (probs of oracle_route), the quantity
 *     the token-choice top-k of s2.1 ranks;
 *   - expert e takes the C tokens of largest p[t,e]; equal values -> lower t;
 *   - a picked token is weighted by p[t,e] itself (no renormalisation);
 *   - expert e's rows are e*C .. e*C + C - 1, its tokens in ascending order.
 * Outputs:
 *   perm[e*C + i] = token of expert e's i-th row; w_row[same] = p[t,e]
 *   inv[t*N + e] = row, or -2 when e did not pick t; w[t*N + e] = p[t,e] or 0
 *   thr[e]  = the C-th largest p[.,e] (the smallest value picked)
 *   next[e] = the (C+1)-th largest (the largest value left), -1 when C == T
 * The combine is then oracle_combine with k = N over inv / w.
 * Returns 0, or -1 on bad arguments (needs 0 <= C <= T).
 * ------------------------------------------------------------------------- */
typedef struct { double p; int64_t t; } ec_item;

static int ec_cmp(const void *a, const void *b)
{
    const ec_item *x = (const ec_item *)a, *y = (const ec_item *)b;
    if (x->p > y->p) return -1;
    if (x->p < y->p) return 1;
    return (x->t < y->t) ? -1 : (x->t > y->t);
}

int oracle_expert_choice(int64_t T, int N, int64_t C, const double *probs,
                         int32_t *perm, double *w_row, int32_t *inv, double *w, double *thr, double *next)
{
    if (T < 0 || N < 1 || C < 0 || C > T) return -1;
    for (int64_t i = 0; i < T * N; ++i) { inv[i] = -2; w[i] = 0.0; }
    ec_item *it = (ec_item *)malloc(sizeof(ec_item) * (size_t)(T > 0 ? T : 1));
    unsigned char *picked = (unsigned char *)malloc((size_t)(T > 0 ? T : 1));
    if (!it || !picked) { free(it); free(picked); return -1; }
    for (int e = 0; e < N; ++e) {
        for (int64_t t = 0; t < T; ++t) { it[t].p = probs[t * N + e]; it[t].t = t; picked[t] = 0; }
        qsort(it, (size_t)T, sizeof(ec_item), ec_cmp);
        for (int64_t i = 0; i < C; ++i) picked[it[i].t] = 1;
        thr[e] = C > 0 ? it[C - 1].p : INFINITY;
        next[e] = C < T ? it[C].p : -1.0;
        int64_t row = (int64_t)e * C;
        for (int64_t t = 0; t < T; ++t) {
            if (!picked[t]) continue;
            perm[row] = (int32_t)t;
            w_row[row] = probs[t * N + e];
            inv[t * N + e] = (int32_t)row;
            w[t * N + e] = probs[t * N + e];
            ++row;
        }
    }
    free(it);
    free(picked);
    return 0;
}

/* SiLU and tanh-GELU, [P3] s3.1 (SiLU(gate) * up). */
/*
 * Expert parallelism, the receiving card's regrouping ([P3] s3.3: experts
 * split over cards by expert id, token rows carried to the card of their
 * expert by an all-to-all). The card received, from each source card g in
 * order, that source's rows for the card's local experts e = 0..E-1 in order
 * (recv_counts[g*E + e] of them, in the source's own row order). The grouped
 * computation wants them ordered by local expert, and within an expert by
 * source card, then source order. This walks the received buffer once, noting
 * where each (g, e) run starts, then lays the runs out expert by expert:
 *   offsets_local[e]   first local row of expert e (offsets_local[E] = rows)
 *   local_src[row]     the received row that local row holds
 * Returns 0, or -1 for a negative count.
 */
int oracle_ep_regroup(int G, int E, const int32_t *recv_counts, int32_t *offsets_local, int32_t *local_src)
{
    int64_t *run_start = (int64_t *)malloc(sizeof(int64_t) * (size_t)G * (size_t)E);
    if (!run_start) return -1;
    int64_t pos = 0;
    for (int g = 0; g < G; ++g)
        for (int e = 0; e < E; ++e) {
            if (recv_counts[g * E + e] < 0) { free(run_start); return -1; }
            run_start[g * E + e] = pos;
            pos += recv_counts[g * E + e];
        }
    int64_t row = 0;
    for (int e = 0; e < E; ++e) {
        offsets_local[e] = (int32_t)row;
        for (int g = 0; g < G; ++g)
            for (int32_t i = 0; i < recv_counts[g * E + e]; ++i)
                local_src[row++] = (int32_t)(run_start[g * E + e] + i);
    }
    offsets_local[E] = (int32_t)row;
    free(run_start);
    return 0;
}

static double silu(double v) { return v / (1.0 + exp(-v)); }
static double gelu_tanh(double v)
{
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * v * (1.0 + tanh(c * (v + 0.044715 * v * v * v)));
}

/* ---------------------------------------------------------------------------
 * One expert's FFN applied to n_rows input rows: [P3] s3.1, [P2] s2.3.
 *   SwiGLU:   h = SiLU(W_gate x) * (W_up x),  y = W_down h
 *   GELU:     h = gelu_tanh(W_1 x),           y = W_2 h     (w_up == NULL)
 * W_gate, W_up: [F, d]; W_down: [d, F] (all [out, in]).
 * x rows: [n_rows, d] in x_dt; y: [n_rows, d] fp64; h (optional): [n_rows, F].
 * ------------------------------------------------------------------------- */
int oracle_expert_rows(int64_t n_rows, int d, int F, int act,
                       const void *x, int x_dt,
                       const void *w_gate, const void *w_up, const void *w_down, int w_dt,
                       double *y, double *h_out)
{
    if (d < 1 || F < 1 || (act != OR_SWIGLU && act != OR_GELU_TANH)) return -1;
    if (act == OR_SWIGLU && !w_up) return -1;
    int bad = 0;
#pragma omp parallel
    {
        double *xr = (double *)malloc(sizeof(double) * d);
        double *h = (double *)malloc(sizeof(double) * F);
        if (!xr || !h) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n_rows; ++r) {
                for (int i = 0; i < d; ++i) xr[i] = rd(x, x_dt, r * d + i);
                for (int f = 0; f < F; ++f) {
                    double g = 0.0;
                    for (int i = 0; i < d; ++i) g += rd(w_gate, w_dt, (int64_t)f * d + i) * xr[i];
                    if (act == OR_SWIGLU) {
                        double up = 0.0;
                        for (int i = 0; i < d; ++i) up += rd(w_up, w_dt, (int64_t)f * d + i) * xr[i];
                        h[f] = silu(g) * up;
                    } else {
                        h[f] = gelu_tanh(g);
                    }
                }
                if (h_out) for (int f = 0; f < F; ++f) h_out[r * F + f] = h[f];
                for (int o = 0; o < d; ++o) {
                    double acc = 0.0;
                    for (int f = 0; f < F; ++f) acc += rd(w_down, w_dt, (int64_t)o * F + f) * h[f];
                    y[r * d + o] = acc;
                }
            }
        }
        free(xr); free(h);
    }
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------------------
 * Combine: [P2] s2.4, [P3] s2.2 / s5.1 step 5.
 *   out[t] = sum_{j<k} w[t,j] * y_perm[inv_perm[t*k+j]]   (j in order;
 *            assignments dropped by a capacity limit, inv_perm < 0, add nothing)
 * Only the listed tokens (or all T when tokens == NULL) are written; out rows
 * are [n_tok, d] in the order of the list.
 * ------------------------------------------------------------------------- */
int oracle_combine(int64_t n_tok, const int64_t *tokens, int d, int k,
                   const double *y_perm, const int32_t *inv_perm, const double *topk_w,
                   double *out)
{
    for (int64_t q = 0; q < n_tok; ++q) {
        int64_t t = tokens ? tokens[q] : q;
        for (int o = 0; o < d; ++o) out[q * d + o] = 0.0;
        for (int j = 0; j < k; ++j) {
            if (inv_perm[t * k + j] < 0) continue;      /* dropped by a capacity limit */
            double w = topk_w[t * k + j];
            const double *yr = y_perm + (int64_t)inv_perm[t * k + j] * d;
            for (int o = 0; o < d; ++o) out[q * d + o] += w * yr[o];
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Whole layer on small inputs, [P3] s6.1 steps 1-5 / s5.1:
 *   route -> permute -> expert FFN per row -> combine.
 * Expert weights are stacked [N,F,d] / [N,d,F]. y_perm [T*k, d] fp64 out,
 * out [T, d] fp64. Routing outputs as in oracle_route / oracle_permute.
 * ------------------------------------------------------------------------- */
int oracle_forward(int64_t T, int d, int N, int k, int F, int act,
                   const void *x, int x_dt, const void *wg, int wg_dt, const void *bias, int b_dt, int bias_mode,
                   int gate_fp32,
                   const void *w_gate, const void *w_up, const void *w_down, int w_dt,
                   int32_t *topk_idx, double *topk_w, double *cert,
                   int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                   double *y_perm, double *out)
{
    const int64_t A = T * k;
    int rc = oracle_route(T, d, N, k, x, x_dt, wg, wg_dt, bias, b_dt, bias_mode, gate_fp32, topk_idx, topk_w, NULL,
                          NULL, cert, NULL);
    if (rc) return rc;
    rc = oracle_permute(T, N, k, topk_idx, counts, offsets, perm, inv_perm);
    if (rc) return rc;
    /* gather the permuted input rows, then run each expert on its rows */
    size_t es = (x_dt == OR_F64) ? 8 : (x_dt == OR_F32) ? 4 : 2;
    unsigned char *xp = (unsigned char *)malloc(es * (size_t)(A > 0 ? A : 1) * (size_t)d);
    if (!xp) return -1;
    for (int64_t row = 0; row < A; ++row)
        memcpy(xp + (size_t)row * d * es, (const unsigned char *)x + (size_t)perm[row] * d * es, (size_t)d * es);
    size_t wes = (w_dt == OR_F64) ? 8 : (w_dt == OR_F32) ? 4 : 2;
    for (int n = 0; n < N && rc == 0; ++n) {
        int64_t r0 = offsets[n], nr = counts[n];
        if (nr == 0) continue;
        rc = oracle_expert_rows(nr, d, F, act, xp + (size_t)r0 * d * es, x_dt,
                                (const unsigned char *)w_gate + (size_t)n * F * d * wes,
                                w_up ? (const unsigned char *)w_up + (size_t)n * F * d * wes : NULL,
                                (const unsigned char *)w_down + (size_t)n * d * F * wes, w_dt,
                                y_perm + r0 * d, NULL);
    }
    free(xp);
    if (rc) return rc;
    return oracle_combine(T, NULL, d, k, y_perm, inv_perm, topk_w, out);
}
