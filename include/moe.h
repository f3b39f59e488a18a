/*
 * moe.h -- C ABI of the GB300-native sparse Mixture-of-Experts feed-forward
 * layer (sm_103a).
 *
 * What the layer computes (the pages that define it):
 *   - "KochiLLM v1.0" model card, Architecture: the MoE FFN applies a shared
 *     expert to every token plus the top-2 of 4 routed experts; the gate
 *     weights are renormalised over the selected experts; the loss adds
 *     0.01 x (E x sum_i f_i p_i) for load balancing.  Configuration: SwiGLU
 *     experts with hidden 2 x dim.
 *   - "spark-gpt" README, feature list: bias-free fp32-softmax top-k routing,
 *     packed SwiGLU experts, BF16 grouped GEMM, selected-probability
 *     renormalisation (optional), and a load-balancing statistic over real
 *     (non-PAD) tokens only.
 *   - "KohakUwULLM" README, Key features: DeepSeekMoE with aux-loss-free load
 *     balancing (a per-expert bias that enters the selection only).
 *
 * Conventions (every entry point):
 *   - Returns MOE_OK (0) or a positive MOE_ERR_* code; nothing is thrown.
 *     moe_strerror() names a code.
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, row-major,
 *     16-byte aligned (MOE_ERR_ALIGN otherwise).  The library allocates no
 *     device or host memory; scratch lives in a caller-owned workspace of
 *     moe_workspace_bytes() bytes (MOE_ERR_WORKSPACE if smaller).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous; none synchronises the host.
 *   - Errors found on the device (expert index out of range, non-finite
 *     logits, a bounded wait that expired) are latched in a status word in
 *     the workspace; moe_get_status() synchronises the stream and reads it.
 *   - bf16 tensors are IEEE bfloat16 stored as uint16; fp32 is IEEE float.
 *   - Shape rules (MOE_ERR_SHAPE otherwise): T >= 1, d % 64 == 0,
 *     H % 64 == 0, 1 <= k <= min(E, 32), E <= 256, n_shared >= 0,
 *     H_shared % 64 == 0
 *     when n_shared > 0, T*k < 2^31, and every row count below < 2^31.
 *     The 64-multiples come from the GEMM tiling: one K step is 64 bf16
 *     values (one 128-byte swizzled row), and the gate/up epilogue writes
 *     hidden units in 64-wide halves, whose a|b copies would otherwise run
 *     into the neighbouring half of the ab row.
 *
 * Symbols: T positions (real + PAD), d model dim, E routed experts, k experts
 * per token, H routed expert hidden, Hs = n_shared * H_shared shared hidden,
 * M = T_real * k routed (token, slot) pairs, R_cap = moe_row_capacity().
 *
 * Routed rows ("permuted order").  Row r of x_perm/ab/h/out_perm holds one
 * (token, slot) pair; pairs are grouped by expert by a stable counting sort
 * (within an expert, ascending token).  Each expert's segment starts at a
 * multiple of MOE_ROW_ALIGN rows: expert e owns rows
 * [row_offsets[e], row_offsets[e+1]), of which the first counts[e] hold
 * pairs and the rest are zero pad rows (perm = -1).  offsets[] is the exact
 * exclusive scan of counts[] (the unpadded positions).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 6
#define MOE_ROW_ALIGN 128

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_NULL = 1,        /* a required pointer is NULL                  */
  MOE_ERR_SHAPE = 2,       /* configuration violates the shape rules      */
  MOE_ERR_ALIGN = 3,       /* a tensor pointer is not 16-byte aligned     */
  MOE_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than required     */
  MOE_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed        */
  MOE_ERR_DEVICE = 6,      /* current device is not sm_100-family (sm_103a build) */
  MOE_ERR_TIMEOUT = 7,     /* device: a bounded wait inside a kernel expired */
  MOE_ERR_INDEX = 8,       /* device: an expert index outside [0, E)      */
  MOE_ERR_NONFINITE = 9,   /* device: a router logit is NaN or infinite   */
  MOE_ERR_BOUNDS = 10      /* device, debug builds only: a row index read from
                            * inv or row_offsets lies outside the rows that
                            * exist (the access is skipped)                 */
};

/* Layer configuration (plain data, passed by pointer, read during the call). */
typedef struct moe_config {
  int32_t T;          /* positions per call (real tokens + PAD filler)         */
  int32_t d;          /* model dim                                              */
  int32_t E;          /* routed experts                                         */
  int32_t k;          /* experts selected per token                             */
  int32_t H;          /* hidden size of one routed expert                       */
  int32_t n_shared;   /* shared (always-on, ungated) experts; 0 = none          */
  int32_t H_shared;   /* hidden size of one shared expert                       */
  int32_t norm_topk;  /* 1: gates renormalised over the selected k; 0: raw p    */
  float aux_coef;     /* weight of aux in the objective differentiated by
                         moe_backward (KochiLLM card, Architecture: 0.01)       */
  float z_coef;       /* weight of the router z-loss in that objective (0 = off)
                         (KohakUwULLM README, Key features: z-loss)             */
} moe_config;

/*
 * Forward tensors.  Which fields a call reads (in) or writes (out) is listed
 * with each entry point; unused fields may be NULL.
 */
typedef struct moe_tensors {
  /* inputs */
  const void* x;        /* [T][d] bf16 token activations                          */
  const float* Wr;      /* [d][E] fp32 router weight (logits = x . Wr)           */
  const float* bias;    /* [E] fp32 selection-only bias, or NULL                 */
  const uint8_t* valid; /* [T] 1 = real token, 0 = PAD; NULL = all real          */
  const void* W_gu;     /* [E][2H][d] bf16: rows [0,H) gate, [H,2H) up           */
  const void* W_down;   /* [E][d][H] bf16                                        */
  const void* Ws_gu;    /* [2Hs][d] bf16 shared gate rows then up rows (n_shared
                           experts concatenated: expert s owns gate rows
                           [s*H_shared, (s+1)*H_shared) and the same up rows)    */
  const void* Ws_down;  /* [d][Hs] bf16 shared down (columns concatenated)        */
  /* routing */
  float* logits;        /* [T][E] fp32                                            */
  int32_t* topk_idx;    /* [T][k] selected experts, slot 0 = largest key; -1 PAD  */
  float* gates;         /* [T][k] fp32 gate weights; 0 on PAD                     */
  int32_t* counts;      /* [E] pairs routed to each expert (real tokens only)     */
  float* f;             /* [E] f_e = counts_e / (k T_real)                        */
  float* p;             /* [E] p_e = mean over real tokens of softmax_e           */
  float* aux;           /* [1] aux = E * sum_e f_e p_e                            */
  float* router_stats;  /* [8] fp32 routing metrics, or NULL to skip them:
                           [0] z_loss = mean over real tokens of logsumexp(L_t)^2
                           [1] router entropy, mean over real tokens of
                               -sum_e s_te ln s_te (nats)
                           [2] min_e counts_e   [3] max_e counts_e
                           [4] CV of counts (population std / mean)
                           [5] unused experts (counts_e == 0)
                           [6] T_real          [7] 0
                           ("spark-gpt" README: assignment min/max/CV, router
                           entropy, unused experts)                               */
  /* dispatch */
  int32_t* offsets;     /* [E+1] exclusive scan of counts (unpadded)              */
  int32_t* row_offsets; /* [E+1] padded segment starts (multiples of 128)        */
  int32_t* perm;        /* [R_cap] pair index t*k+j of each row; -1 = pad row    */
  int32_t* inv;         /* [T*k] row of pair (t,j); -1 for PAD tokens             */
  void* x_perm;         /* [R_cap][d] bf16 x rows in permuted order (pad rows 0) */
  /* experts */
  void* ab;             /* [R_cap][2H] bf16 pre-activations a|b (saved for
                           backward; NULL skips the save)                         */
  void* h;              /* [R_cap][H] bf16 silu(a) * b                            */
  void* out_perm;       /* [R_cap][d] bf16 expert output per row (each slot's
                           output, summed by the combine in fp32)                 */
  void* s_ab;           /* [T][2Hs] bf16 shared pre-activations (or NULL)         */
  void* s_h;            /* [T][Hs] bf16 shared hidden (0 on PAD rows)             */
  float* s_out;         /* [T][d] fp32 shared expert output (0 on PAD rows):
                           written by moe_shared_ffn and read by moe_combine;
                           moe_forward and moe_shared_ffn_combine do not use it
                           (may be NULL for them)                               */
  /* output */
  void* y;              /* [T][d] bf16 layer output                               */
} moe_tensors;

/* Backward tensors (gradients of J = <dY, y> + aux_coef * aux + z_coef * z_loss). */
typedef struct moe_grads {
  const void* dY;       /* [T][d] bf16 upstream gradient of y                     */
  void* dx;             /* [T][d] bf16 gradient of x (expert, shared and router
                           paths)                                                 */
  float* dWr;           /* [d][E] fp32                                            */
  void* dW_gu;          /* [E][2H][d] bf16                                        */
  void* dW_down;        /* [E][d][H] bf16                                         */
  void* dWs_gu;         /* [2Hs][d] bf16 (NULL when n_shared == 0)                */
  void* dWs_down;       /* [d][Hs] bf16                                           */
  float* d_logits;      /* [T][E] fp32 gradient of the router logits, including
                           the aux term (f held constant) and the z-loss term    */
} moe_grads;

/* ---------------------------------------------------------------- queries */

/* ABI version (MOE_ABI_VERSION). */
int moe_abi_version(void);

/* 1 if this library was built with the debug bounds checks (MOE_DEBUG_BOUNDS:
 * row indices read from inv and row_offsets are checked on the device,
 * MOE_ERR_BOUNDS latched and the access skipped), else 0. */
int moe_debug_bounds(void);

/* Static message for a status code (never NULL). */
const char* moe_strerror(int code);

/* MOE_OK if *cfg satisfies the shape rules above, else MOE_ERR_SHAPE/NULL. */
int moe_check_config(const moe_config* cfg);

/* Rows a permuted buffer must hold: the largest padded row total,
 * floor((T*k + (MOE_ROW_ALIGN-1)*E) / MOE_ROW_ALIGN) * MOE_ROW_ALIGN.        */
int moe_row_capacity(const moe_config* cfg, int64_t* rows);

/* Workspace bytes for forward (training = 0) or forward + backward
 * (training = 1).  The same workspace must be passed to every call of one
 * layer step; its contents between calls are private to the library. */
int moe_workspace_bytes(const moe_config* cfg, int training, size_t* bytes);

/* Byte offsets, within a training workspace (moe_workspace_bytes with
 * training = 1), of the intermediates moe_backward stores there, for
 * inspection by tests and debuggers after the call:
 *   out[0] d_out   [R_cap][d]  bf16  g * dY of each routed row
 *   out[1] d_gu    [R_cap][2H] bf16  (da | db) of each routed row
 *   out[2] dx_perm [R_cap][d]  bf16  the dX product of each routed row
 *   out[3] ds_gu   [T][2Hs]    bf16  the shared expert's (da | db); 0 when
 *                                    n_shared == 0
 * Rows follow perm (pad rows hold unspecified values).  The layout is part
 * of this ABI version only.  Host-side query: nothing runs on the device. */
int moe_workspace_offsets(const moe_config* cfg, size_t* out);

/* Synchronise `stream`, copy the device status word to *status and reset it
 * to MOE_OK.  The only entry point that blocks the host. */
int moe_get_status(void* workspace, void* stream, int* status);

/* Self-test of the device failure path: one GPU thread waits, with the
 * bounded wait every GEMM role uses, on an mbarrier that nothing arrives on;
 * after limit_ns (1 ns .. 10 s) it gives up, stores MOE_ERR_TIMEOUT in the
 * workspace status word (read it with moe_get_status) and the kernel returns
 * normally -- no trap, no fault, the context stays usable.  Asynchronous on
 * `stream`.  Errors: NULL, SHAPE (limit out of range), DEVICE. */
int moe_selftest_wait_timeout(void* workspace, uint64_t limit_ns, void* stream);

/* ---------------------------------------------------------------- forward */

/* a0. logits = x . Wr in fp32 (x widened exactly from bf16).
 * "spark-gpt" README, feature list: bias-free router, fp32 routing.
 * in: x, Wr.  out: logits. */
int moe_router_logits(const moe_config* cfg, const moe_tensors* t,
                      void* workspace, size_t workspace_bytes, void* stream);

/* a1. Top-k routing and the load-balancing statistic.
 * "KochiLLM v1.0" card, Architecture; "spark-gpt" README, feature list.
 * key = logits (+ bias, one fp32 add); the k largest keys are selected, equal
 * keys lower index first; s = fp32 softmax(logits) over all E (unbiased);
 * gates = s_sel / sum s_sel if norm_topk else s_sel; counts, f, p, aux over
 * real tokens.  in: logits, bias, valid.
 * out: topk_idx, gates, counts, f, p, aux, router_stats (if non-NULL).
 * Device errors: NONFINITE. */
int moe_route(const moe_config* cfg, const moe_tensors* t,
              void* workspace, size_t workspace_bytes, void* stream);

/* a0 + a1 in one call: the same results as moe_router_logits followed by
 * moe_route (logits may differ from moe_router_logits' in the last bits,
 * since the fp32 sums are added in another order; the routing is taken on
 * the logits this call writes).  For E of 4, 8 or 16 with Wr in 96 KiB this
 * is one kernel that reads x once and never reads the logits back; otherwise
 * it runs the two steps.  "spark-gpt" README, feature list (fp32-softmax
 * top-k router).  in: x, Wr, bias, valid.  out: logits and the outputs of
 * moe_route.  Device errors: NONFINITE. */
int moe_router_route(const moe_config* cfg, const moe_tensors* t,
                     void* workspace, size_t workspace_bytes, void* stream);

/* a2. Stable counting-sort dispatch into expert-contiguous padded rows: the
 * layout a grouped GEMM over the experts needs ("spark-gpt" README, feature
 * list: BF16 grouped GEMM over packed SwiGLU experts; Hard-won facts: the
 * experts run on grouped GEMMs, not a per-expert loop).  Pair (t, j) with
 * t*k + j as the sort key goes to expert topk_idx[t][j]'s segment, tokens in
 * ascending order within it.
 * in: x, topk_idx.  out: counts, offsets, row_offsets, perm, inv, x_perm.
 * x_perm may be NULL: then no rows are copied, and moe_expert_gate_up (with
 * x_perm NULL too) gathers the rows from x through perm instead.  The
 * backward needs x_perm, so a training forward passes it.
 * Device errors: INDEX (the pair is then dropped). */
int moe_permute(const moe_config* cfg, const moe_tensors* t,
                void* workspace, size_t workspace_bytes, void* stream);

/* a3. Grouped gate/up GEMM with SwiGLU in the epilogue (tcgen05, bf16 in,
 * fp32 accumulate): per expert e and row r of its segment,
 * a = x_perm[r] W_gate[e]^T, b = x_perm[r] W_up[e]^T, h[r] = silu(a) * b.
 * "KochiLLM v1.0" card (SwiGLU experts); "spark-gpt" README, Hard-won facts
 * (grouped GEMM with the SwiGLU fused into the epilogue).
 * With x_perm NULL the permute is folded into the GEMM's A load: row r is
 * token perm[r] / k of x, fetched by TMA four rows at a time (tile::gather4),
 * pad rows read as zeros -- the same products as from x_perm, without the
 * x_perm buffer (2 d T k bytes); a memory-saving mode, several times slower
 * than copied rows on GB300 (the gathers, not the MMAs, set its pace).
 * in: x_perm (or x and perm), row_offsets, W_gu.  out: h, ab (if non-NULL). */
int moe_expert_gate_up(const moe_config* cfg, const moe_tensors* t,
                       void* workspace, size_t workspace_bytes, void* stream);

/* a4. Grouped down GEMM: out_perm[r] = h[r] W_down[e]^T (tcgen05, bf16 in,
 * fp32 accumulate, bf16 out).  The down projection of each SwiGLU expert
 * ("KochiLLM v1.0" card, Configuration: SwiGLU experts, hidden 2 x dim), run
 * as one grouped GEMM over all experts' segments ("spark-gpt" README,
 * Hard-won facts: the MoE experts run on hand-written grouped GEMMs).
 * in: h, row_offsets, W_down.  out: out_perm. */
int moe_expert_down(const moe_config* cfg, const moe_tensors* t,
                    void* workspace, size_t workspace_bytes, void* stream);

/* a5. Shared expert on every real token ("KochiLLM v1.0" card, Architecture):
 * s_out[t] = SwiGLU_shared(x[t]) for real t, 0 on PAD.  No-op if n_shared=0.
 * in: x, valid, Ws_gu, Ws_down.  out: s_h, s_out, s_ab (if non-NULL). */
int moe_shared_ffn(const moe_config* cfg, const moe_tensors* t,
                   void* workspace, size_t workspace_bytes, void* stream);

/* a6. Weighted un-permute: y[t] = sum_j gates[t][j] out_perm[inv[t,j]]
 * (+ s_out[t]), fp32 sum in slot order, one rounding to bf16; PAD rows 0.
 * The MoE FFN's output: the shared expert on every token plus the selected
 * routed experts weighted by their renormalised gates ("KochiLLM v1.0" card,
 * Architecture). 
 * in: out_perm, inv, gates, valid, s_out (if n_shared > 0).  out: y. */
int moe_combine(const moe_config* cfg, const moe_tensors* t,
                void* workspace, size_t workspace_bytes, void* stream);

/* a5 + a6 in one call.  With a shared expert (n_shared > 0) the combine runs
 * in the epilogue of the shared expert's down GEMM: for token t the fp32 sum
 * over slots j of gates[t][j] * out_perm[inv[t][j]] (slot order, unused
 * slots skipped) plus the shared output, one rounding to bf16 -- the same
 * operations, in the same order, as moe_shared_ffn followed by moe_combine,
 * so y is identical; s_out is neither written nor read.  Without a shared
 * expert it is moe_combine.  "KochiLLM v1.0" card, Architecture (shared
 * expert beside the routed top-k).  in: x, valid, Ws_gu, Ws_down, out_perm,
 * inv, gates.  out: s_h, s_ab (if non-NULL), y. */
int moe_shared_ffn_combine(const moe_config* cfg, const moe_tensors* t,
                           void* workspace, size_t workspace_bytes, void* stream);

/* a3 + a4 + a5: the experts in one call -- moe_expert_gate_up,
 * moe_expert_down, then moe_shared_ffn (no-op without a shared expert), in
 * that order on `stream`.  The experts of the MoE FFN: SwiGLU experts
 * ("KochiLLM v1.0" card, Configuration), routed ones on their tokens' rows
 * and the shared one on every token (Architecture), as grouped GEMMs with the
 * SwiGLU in the gate/up epilogue ("spark-gpt" README, Hard-won facts).
 * in: x_perm (or x and perm, see moe_expert_gate_up), row_offsets, W_gu,
 * W_down, and with a shared expert x, valid, Ws_gu, Ws_down.
 * out: h, ab (if non-NULL), out_perm, and with a shared expert s_h, s_out,
 * s_ab (if non-NULL).  moe_combine then forms y. */
int moe_expert_ffn(const moe_config* cfg, const moe_tensors* t,
                   void* workspace, size_t workspace_bytes, void* stream);

/* a0..a6 in order on one stream (a0 + a1 as moe_router_route, a5 + a6 as
 * moe_shared_ffn_combine). */
int moe_forward(const moe_config* cfg, const moe_tensors* t,
                void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------ data-parallel statistics */

/* One data-parallel exchange ("spark-gpt" README: hard counts are
 * synchronised across DDP ranks and the differentiable local proxy is
 * scaled so DDP averaging yields the global-batch gradient).  Each rank
 * routes its own tokens, exports its sums with moe_route_partials, the
 * caller all-reduces (sums) them with its collective library, and
 * moe_route_finalize turns the global sums into the global f, p and aux.
 *
 * moe_route_partials: in: counts, p (from moe_route on this rank's tokens).
 * out: sums [2E+1] fp64 device = { counts_e (E), p_e * T_real (E), T_real }.
 * T_real is sum(counts) / k. */
int moe_route_partials(const moe_config* cfg, const moe_tensors* t, double* sums, void* stream);

/* moe_route_finalize: in: sums [2E+1] fp64 device (already summed over the
 * ranks).  out: f, p, aux of `t` for the whole data-parallel batch
 * (f_e = counts_e / (k T), p_e = psum_e / T, aux = E sum f p).  counts keep
 * the rank's own values.  For the backward of the global objective, scale
 * aux_coef and z_coef by T_real(rank) / T_real(global), and by the rank
 * count when the caller's gradient reduction averages over ranks. */
int moe_route_finalize(const moe_config* cfg, const moe_tensors* t, const double* sums,
                       void* stream);

/* ---------------------------------------------------------------- backward */

/* a7. Gradients of J = <dY, y> + aux_coef * aux + z_coef * z_loss with the
 * hard counts (f) held constant; the selection bias receives no gradient.
 * The training objective of the layer: the loss adds 0.01 x (E x sum_i f_i
 * p_i) for load balancing ("KochiLLM v1.0" card, Architecture), p being the
 * differentiable proxy and the hard counts f not differentiated ("spark-gpt"
 * README, compute-matched MoE paragraph); the router z-loss ("KohakUwULLM"
 * README, Key features) enters through z_coef.
 * Reads every forward tensor of `t` written by moe_forward (x, Wr, valid,
 * weights, logits, topk_idx, gates, counts, f, row_offsets, inv, x_perm, ab,
 * h, out_perm, s_ab, s_h); ab and (if n_shared > 0) s_ab must have been saved.
 * Writes every field of `g` (dWs_* only when n_shared > 0).
 * Steps: combine backward (d_out = g dY, dg = <dY, out_perm>), router-logit
 * gradient with the aux term, grouped dH GEMM with the SwiGLU backward in its
 * epilogue, grouped dX GEMM, ragged-K grouped dW GEMMs, the shared expert's
 * backward, the router's input gradients, and the un-permute sum of dx. */
int moe_backward(const moe_config* cfg, const moe_tensors* t, const moe_grads* g,
                 void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------ MXFP8 experts */

/* The experts in MXFP8 ("KohakUwULLM" README, Key features: e4m3 values with
 * UE8M0 scales, one per 32 values, on the feed-forward pair and the routed
 * experts, with fully fused MXFP8 expert kernels).  Forward only (inference).
 * The routed experts and the shared expert (the dense feed-forward pair) run
 * on MXFP8 operands; router, route and combine are the bf16 path's.
 *
 * Format.  A block is 32 consecutive values along the reduction axis of a
 * product (d for x and the gate/up rows, H for h and the down rows).  Its
 * scale byte is X + 127 with X = floor(log2 max|v|) - 8, clamped to >= -127
 * (all-zero blocks: -127); each value is the e4m3 code of v / 2^X, rounded to
 * nearest even and saturated to +-448.  Codes keep the element order of the
 * bf16 tensor they replace.  Scale bytes sit in 512-byte atoms, each covering
 * 128 rows x 4 blocks (128 values along K): row r, block kb at byte
 * (r % 32) * 16 + (r / 32) * 4 + kb; atoms are indexed [128-row block][K/128].
 *
 * Shapes: d a multiple of 256, H and n_shared * H_shared of 128, else
 * MOE_ERR_SHAPE.  All buffers are caller-owned device memory, 16-byte aligned,
 * and the code buffers and t->out_perm 32-byte aligned (the kernels store 32
 * bytes per thread), else MOE_ERR_ALIGN; moe_mx_sizes gives their sizes. */
typedef struct moe_mx_tensors {
  uint8_t* W_gu_q;    /* [E][2H][d] codes of W_gu                                */
  uint8_t* W_gu_s;    /* [E][2H/128][d/128] atoms (128-row blocks of W_gu[e])    */
  uint8_t* W_down_q;  /* [E][d][H] codes of W_down                               */
  uint8_t* W_down_s;  /* [E][d/128][H/128] atoms                                 */
  uint8_t* x_q;       /* [R_cap][d] permuted x rows (pad rows zero)              */
  uint8_t* x_s;       /* [R_cap/128][d/128] atoms                                */
  uint8_t* h_q;       /* [R_cap][H] hidden rows                                  */
  uint8_t* h_s;       /* [R_cap/128][H/128] atoms                                */
  /* the shared expert (n_shared > 0; Hs = n_shared * H_shared, Tp = T rounded
     up to a multiple of 128); unused without a shared expert                */
  uint8_t* Ws_gu_q;   /* [2Hs][d] codes of Ws_gu                                 */
  uint8_t* Ws_gu_s;   /* [2Hs/128][d/128] atoms                                  */
  uint8_t* Ws_down_q; /* [d][Hs] codes of Ws_down                                */
  uint8_t* Ws_down_s; /* [d/128][Hs/128] atoms                                   */
  uint8_t* xt_q;      /* [Tp][d] x in token order (PAD and padding rows zero)    */
  uint8_t* xt_s;      /* [Tp/128][d/128] atoms                                   */
  uint8_t* hs_q;      /* [Tp][Hs] the shared expert's hidden rows                */
  uint8_t* hs_s;      /* [Tp/128][Hs/128] atoms                                  */
  /* the training step's data gradients (moe_mx_backward); unused otherwise  */
  uint8_t* W_gu_tq;   /* [E][d][2H] codes of each W_gu[e]^T: blocks along 2H     */
  uint8_t* W_gu_ts;   /* [E][d/128][2H/128] atoms                                */
  uint8_t* W_down_tq; /* [E][H][d] codes of each W_down[e]^T: blocks along d     */
  uint8_t* W_down_ts; /* [E][H/128][d/128] atoms                                 */
  uint8_t* dout_q;    /* [R_cap][d] codes of d_out = g dY (blocks along d)       */
  uint8_t* dout_s;    /* [R_cap/128][d/128] atoms                                */
  uint8_t* dgu_q;     /* [R_cap][2H] codes of d_gu = da | db (blocks along 2H)   */
  uint8_t* dgu_s;     /* [R_cap/128][2H/128] atoms                               */
  void* ab16;         /* [R_cap][2H] fp16 the forward's a | b, for the chain rule */
} moe_mx_tensors;

#define MOE_MX_FIELDS 25

/* Bytes of each field of moe_mx_tensors, in field order, into bytes[25]
 * (the shared expert's eight are 0 without one). */
int moe_mx_sizes(const moe_config* cfg, size_t* bytes);

/* Weights -> MXFP8: in: t->W_gu, t->W_down (and Ws_gu, Ws_down with a shared
 * expert), bf16.  out: W_gu_q, W_gu_s, W_down_q, W_down_s (and Ws_*_q, Ws_*_s),
 * and, when W_gu_tq / W_down_tq are non-NULL (training), each expert's
 * transposed weights quantised along the axis the data-gradient products
 * sum over: W_gu_tq/ts, W_down_tq/ts.  Run once per weight update. */
int moe_mx_quantize_weights(const moe_config* cfg, const moe_tensors* t,
                            const moe_mx_tensors* mx, void* stream);

/* a2 with the rows quantised: offsets, perm, inv exactly as moe_permute,
 * and x_q / x_s instead of x_perm (each token's row quantised once).
 * in: x, topk_idx.  out: counts, offsets, row_offsets, perm, inv, x_q, x_s. */
int moe_mx_permute(const moe_config* cfg, const moe_tensors* t, const moe_mx_tensors* mx,
                   void* workspace, size_t workspace_bytes, void* stream);

/* a3 on MXFP8 operands: a = x_q W_gate_q^T, b = x_q W_up_q^T (block-scaled
 * tcgen05 MMAs, fp32 accumulate), h = silu(a) * b quantised straight to h_q
 * / h_s in the epilogue.  in: x_q, x_s, row_offsets, W_gu_q, W_gu_s.
 * out: h_q, h_s. */
int moe_mx_expert_gate_up(const moe_config* cfg, const moe_tensors* t, const moe_mx_tensors* mx,
                          void* workspace, size_t workspace_bytes, void* stream);

/* a4 on MXFP8 operands: out_perm = h_q W_down_q^T (fp32 accumulation, bf16
 * rows).
 * in: h_q, h_s, row_offsets, W_down_q, W_down_s.  out: out_perm. */
int moe_mx_expert_down(const moe_config* cfg, const moe_tensors* t, const moe_mx_tensors* mx,
                       void* workspace, size_t workspace_bytes, void* stream);

/* a5 on MXFP8 operands: x quantised in token order (PAD tokens as zeros),
 * the block-scaled gate/up GEMM with the SwiGLU and h quantiser, the
 * block-scaled down GEMM -> s_out (fp32; 0 on PAD rows).  No-op without a
 * shared expert.  in: x, valid, Ws_gu_q/s, Ws_down_q/s.
 * out: xt_q/s, hs_q/s, s_out. */
int moe_mx_shared_ffn(const moe_config* cfg, const moe_tensors* t, const moe_mx_tensors* mx,
                      void* workspace, size_t workspace_bytes, void* stream);

/* The forward with MXFP8 experts: moe_router_route, moe_mx_permute,
 * moe_mx_expert_gate_up, moe_mx_expert_down, moe_mx_shared_ffn, moe_combine.
 * With a shared expert its permute also writes x's token-order codes
 * (xt_q / xt_s), so x is read and quantised once and moe_mx_shared_ffn's own
 * quantiser pass is skipped; y is the same as from the separate calls.
 * The weights must have been quantised (moe_mx_quantize_weights). */
int moe_mx_forward(const moe_config* cfg, const moe_tensors* t, const moe_mx_tensors* mx,
                   void* workspace, size_t workspace_bytes, void* stream);

/* The forward of the MXFP8 training step ("KohakUwULLM" README, Key
 * features: native MXFP8 training of the routed experts; Selected
 * measurements: MXFP8 end-to-end training speed-ups on MoE models).  The
 * routed experts run as in moe_mx_forward; the shared expert runs in bf16
 * (moe_shared_ffn_combine, the combine in its down GEMM).  It also stores
 * what moe_mx_backward needs: x_perm (bf16 rows), h (bf16, before its MX
 * rounding), mx->ab16 (the pre-activations a | b in fp16, magnitudes past
 * 65504 clamped: the chain rule's results are quantised to e4m3, whose codes
 * a bf16 copy of its inputs (8 significant bits to fp16's 11) would move
 * about 8 times as often) and out_perm.  t->ab is not used.
 * in: as moe_mx_forward.  out: as moe_mx_forward plus x_perm, h, ab16, and
 * the shared expert's s_h, s_ab (if non-NULL). */
int moe_mx_forward_train(const moe_config* cfg, const moe_tensors* t, const moe_mx_tensors* mx,
                         void* workspace, size_t workspace_bytes, void* stream);

/* The backward of the MXFP8 training step: moe_backward with the routed
 * experts' two data-gradient products on MXFP8 operands, each quantised in
 * blocks of 32 along the product's reduction axis: d_out = g dY is
 * quantised along d (dout_q/s) from its fp32 value, in the kernel that forms
 * it; dH = Q(d_out) Q(W_down[e]^T) runs on the block-scaled tcgen05 kernel
 * with the SwiGLU chain rule (on ab16) in its epilogue, which quantises the
 * fp32 d_gu = da | db along 2H (dgu_q/s) and stores it in bf16 for the
 * weight gradient; and dx = Q(d_gu) Q(W_gu[e]^T), written as bf16 dx_perm
 * rows.  Each MX operand is thus one rounding of its fp32 value, never of a
 * bf16 copy.  The weight gradients, the shared expert and the router are
 * moe_backward's (bf16 operands, fp32 accumulation).  Needs a
 * training workspace (moe_workspace_bytes with training = 1), the forward
 * tensors of moe_mx_forward_train, the transposed weight codes of
 * moe_mx_quantize_weights, ab16, and dout_q/s, dgu_q/s (32-byte aligned
 * codes).
 * out: every field of `g`, as moe_backward. */
int moe_mx_backward(const moe_config* cfg, const moe_tensors* t, const moe_mx_tensors* mx,
                    const moe_grads* g, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------- no-allocation routing */

/* Bytes of the fixed device scratch array behind moe_route_static (per GPU). */
#define MOE_ROUTE_STATIC_SCRATCH_BYTES (512 * 1024)

/* a1 without a workspace.  The pages have no counterpart to this entry point;
 * it exists for callers that cannot allocate device memory at all -- code
 * running under a host framework that owns every allocation, inside a region
 * where cudaMalloc is forbidden, or with a fixed memory plan -- and so cannot
 * supply the workspace moe_route needs.
 *
 * Computes exactly what moe_route computes (same kernel, same launch shape,
 * same bytes out).  Reads logits, bias, valid; writes topk_idx, gates,
 * counts, f, p, aux of `t` (other fields are ignored).  `device_status` is an
 * optional device int (NULL = not reported) where a device-side error
 * (MOE_ERR_NONFINITE) is stored if it is still 0; the caller clears it.
 *
 * Scratch: a fixed array of MOE_ROUTE_STATIC_SCRATCH_BYTES in the library's
 * device memory, held by every GPU that loads the library until the process
 * exits.  A call needs 3328 + 4 B bytes of it, B <= 456 being the route
 * kernel's block count (the same grid as moe_route), so every valid
 * configuration fits (MOE_ERR_WORKSPACE is kept as a guard).
 * Set-up: the first call on each device resolves the array's device address
 * (a runtime symbol query, no allocation); make that first call before any
 * stream capture.  If that query fails the call returns MOE_ERR_CUDA and
 * nothing is cached: the next call on the device queries again.  The call itself allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 * Sharing: all calls on a GPU use the same array, which keeps the last call's
 * contents; the ticket counter that must start at zero is cleared at the
 * start of each call.  Calls that overlap on the GPU (two streams at once)
 * race on the array: serialise them. */
int moe_route_static(const moe_config* cfg, const moe_tensors* t, int* device_status,
                     void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
