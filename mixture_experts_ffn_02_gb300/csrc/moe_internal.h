// Host-side declarations shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kRowAlign = MOE_ROW_ALIGN;  // expert segments start at multiples
constexpr size_t kRouteAccCnt = 256;
constexpr size_t kRouteAccPsum = kRouteAccCnt + 256 * 4;
constexpr size_t kRouteAccBytes = kRouteAccPsum + 256 * 8;   // E <= 256
constexpr int kPermChunk = 128;           // tokens per block in the dispatch kernels
constexpr int kMaxK = 32;                 // experts per token supported
constexpr int kDwTokPerBlk = 128;         // tokens per slice of a small-E dW_r block

// Per-device facts, cached after the first query.
struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int cc_major = 0;
  int cc_minor = 0;
  size_t max_smem_optin = 0;
};
int device_info(DeviceInfo* out);

// ---- workspace layout (byte offsets into the caller's workspace) -----------
struct WsLayout {
  size_t status;        // int32 status word
  size_t route_done;    // route totals, zeroed before each routing launch
                        // (kRouteAccBytes): ticket counter at +0, expert
                        // counts int32 [E] at +kRouteAccCnt, probability sums
                        // in 2^-32 fixed point uint64 [E] at +kRouteAccPsum
  size_t route_treal;   // [route_blocks] int32
  size_t route_zent;    // [route_blocks][2] fp32 (z-loss, entropy partials)
  size_t perm_hist;     // [perm_blocks][E] int32
  size_t perm_base;     // [perm_blocks][E] int32
  // backward scratch
  size_t d_out;         // [R_cap][d] bf16
  size_t d_gu;          // [R_cap][2H] bf16
  size_t dx_perm;       // [R_cap][d] fp32
  size_t ds_gu;         // [T][2Hs] bf16
  size_t dxr;           // [T][d] fp32 (router input gradient, large E)
  size_t dwr_part;      // [splits][d][E] fp32
  // tensor-core router (router_tc_path)
  size_t wr2;           // [d][3E] bf16
  size_t dl3;           // [T][3E] bf16
  size_t dl2;           // [2 Tp][E] bf16
  size_t goff;          // [G+1] int32 split-K row groups
  size_t total;
  int route_blocks;
  int perm_blocks;
  int dwr_splits;
  int64_t R_cap;
};
int ws_layout(const moe_config* c, int training, WsLayout* out);

// ---- launchers of the memory-bound / SIMT kernels (moe_dispatch.cu) --------
cudaError_t launch_router_logits(const moe_config& c, const void* x, const float* Wr,
                                 float* L, cudaStream_t s);
// a0 + a1 fused (router_small_path only).
cudaError_t launch_router_route(const moe_config& c, const void* x, const float* Wr,
                                const float* bias, const uint8_t* valid, float* L, int32_t* topk,
                                float* gates, int32_t* counts, float* f, float* p, float* aux,
                                float* stats, char* ws, const WsLayout& w, cudaStream_t s);
cudaError_t launch_route(const moe_config& c, const float* L, const float* bias,
                         const uint8_t* valid, int32_t* topk, float* gates, int32_t* counts,
                         float* f, float* p, float* aux, float* stats, char* ws,
                         const WsLayout& w, cudaStream_t s);
// `acc` is a route-totals region of kRouteAccBytes (layout as WsLayout::
// route_done); it is zeroed here before the kernel.
cudaError_t launch_route_scratch(const moe_config& c, const float* L, const float* bias,
                                 const uint8_t* valid, int32_t* topk, float* gates,
                                 int32_t* counts, float* f, float* p, float* aux, char* acc,
                                 int* blk_treal, int* status, int grid, cudaStream_t s);
cudaError_t launch_route_partials(const moe_config& c, const int32_t* counts, const float* p,
                                  double* sums, cudaStream_t s);
cudaError_t launch_route_finalize(const moe_config& c, const double* sums, float* f, float* p,
                                  float* aux, cudaStream_t s);
cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* topk,
                           int32_t* counts, int32_t* offsets, int32_t* row_offsets,
                           int32_t* perm, int32_t* inv, void* x_perm, char* ws,
                           const WsLayout& w, cudaStream_t s);
// rows: the permuted rows that exist (R_cap); status: the workspace status
// word, where debug builds latch MOE_ERR_BOUNDS for an inv entry past rows.
cudaError_t launch_combine(const moe_config& c, const void* out_perm, const int32_t* inv,
                           const float* gates, const uint8_t* valid, const float* s_out,
                           void* y, long long rows, int* status, cudaStream_t s);
cudaError_t launch_combine_bwd(const moe_config& c, const void* dY, const void* out_perm,
                               const int32_t* inv, const int32_t* topk, const float* gates,
                               const float* L, const float* f, const int32_t* counts,
                               const uint8_t* valid, const int32_t* row_offsets,
                               void* d_out, uint8_t* dout_q, uint8_t* dout_s,
                               float* d_logits, long long rows, int* status, cudaStream_t s);
cudaError_t launch_dx_gather(const moe_config& c, const void* dx_perm, const int32_t* inv,
                             const float* dxr, const float* d_logits,
                             const float* Wr, const uint8_t* valid, void* dx, long long rows,
                             int* status, cudaStream_t s);
// Router GEMMs on the CUDA cores (fp32 FMA).
cudaError_t launch_router_dx(const moe_config& c, const float* d_logits, const float* Wr,
                             float* dxr, cudaStream_t s);
cudaError_t launch_router_dw(const moe_config& c, const void* x, const float* d_logits,
                             float* dWr, float* part, int splits, cudaStream_t s);
// Lanes that route one token: the power of two >= E, at least 8 (so the
// fused small-E router and the route kernel share one token-to-lane layout)
// and at most 32.
int route_group_lanes(int E);
bool router_small_path(const moe_config& c);
// Router backward products on the tensor cores (E a multiple of 32 beyond the
// small path): moe_router_tc.cu.
bool router_tc_path(const moe_config& c);
void router_tc_sizes(const moe_config& c, int* Tp, int* G, int* chunk);
cudaError_t launch_router_bwd_tc(const moe_config& c, const void* x, const float* dL,
                                 const float* Wr, float* dxr, float* dWr, void* wr2, void* dl3,
                                 void* dl2, int* goff, float* part, int* status, cudaStream_t s);
cudaError_t launch_sum_splits(const float* part, float* out, int n, int splits, cudaStream_t s);
int router_dw_small_parts(const moe_config& c);   // partial slices of the small-E dW_r

// ---- tcgen05 grouped GEMMs (moe_gemm.cu) -----------------------------------
// Which product a launch computes (operand majorness and epilogue).
enum GemmKind {
  GK_GATE_UP = 0,   // h = silu(A Wg^T) * (A Wu^T)          A K-major, B K-major
  GK_DOWN = 1,      // out = A Wd^T                          A K-major, B K-major
  GK_DH = 2,        // d_gu = swiglu_bwd(A Wd, ab)           A K-major, B MN-major
  GK_DX = 3,        // dx = A Wgu                            A K-major, B MN-major
  GK_DW = 4         // dW = A^T B over a row segment         A MN-major, B MN-major
};

struct GemmCall {
  GemmKind kind;
  // Row grouping: routed (row_offsets != NULL, E groups) or dense (rows).
  const int32_t* row_offsets;  // [E+1] padded, device
  int E;                       // groups (1 for dense)
  int rows;                    // dense: number of rows; routed: R_cap
  // Operand A (activations)
  const void* A;               // [rows][lda] bf16
  int lda;                     // elements
  // Operand B (weights) or second activation (GK_DW)
  const void* B;
  // Problem dims
  int K;                       // reduction length (not for GK_DW)
  int N;                       // output columns (H for gate/up, d for down, ...)
  int H;                       // gate/up split (GK_GATE_UP: rows [0,H) gate; GK_DH)
  int Mdw;                     // GK_DW: rows of each dW matrix
  // Outputs
  void* out0;                  // main output
  int ld0;
  int out_f32;                 // GK_DOWN / GK_DX / GK_DW: store fp32 instead of bf16
  int a_mod;                   // GK_DOWN: A's K coordinate mod a_mod (A repeated along K);
                               // GK_DW: A's row coordinate mod a_mod
  int a_rows;                  // GK_DW: rows of A when they differ from B's (0 = rows)
  void* out1;                  // GK_GATE_UP: ab save (or NULL)
  int ld1;
  const void* aux_in;          // GK_DH: ab (a|b) saved by the forward
  int ld_aux;
  const uint8_t* valid;        // GK_GATE_UP dense: zero PAD rows; combine: PAD tokens
  int* status;
  // GK_DOWN over dense token rows with the combine folded into the epilogue:
  // out0 = y (bf16) = sum_j comb_gates[t][j] comb_src[comb_inv[t][j]] + result
  const void* comb_src;        // out_perm (dx_perm) [R][N] bf16, or NULL (no fold)
  const int32_t* comb_inv;     // [rows][comb_k], -1 = unused slot
  int comb_rows;               // rows of comb_src (R_cap), for debug bounds checks
  const float* comb_gates;     // [rows][comb_k]
  int comb_k;
  // GK_DX over dense token rows with the dx gather folded into the epilogue:
  // out0 = dx (bf16) = sum_j comb_src[comb_inv[t][j]] + result + router term,
  // the router term sum_e dl[t][e] wr[c][e] (rE in {4, 8, 16}) or dxr[t][c]
  const float* dl;             // d_logits [rows][rE]
  const float* wr;             // W_r [N][rE]
  int rE;                      // 0: no inline router term
  const float* dxr;            // [rows][N] fp32 router term, or NULL
  // GK_GATE_UP with the permute folded into the A load: A is x [gT][K] and row
  // r of the padded permuted layout is token gperm[r] / gk (pad rows: zeros)
  const int32_t* gperm;        // perm [grows], -1 on pad rows; NULL = A is given
  int gk;
  int gT;
  int grows;
};
cudaError_t launch_gemm(const GemmCall& g, cudaStream_t s);

// ---- MXFP8 routed experts (moe_mx.cu) --------------------------------------
// Quantising permute: offsets, perm, inv as launch_permute, and x rows as
// e4m3 codes x_q [R_cap][d] with scale atoms x_s [R_cap/128][d/128][512];
// with xt_q non-NULL also the same codes in token order (xt_q [Tp][d], xt_s;
// PAD tokens and rows T..Tp-1 as zeros) for the shared expert.
cudaError_t launch_permute_mx(const moe_config& c, const void* x, const int32_t* topk,
                              int32_t* counts, int32_t* offsets, int32_t* row_offsets,
                              int32_t* perm, int32_t* inv, uint8_t* x_q, uint8_t* x_s,
                              uint8_t* xt_q, uint8_t* xt_s, void* x_perm, char* ws,
                              const WsLayout& w, cudaStream_t s);
// Rows of a bf16 [rows][K] matrix -> codes [rows][K] and scale atoms per
// 128-row block of each group of rows_per_group rows; rows past rows_real or
// with valid == 0 (valid may be NULL) quantise as zeros.
cudaError_t launch_mx_quant_rows(const void* W, uint8_t* Wq, uint8_t* Ws, long long rows,
                                 long long rows_real, int K, int rows_per_group,
                                 const uint8_t* valid, cudaStream_t s);
struct MxGemmCall {
  int gate_up;                 // 1: h = silu(a) * b quantised; 0: out = h W_down^T (fp32)
  int dh;                      // 1 (gate_up 0): dH = d_out W_down with the SwiGLU chain rule:
                               // A = d_out codes [rows][d], B = W_down^T codes [E][H][d]
  const int32_t* row_offsets;  // [E+1] padded, device; NULL: dense rows
  int dense_rows;              // dense: rows (the tile grid pads them to 128)
  int E;
  int rows;                    // routed: R_cap; dense: rows of A's buffer (padded)
  int d, H;                    // d a multiple of 256, H of 128
  const uint8_t* A;            // x codes [rows][d] or h codes [rows][H]
  const uint8_t* sfa;          // their scale atoms
  const uint8_t* B;            // W_gu codes [E][2H][d] or W_down codes [E][d][H]
  const uint8_t* sfb;          // their scale atoms
  uint8_t* hq;                 // gate/up out: h codes [rows][H]
  uint8_t* hs;                 // gate/up out: h scale atoms
  void* hb;                    // gate/up out (training): h [rows][H] bf16, or NULL
  void* abo;                   // gate/up out (training): a | b [rows][2H] fp16, or NULL
  void* out;                   // down out: [rows][d] (d is the output width), fp32 or,
  int out_bf16;                //   with out_bf16, bf16 (the per-slot out_perm, dx_perm)
  const void* abi;             // dH in: saved a | b [rows][2H] fp16
  void* dgu;                   // dH out: da | db [rows][2H] bf16
  uint8_t* dgq;                // dH out: codes of d_gu [rows][2H]
  uint8_t* dgs;                // dH out: their scale atoms [rows/128][2H/128]
  int* status;
};
// W [groups][R][C] bf16 -> codes of each group's transpose [groups][C][R],
// blocks of 32 along R, and scale atoms [groups][C/128][R/128] (a weight
// quantised along the axis a data-gradient product sums over).
cudaError_t launch_mx_quant_cols(const void* W, uint8_t* Wq, uint8_t* Ws, int groups, int R, int C,
                                 cudaStream_t s);
cudaError_t launch_mx_gemm(const MxGemmCall& g, cudaStream_t s);
cudaError_t launch_wait_timeout_selftest(int* status, unsigned long long limit_ns,
                                         cudaStream_t s);

}  // namespace moe
