// C-ABI entry points of the MoE layer: argument checks, the workspace
// layout, and the launch order of the kernels on the caller's stream.
#include <cstring>
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr size_t kAlign = 256;
// Route blocks: three per SM of a 152-SM GB300 (for the fused small-E
// router, as many as its registers let reside).  moe_route_static runs the
// same grid (its scratch holds the per-block slots of 456 blocks).
constexpr int kRouteBlocksCap = 456;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t row_capacity(const moe_config& c) {
  const int64_t a = (int64_t)c.T * c.k + (int64_t)(kRowAlign - 1) * c.E;
  return a / kRowAlign * kRowAlign;
}

int hs_total(const moe_config& c) { return c.n_shared > 0 ? c.n_shared * c.H_shared : 0; }

}  // namespace

int device_info(DeviceInfo* out) {
  static DeviceInfo cache[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& di = cache[dev];
  if (di.device != dev) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MOE_ERR_CUDA;
    di.num_sms = prop.multiProcessorCount;
    di.cc_major = prop.major;
    di.cc_minor = prop.minor;
    di.max_smem_optin = prop.sharedMemPerBlockOptin;
    di.device = dev;
  }
  *out = di;
  return MOE_OK;
}

int ws_layout(const moe_config* c, int training, WsLayout* w) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  const int G = route_group_lanes(c->E);
  const int groups = 256 / G;
  long long rb = ((long long)c->T + groups - 1) / groups;
  if (rb > kRouteBlocksCap) rb = kRouteBlocksCap;
  if (rb < 1) rb = 1;
  w->route_blocks = (int)rb;
  w->perm_blocks = (c->T + kPermChunk - 1) / kPermChunk;
  w->R_cap = row_capacity(*c);
  const int Hs = hs_total(*c);
  w->status = take(sizeof(int));
  w->route_done = take(kRouteAccBytes);
  w->route_treal = take((size_t)w->route_blocks * sizeof(int));
  w->route_zent = take((size_t)w->route_blocks * 2 * sizeof(float));
  w->perm_hist = take((size_t)w->perm_blocks * c->E * sizeof(int));
  w->perm_base = take((size_t)w->perm_blocks * c->E * sizeof(int));
  w->d_out = w->d_gu = w->dx_perm = w->ds_gu = w->dxr = w->dwr_part = 0;
  w->wr2 = w->dl3 = w->dl2 = w->goff = 0;
  w->dwr_splits = 1;
  const bool tc_router = router_tc_path(*c);
  if (training) {
    const size_t R = (size_t)w->R_cap;
    w->d_out = take(R * c->d * 2);
    w->d_gu = take(R * 2 * (size_t)c->H * 2);
    w->dx_perm = take(R * c->d * 2);
    if (Hs > 0) {
      w->ds_gu = take((size_t)c->T * 2 * Hs * 2);
    }
    if (!router_small_path(*c)) w->dxr = take((size_t)c->T * c->d * 4);
    int splits = c->T / 1024;
    if (splits < 1) splits = 1;
    if (splits > 64) splits = 64;
    if (router_small_path(*c)) splits = router_dw_small_parts(*c);
    if (tc_router) {
      int Tp, G, chunk;
      router_tc_sizes(*c, &Tp, &G, &chunk);
      splits = G;
      w->wr2 = take((size_t)c->d * 3 * c->E * 2);
      w->dl3 = take((size_t)c->T * 3 * c->E * 2);
      w->dl2 = take((size_t)2 * Tp * c->E * 2);
      w->goff = take((size_t)(G + 1) * sizeof(int));
    }
    w->dwr_splits = splits;
    w->dwr_part = take((size_t)splits * c->d * c->E * 4);
  }
  w->total = off;
  return MOE_OK;
}

namespace {

int check_cfg(const moe_config* c) {
  if (!c) return MOE_ERR_NULL;
  if (c->T < 1 || c->d < 64 || c->d % 64 || c->H < 64 || c->H % 64) return MOE_ERR_SHAPE;
  if (c->E < 1 || c->E > 256 || c->k < 1 || c->k > c->E || c->k > kMaxK) return MOE_ERR_SHAPE;
  if (c->n_shared < 0) return MOE_ERR_SHAPE;
  if (!(c->aux_coef == c->aux_coef) || !(c->z_coef == c->z_coef)) return MOE_ERR_SHAPE;
  if (c->n_shared > 0 && (c->H_shared < 64 || c->H_shared % 64)) return MOE_ERR_SHAPE;
  if ((int64_t)c->T * c->k >= (1ll << 31)) return MOE_ERR_SHAPE;
  if (row_capacity(*c) >= (1ll << 31)) return MOE_ERR_SHAPE;
  if ((int64_t)c->n_shared * c->H_shared >= (1ll << 30)) return MOE_ERR_SHAPE;
  if ((int64_t)c->E * 2 * c->H * c->d >= (1ll << 40)) return MOE_ERR_SHAPE;
  return MOE_OK;
}

int check_device() {
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return MOE_ERR_CUDA;
  if (di.cc_major != 10) return MOE_ERR_DEVICE;
  return MOE_OK;
}

struct Call {
  WsLayout w;
  char* ws;
  int* status;
  cudaStream_t s;
};

// Common prologue: config, device and workspace checks.
int begin(const moe_config* c, int training, void* ws, size_t ws_bytes, void* stream,
          Call* call) {
  int rc = check_cfg(c);
  if (rc) return rc;
  rc = check_device();
  if (rc) return rc;
  ws_layout(c, training, &call->w);
  if (!ws || ws_bytes < call->w.total) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_ALIGN;
  call->ws = static_cast<char*>(ws);
  call->status = reinterpret_cast<int*>(call->ws + call->w.status);
  call->s = static_cast<cudaStream_t>(stream);
  return MOE_OK;
}

#define MOE_NEED(p)                    \
  do {                                 \
    if (!(p)) return MOE_ERR_NULL;     \
    if (!aligned16(p)) return MOE_ERR_ALIGN; \
  } while (0)
#define MOE_OPT(p)                     \
  do {                                 \
    if ((p) && !aligned16(p)) return MOE_ERR_ALIGN; \
  } while (0)
#define MOE_CUDA(expr)                 \
  do {                                 \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

int do_router_logits(const moe_config* c, const moe_tensors* t, Call& k) {
  MOE_NEED(t->x); MOE_NEED(t->Wr); MOE_NEED(t->logits);
  MOE_CUDA(launch_router_logits(*c, t->x, t->Wr, t->logits, k.s));
  return MOE_OK;
}

int do_route(const moe_config* c, const moe_tensors* t, Call& k) {
  MOE_NEED(t->logits); MOE_OPT(t->bias); MOE_OPT(t->valid);
  MOE_NEED(t->topk_idx); MOE_NEED(t->gates); MOE_NEED(t->counts);
  MOE_NEED(t->f); MOE_NEED(t->p); MOE_NEED(t->aux); MOE_OPT(t->router_stats);
  MOE_CUDA(launch_route(*c, t->logits, t->bias, t->valid, t->topk_idx, t->gates, t->counts,
                        t->f, t->p, t->aux, t->router_stats, k.ws, k.w, k.s));
  return MOE_OK;
}

int do_router_route(const moe_config* c, const moe_tensors* t, Call& k) {
  if (!router_small_path(*c)) {
    int rc = do_router_logits(c, t, k);
    return rc ? rc : do_route(c, t, k);
  }
  MOE_NEED(t->x); MOE_NEED(t->Wr); MOE_NEED(t->logits);
  MOE_OPT(t->bias); MOE_OPT(t->valid);
  MOE_NEED(t->topk_idx); MOE_NEED(t->gates); MOE_NEED(t->counts);
  MOE_NEED(t->f); MOE_NEED(t->p); MOE_NEED(t->aux); MOE_OPT(t->router_stats);
  MOE_CUDA(launch_router_route(*c, t->x, t->Wr, t->bias, t->valid, t->logits, t->topk_idx,
                               t->gates, t->counts, t->f, t->p, t->aux, t->router_stats, k.ws,
                               k.w, k.s));
  return MOE_OK;
}

// x_perm may be NULL: then only offsets, perm and inv are produced, and the
// gate/up GEMM gathers its rows from x.
int do_permute(const moe_config* c, const moe_tensors* t, Call& k) {
  MOE_NEED(t->x); MOE_NEED(t->topk_idx); MOE_NEED(t->counts); MOE_NEED(t->offsets);
  MOE_NEED(t->row_offsets); MOE_NEED(t->perm); MOE_NEED(t->inv); MOE_OPT(t->x_perm);
  MOE_CUDA(launch_permute(*c, t->x, t->topk_idx, t->counts, t->offsets, t->row_offsets,
                          t->perm, t->inv, t->x_perm, k.ws, k.w, k.s));
  return MOE_OK;
}

int do_gate_up(const moe_config* c, const moe_tensors* t, Call& k) {
  MOE_OPT(t->x_perm); MOE_NEED(t->row_offsets); MOE_NEED(t->W_gu); MOE_NEED(t->h);
  MOE_OPT(t->ab);
  GemmCall g{};
  g.kind = GK_GATE_UP;
  g.row_offsets = t->row_offsets;
  g.E = c->E;
  g.rows = (int)k.w.R_cap;
  if (t->x_perm) {
    g.A = t->x_perm;
  } else {
    // the permute folded into the A load: rows gathered from x through perm
    MOE_NEED(t->x); MOE_NEED(t->perm);
    g.A = t->x;
    g.gperm = t->perm;
    g.gk = c->k;
    g.gT = c->T;
    g.grows = (int)k.w.R_cap;
  }
  g.lda = c->d;
  g.B = t->W_gu;
  g.K = c->d;
  g.N = c->H;
  g.H = c->H;
  g.out0 = t->h;
  g.ld0 = c->H;
  g.out1 = t->ab;
  g.ld1 = 2 * c->H;
  g.status = k.status;
  MOE_CUDA(launch_gemm(g, k.s));
  return MOE_OK;
}

int do_down(const moe_config* c, const moe_tensors* t, Call& k) {
  MOE_NEED(t->h); MOE_NEED(t->row_offsets); MOE_NEED(t->W_down); MOE_NEED(t->out_perm);
  GemmCall g{};
  g.kind = GK_DOWN;
  g.row_offsets = t->row_offsets;
  g.E = c->E;
  g.rows = (int)k.w.R_cap;
  g.A = t->h;
  g.lda = c->H;
  g.B = t->W_down;
  g.K = c->H;
  g.N = c->d;
  g.out0 = t->out_perm;                        // bf16: each slot's output row
  g.ld0 = c->d;
  g.out_f32 = 0;
  g.status = k.status;
  MOE_CUDA(launch_gemm(g, k.s));
  return MOE_OK;
}

int do_combine(const moe_config* c, const moe_tensors* t, Call& k);

// The shared expert; with `fold_combine` its down GEMM also performs the
// combine (out_perm, inv, gates -> y) in its epilogue instead of writing s_out.
int shared_ffn(const moe_config* c, const moe_tensors* t, Call& k, bool fold_combine) {
  const int Hs = hs_total(*c);
  if (Hs == 0) return MOE_OK;
  MOE_NEED(t->x); MOE_OPT(t->valid); MOE_NEED(t->Ws_gu); MOE_NEED(t->Ws_down);
  MOE_NEED(t->s_h); MOE_OPT(t->s_ab);
  if (fold_combine) {
    MOE_NEED(t->out_perm); MOE_NEED(t->inv); MOE_NEED(t->gates); MOE_NEED(t->y);
  } else {
    MOE_NEED(t->s_out);
  }
  GemmCall g{};
  g.kind = GK_GATE_UP;
  g.row_offsets = nullptr;
  g.E = 1;
  g.rows = c->T;
  g.A = t->x;
  g.lda = c->d;
  g.B = t->Ws_gu;
  g.K = c->d;
  g.N = Hs;
  g.H = Hs;
  g.out0 = t->s_h;
  g.ld0 = Hs;
  g.out1 = t->s_ab;
  g.ld1 = 2 * Hs;
  g.valid = t->valid;
  g.status = k.status;
  MOE_CUDA(launch_gemm(g, k.s));
  GemmCall d{};
  d.kind = GK_DOWN;
  d.row_offsets = nullptr;
  d.E = 1;
  d.rows = c->T;
  d.A = t->s_h;
  d.lda = Hs;
  d.B = t->Ws_down;
  d.K = Hs;
  d.N = c->d;
  d.ld0 = c->d;
  d.status = k.status;
  if (fold_combine) {
    d.out0 = t->y;
    d.out_f32 = 0;
    d.valid = t->valid;
    d.comb_src = t->out_perm;
    d.comb_inv = t->inv;
    d.comb_rows = (int)k.w.R_cap;
    d.comb_gates = t->gates;
    d.comb_k = c->k;
  } else {
    d.out0 = t->s_out;
    d.out_f32 = 1;
  }
  MOE_CUDA(launch_gemm(d, k.s));
  return MOE_OK;
}

int do_shared(const moe_config* c, const moe_tensors* t, Call& k) {
  return shared_ffn(c, t, k, false);
}

// a5 + a6: with a shared expert, the combine runs in its down GEMM's
// epilogue; without one, the combine kernel.
int do_shared_combine(const moe_config* c, const moe_tensors* t, Call& k) {
  if (hs_total(*c) == 0) return do_combine(c, t, k);
  return shared_ffn(c, t, k, true);
}

int do_combine(const moe_config* c, const moe_tensors* t, Call& k) {
  MOE_NEED(t->out_perm); MOE_NEED(t->inv); MOE_NEED(t->gates); MOE_OPT(t->valid);
  MOE_NEED(t->y);
  const float* s_out = nullptr;
  if (hs_total(*c) > 0) {
    MOE_NEED(t->s_out);
    s_out = t->s_out;
  }
  MOE_CUDA(launch_combine(*c, t->out_perm, t->inv, t->gates, t->valid, s_out, t->y,
                          (long long)k.w.R_cap, k.status, k.s));
  return MOE_OK;
}

bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }
#define MOE_NEED32(p)                          \
  do {                                         \
    if (!(p)) return MOE_ERR_NULL;             \
    if (!aligned32(p)) return MOE_ERR_ALIGN;   \
  } while (0)

// The backward; with `m` (the MXFP8 training step) the routed experts' two
// data-gradient products run on MXFP8 operands: d_out quantised along d,
// dH = Q(d_out) Q(W_down^T) with the SwiGLU chain rule in its epilogue (which
// also quantises d_gu along 2H), then dx_perm = Q(d_gu) Q(W_gu^T).
int do_backward(const moe_config* c, const moe_tensors* t, const moe_grads* g, Call& k,
                const moe_mx_tensors* m = nullptr) {
  if (!g) return MOE_ERR_NULL;
  const int Hs = hs_total(*c);
  MOE_NEED(g->dY); MOE_NEED(g->dx); MOE_NEED(g->dWr); MOE_NEED(g->dW_gu);
  MOE_NEED(g->dW_down); MOE_NEED(g->d_logits);
  MOE_NEED(t->x); MOE_NEED(t->Wr); MOE_OPT(t->valid); MOE_NEED(t->W_gu); MOE_NEED(t->W_down);
  MOE_NEED(t->logits); MOE_NEED(t->topk_idx); MOE_NEED(t->gates); MOE_NEED(t->counts);
  MOE_NEED(t->f); MOE_NEED(t->row_offsets); MOE_NEED(t->inv); MOE_NEED(t->x_perm);
  MOE_NEED(t->h); MOE_NEED(t->out_perm);
  if (!m) MOE_NEED(t->ab);                      // the MX step keeps a | b in mx->ab16
  if (Hs > 0) {
    MOE_NEED(t->Ws_gu); MOE_NEED(t->Ws_down); MOE_NEED(t->s_ab); MOE_NEED(t->s_h);
    MOE_NEED(g->dWs_gu); MOE_NEED(g->dWs_down);
  }
  const WsLayout& w = k.w;
  void* d_out = k.ws + w.d_out;
  void* d_gu = k.ws + w.d_gu;
  void* dx_perm = k.ws + w.dx_perm;           // bf16 [R][d]
  const int R = (int)w.R_cap;

  if (m) {
    MOE_NEED32(m->W_gu_tq); MOE_NEED(m->W_gu_ts); MOE_NEED32(m->W_down_tq);
    MOE_NEED(m->W_down_ts); MOE_NEED32(m->dout_q); MOE_NEED(m->dout_s);
    MOE_NEED32(m->dgu_q); MOE_NEED(m->dgu_s); MOE_NEED(m->ab16);
  }
  // (i) + (vii): d_out (with the MX step, also its codes along d, quantised
  // from the fp32 g dY), dg and the router-logit gradient
  MOE_CUDA(launch_combine_bwd(*c, g->dY, t->out_perm, t->inv, t->topk_idx, t->gates, t->logits,
                              t->f, t->counts, t->valid, t->row_offsets, d_out,
                              m ? m->dout_q : nullptr, m ? m->dout_s : nullptr, g->d_logits,
                              (long long)R, k.status, k.s));
  if (m) {
    // (ii) dH = Q(d_out) Q(W_down^T) -> SwiGLU backward -> d_gu = [da | db]
    // in bf16 and, from the fp32 values, its codes along 2H
    MxGemmCall h{};
    h.dh = 1; h.row_offsets = t->row_offsets; h.E = c->E; h.rows = R; h.d = c->d; h.H = c->H;
    h.A = m->dout_q; h.sfa = m->dout_s; h.B = m->W_down_tq; h.sfb = m->W_down_ts;
    h.abi = m->ab16; h.dgu = d_gu; h.dgq = m->dgu_q; h.dgs = m->dgu_s; h.status = k.status;
    MOE_CUDA(launch_mx_gemm(h, k.s));
    // (iii) dx_perm = Q(d_gu) Q(W_gu^T): the down kind with K = 2H, N = d
    MxGemmCall x{};
    x.row_offsets = t->row_offsets; x.E = c->E; x.rows = R; x.d = c->d; x.H = 2 * c->H;
    x.A = m->dgu_q; x.sfa = m->dgu_s; x.B = m->W_gu_tq; x.sfb = m->W_gu_ts; x.out = dx_perm;
    x.out_bf16 = 1;
    x.status = k.status;
    MOE_CUDA(launch_mx_gemm(x, k.s));
  } else {
    // (ii) dH = d_out W_down[e], SwiGLU backward -> d_gu = [da | db]
    GemmCall gh{};
    gh.kind = GK_DH; gh.row_offsets = t->row_offsets; gh.E = c->E; gh.rows = R;
    gh.A = d_out; gh.lda = c->d; gh.B = t->W_down; gh.K = c->d; gh.N = c->H; gh.H = c->H;
    gh.out0 = d_gu; gh.ld0 = 2 * c->H; gh.aux_in = t->ab; gh.ld_aux = 2 * c->H;
    gh.status = k.status;
    MOE_CUDA(launch_gemm(gh, k.s));
    // (iii) dx_perm = d_gu W_gu[e]
    GemmCall gx{};
    gx.kind = GK_DX; gx.row_offsets = t->row_offsets; gx.E = c->E; gx.rows = R;
    gx.A = d_gu; gx.lda = 2 * c->H; gx.B = t->W_gu; gx.K = 2 * c->H; gx.N = c->d;
    gx.out0 = dx_perm; gx.ld0 = c->d; gx.out_f32 = 0; gx.status = k.status;
    MOE_CUDA(launch_gemm(gx, k.s));
  }
  // (iv) dW_down[e] = d_out_e^T h_e ; dW_gu[e] = d_gu_e^T x_perm_e
  GemmCall wd{};
  wd.kind = GK_DW; wd.row_offsets = t->row_offsets; wd.E = c->E; wd.rows = R;
  wd.A = d_out; wd.lda = c->d; wd.Mdw = c->d; wd.B = t->h; wd.N = c->H;
  wd.out0 = g->dW_down; wd.ld0 = c->H; wd.status = k.status;
  MOE_CUDA(launch_gemm(wd, k.s));
  GemmCall wg{};
  wg.kind = GK_DW; wg.row_offsets = t->row_offsets; wg.E = c->E; wg.rows = R;
  wg.A = d_gu; wg.lda = 2 * c->H; wg.Mdw = 2 * c->H; wg.B = t->x_perm; wg.N = c->d;
  wg.out0 = g->dW_gu; wg.ld0 = c->d; wg.status = k.status;
  MOE_CUDA(launch_gemm(wg, k.s));
  // router input gradient: on the tensor cores (E a multiple of 32), the
  // CUDA cores (other large E), or inline in the dx sum (small E)
  float* dxr = nullptr;
  float* part = reinterpret_cast<float*>(k.ws + w.dwr_part);
  if (router_tc_path(*c)) {
    dxr = reinterpret_cast<float*>(k.ws + w.dxr);
    MOE_CUDA(launch_router_bwd_tc(*c, t->x, g->d_logits, t->Wr, dxr, g->dWr, k.ws + w.wr2,
                                  k.ws + w.dl3, k.ws + w.dl2,
                                  reinterpret_cast<int*>(k.ws + w.goff), part, k.status, k.s));
  } else if (!router_small_path(*c)) {
    dxr = reinterpret_cast<float*>(k.ws + w.dxr);
    MOE_CUDA(launch_router_dx(*c, g->d_logits, t->Wr, dxr, k.s));
  }
  // (v) shared expert; (vi) the un-permute sum of dx runs in the epilogue of
  // its dx GEMM (or, without a shared expert, in the gather kernel)
  if (Hs > 0) {
    void* ds_gu = k.ws + w.ds_gu;
    GemmCall sh{};
    sh.kind = GK_DH; sh.row_offsets = nullptr; sh.E = 1; sh.rows = c->T;
    sh.A = g->dY; sh.lda = c->d; sh.B = t->Ws_down; sh.K = c->d; sh.N = Hs; sh.H = Hs;
    sh.out0 = ds_gu; sh.ld0 = 2 * Hs; sh.aux_in = t->s_ab; sh.ld_aux = 2 * Hs;
    sh.status = k.status;
    MOE_CUDA(launch_gemm(sh, k.s));
    GemmCall sx{};
    sx.kind = GK_DX; sx.row_offsets = nullptr; sx.E = 1; sx.rows = c->T;
    sx.A = ds_gu; sx.lda = 2 * Hs; sx.B = t->Ws_gu; sx.K = 2 * Hs; sx.N = c->d;
    sx.out0 = g->dx; sx.ld0 = c->d; sx.out_f32 = 0; sx.status = k.status;
    sx.valid = t->valid;
    sx.comb_src = dx_perm; sx.comb_inv = t->inv; sx.comb_k = c->k; sx.comb_rows = R;
    sx.dl = g->d_logits; sx.wr = t->Wr; sx.rE = router_small_path(*c) ? c->E : 0;
    sx.dxr = dxr;
    MOE_CUDA(launch_gemm(sx, k.s));
    GemmCall sw{};
    sw.kind = GK_DW; sw.row_offsets = nullptr; sw.E = 1; sw.rows = c->T;
    sw.A = g->dY; sw.lda = c->d; sw.Mdw = c->d; sw.B = t->s_h; sw.N = Hs;
    sw.out0 = g->dWs_down; sw.ld0 = Hs; sw.status = k.status;
    MOE_CUDA(launch_gemm(sw, k.s));
    GemmCall sg{};
    sg.kind = GK_DW; sg.row_offsets = nullptr; sg.E = 1; sg.rows = c->T;
    sg.A = ds_gu; sg.lda = 2 * Hs; sg.Mdw = 2 * Hs; sg.B = t->x; sg.N = c->d;
    sg.out0 = g->dWs_gu; sg.ld0 = c->d; sg.status = k.status;
    MOE_CUDA(launch_gemm(sg, k.s));
  } else {
    MOE_CUDA(launch_dx_gather(*c, dx_perm, t->inv, dxr, g->d_logits, t->Wr, t->valid, g->dx,
                              (long long)R, k.status, k.s));
  }
  if (!router_tc_path(*c))
    MOE_CUDA(launch_router_dw(*c, t->x, g->d_logits, g->dWr, part, w.dwr_splits, k.s));
  return MOE_OK;
}

// ---- MXFP8 routed experts
// The MX kernels store 32 bytes per lane: their code buffers and out_perm
// must be 32-byte aligned (MOE_NEED32).

int check_mx(const moe_config* c) {
  if (c->d % 256 || c->H % 128 || hs_total(*c) % 128) return MOE_ERR_SHAPE;
  return MOE_OK;
}

void mx_sizes(const moe_config& c, size_t* b) {
  const size_t E = c.E, d = c.d, H = c.H, R = (size_t)row_capacity(c);
  b[0] = E * 2 * H * d;                                  // W_gu_q
  b[1] = E * (2 * H / 128) * (d / 128) * 512;            // W_gu_s
  b[2] = E * d * H;                                      // W_down_q
  b[3] = E * (d / 128) * (H / 128) * 512;                // W_down_s
  b[4] = R * d;                                          // x_q
  b[5] = (R / 128) * (d / 128) * 512;                    // x_s
  b[6] = R * H;                                          // h_q
  b[7] = (R / 128) * (H / 128) * 512;                    // h_s
  const size_t Hs = (size_t)hs_total(c), Tp = ((size_t)c.T + 127) / 128 * 128;
  b[8] = 2 * Hs * d;                                     // Ws_gu_q
  b[9] = (2 * Hs / 128) * (d / 128) * 512;               // Ws_gu_s
  b[10] = d * Hs;                                        // Ws_down_q
  b[11] = (d / 128) * (Hs / 128) * 512;                  // Ws_down_s
  b[12] = Hs ? Tp * d : 0;                               // xt_q
  b[13] = Hs ? (Tp / 128) * (d / 128) * 512 : 0;         // xt_s
  b[14] = Tp * Hs;                                       // hs_q
  b[15] = (Tp / 128) * (Hs / 128) * 512;                 // hs_s
  // the training step's data gradients
  b[16] = E * d * 2 * H;                                 // W_gu_tq: [E][d][2H]
  b[17] = E * (d / 128) * (2 * H / 128) * 512;           // W_gu_ts
  b[18] = E * H * d;                                     // W_down_tq: [E][H][d]
  b[19] = E * (H / 128) * (d / 128) * 512;               // W_down_ts
  b[20] = R * d;                                         // dout_q
  b[21] = (R / 128) * (d / 128) * 512;                   // dout_s
  b[22] = R * 2 * H;                                     // dgu_q
  b[23] = (R / 128) * (2 * H / 128) * 512;               // dgu_s
  b[24] = R * 2 * H * 2;                                 // ab16: [R][2H] fp16
}

// The shared expert on MXFP8 operands: x quantised in token order (PAD and
// the padding to 128 rows as zeros), then the two block-scaled GEMMs over
// the dense token rows; s_out = 0 on PAD rows because their codes are 0.
// quantise_x: x's token-order codes are made here (moe_mx_shared_ffn), or
// were written by the permute (moe_mx_forward).
int do_mx_shared(const moe_config* c, const moe_tensors* t, const moe_mx_tensors* m, Call& k,
                 bool quantise_x) {
  const int Hs = hs_total(*c);
  if (Hs == 0) return MOE_OK;
  MOE_NEED(t->x); MOE_OPT(t->valid); MOE_NEED32(t->s_out);
  MOE_NEED32(m->Ws_gu_q); MOE_NEED(m->Ws_gu_s); MOE_NEED32(m->Ws_down_q); MOE_NEED(m->Ws_down_s);
  MOE_NEED32(m->xt_q); MOE_NEED(m->xt_s); MOE_NEED32(m->hs_q); MOE_NEED(m->hs_s);
  const int Tp = (c->T + 127) / 128 * 128;
  if (quantise_x)
    MOE_CUDA(launch_mx_quant_rows(t->x, m->xt_q, m->xt_s, Tp, c->T, c->d, Tp, t->valid, k.s));
  MxGemmCall g{};
  g.row_offsets = nullptr;
  g.dense_rows = c->T;
  g.E = 1;
  g.rows = Tp;
  g.d = c->d;
  g.H = Hs;
  g.status = k.status;
  g.gate_up = 1;
  g.A = m->xt_q; g.sfa = m->xt_s; g.B = m->Ws_gu_q; g.sfb = m->Ws_gu_s;
  g.hq = m->hs_q; g.hs = m->hs_s;
  MOE_CUDA(launch_mx_gemm(g, k.s));
  g.gate_up = 0;
  g.A = m->hs_q; g.sfa = m->hs_s; g.B = m->Ws_down_q; g.sfb = m->Ws_down_s;
  g.hq = nullptr; g.hs = nullptr;
  g.out = t->s_out;
  MOE_CUDA(launch_mx_gemm(g, k.s));
  return MOE_OK;
}

// with_xt: also write x's codes in token order for the shared expert
// (moe_mx_forward with a shared expert), so x is read and quantised once.
int do_mx_permute(const moe_config* c, const moe_tensors* t, const moe_mx_tensors* m, Call& k,
                  bool with_xt, bool with_rows = false) {
  MOE_NEED(t->x); MOE_NEED(t->topk_idx); MOE_NEED(t->counts); MOE_NEED(t->offsets);
  MOE_NEED(t->row_offsets); MOE_NEED(t->perm); MOE_NEED(t->inv);
  MOE_NEED32(m->x_q); MOE_NEED(m->x_s);
  if (with_xt) {
    MOE_NEED32(m->xt_q); MOE_NEED(m->xt_s);
  }
  MOE_CUDA(launch_permute_mx(*c, t->x, t->topk_idx, t->counts, t->offsets, t->row_offsets,
                             t->perm, t->inv, m->x_q, m->x_s, with_xt ? m->xt_q : nullptr,
                             with_xt ? m->xt_s : nullptr, with_rows ? t->x_perm : nullptr, k.ws,
                             k.w, k.s));
  return MOE_OK;
}

int do_mx_gemm(const moe_config* c, const moe_tensors* t, const moe_mx_tensors* m, Call& k,
               bool gate_up, bool save = false) {
  MOE_NEED(t->row_offsets);
  MxGemmCall g{};
  g.gate_up = gate_up ? 1 : 0;
  g.row_offsets = t->row_offsets;
  g.E = c->E;
  g.rows = (int)k.w.R_cap;
  g.d = c->d;
  g.H = c->H;
  g.status = k.status;
  if (gate_up) {
    MOE_NEED(m->x_q); MOE_NEED(m->x_s); MOE_NEED(m->W_gu_q); MOE_NEED(m->W_gu_s);
    MOE_NEED32(m->h_q); MOE_NEED(m->h_s);
    g.A = m->x_q; g.sfa = m->x_s; g.B = m->W_gu_q; g.sfb = m->W_gu_s;
    g.hq = m->h_q; g.hs = m->h_s;
    if (save) {                          // training: h in bf16, a | b in fp16
      MOE_NEED(t->h); MOE_NEED32(m->ab16);
      g.hb = t->h;
      g.abo = m->ab16;
    }
  } else {
    MOE_NEED(m->h_q); MOE_NEED(m->h_s); MOE_NEED(m->W_down_q); MOE_NEED(m->W_down_s);
    MOE_NEED32(t->out_perm);
    g.A = m->h_q; g.sfa = m->h_s; g.B = m->W_down_q; g.sfb = m->W_down_s;
    g.out = t->out_perm;
    g.out_bf16 = 1;
  }
  MOE_CUDA(launch_mx_gemm(g, k.s));
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

int moe_debug_bounds(void) { return moe::kDebugBounds ? 1 : 0; }

const char* moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "a required pointer is NULL";
    case MOE_ERR_SHAPE: return "configuration violates the shape rules";
    case MOE_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
    case MOE_ERR_DEVICE: return "current device is not an sm_100-family GPU";
    case MOE_ERR_TIMEOUT: return "a bounded wait inside a kernel expired";
    case MOE_ERR_INDEX: return "expert index out of range";
    case MOE_ERR_NONFINITE: return "non-finite router logit";
    case MOE_ERR_BOUNDS: return "row index outside the buffer (debug bounds check)";
    default: return "unknown status code";
  }
}

int moe_check_config(const moe_config* cfg) { return check_cfg(cfg); }

int moe_row_capacity(const moe_config* cfg, int64_t* rows) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!rows) return MOE_ERR_NULL;
  *rows = row_capacity(*cfg);
  return MOE_OK;
}

int moe_workspace_bytes(const moe_config* cfg, int training, size_t* bytes) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!bytes) return MOE_ERR_NULL;
  WsLayout w;
  ws_layout(cfg, training, &w);
  *bytes = w.total;
  return MOE_OK;
}

int moe_workspace_offsets(const moe_config* cfg, size_t* out) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!out) return MOE_ERR_NULL;
  WsLayout w;
  ws_layout(cfg, 1, &w);
  out[0] = w.d_out;
  out[1] = w.d_gu;
  out[2] = w.dx_perm;
  out[3] = hs_total(*cfg) > 0 ? w.ds_gu : 0;
  return MOE_OK;
}

int moe_get_status(void* workspace, void* stream, int* status) {
  if (!workspace || !status) return MOE_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  int* dev = static_cast<int*>(workspace);  // the status word sits at offset 0
  if (cudaMemcpyAsync(&v, dev, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(dev, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  *status = v;
  return MOE_OK;
}

int moe_selftest_wait_timeout(void* workspace, uint64_t limit_ns, void* stream) {
  if (!workspace) return MOE_ERR_NULL;
  if (limit_ns == 0 || limit_ns > 10000000000ull) return MOE_ERR_SHAPE;
  int rc = check_device();
  if (rc) return rc;
  MOE_CUDA(launch_wait_timeout_selftest(static_cast<int*>(workspace), limit_ns,
                                        static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

#define MOE_ENTRY(name, training, body)                                                      \
  int name(const moe_config* cfg, const moe_tensors* t, void* workspace,                     \
           size_t workspace_bytes, void* stream) {                                           \
    Call k;                                                                                  \
    int rc = begin(cfg, training, workspace, workspace_bytes, stream, &k);                   \
    if (rc) return rc;                                                                       \
    if (!t) return MOE_ERR_NULL;                                                             \
    body                                                                                     \
  }

MOE_ENTRY(moe_router_logits, 0, { return do_router_logits(cfg, t, k); })
MOE_ENTRY(moe_route, 0, { return do_route(cfg, t, k); })
MOE_ENTRY(moe_router_route, 0, { return do_router_route(cfg, t, k); })
MOE_ENTRY(moe_permute, 0, { return do_permute(cfg, t, k); })
MOE_ENTRY(moe_expert_gate_up, 0, { return do_gate_up(cfg, t, k); })
MOE_ENTRY(moe_expert_down, 0, { return do_down(cfg, t, k); })
MOE_ENTRY(moe_shared_ffn, 0, { return do_shared(cfg, t, k); })
MOE_ENTRY(moe_combine, 0, { return do_combine(cfg, t, k); })
MOE_ENTRY(moe_shared_ffn_combine, 0, { return do_shared_combine(cfg, t, k); })
MOE_ENTRY(moe_expert_ffn, 0, {
  if ((rc = do_gate_up(cfg, t, k))) return rc;
  if ((rc = do_down(cfg, t, k))) return rc;
  return do_shared(cfg, t, k);
})
MOE_ENTRY(moe_forward, 0, {
  if ((rc = do_router_route(cfg, t, k))) return rc;
  if ((rc = do_permute(cfg, t, k))) return rc;
  if ((rc = do_gate_up(cfg, t, k))) return rc;
  if ((rc = do_down(cfg, t, k))) return rc;
  return do_shared_combine(cfg, t, k);
})

int moe_mx_sizes(const moe_config* cfg, size_t* bytes) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_mx(cfg))) return rc;
  if (!bytes) return MOE_ERR_NULL;
  mx_sizes(*cfg, bytes);
  return MOE_OK;
}

int moe_mx_quantize_weights(const moe_config* cfg, const moe_tensors* t,
                            const moe_mx_tensors* mx, void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_mx(cfg))) return rc;
  if ((rc = check_device())) return rc;
  if (!t || !mx) return MOE_ERR_NULL;
  MOE_NEED(t->W_gu); MOE_NEED(t->W_down);
  MOE_NEED32(mx->W_gu_q); MOE_NEED(mx->W_gu_s); MOE_NEED32(mx->W_down_q);
  MOE_NEED(mx->W_down_s);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long E = cfg->E, d = cfg->d, H = cfg->H, Hs = hs_total(*cfg);
  MOE_CUDA(launch_mx_quant_rows(t->W_gu, mx->W_gu_q, mx->W_gu_s, E * 2 * H, E * 2 * H, (int)d,
                                (int)(2 * H), nullptr, s));
  MOE_CUDA(launch_mx_quant_rows(t->W_down, mx->W_down_q, mx->W_down_s, E * d, E * d, (int)H,
                                (int)d, nullptr, s));
  if (mx->W_gu_tq || mx->W_down_tq) {
    // the training step's weights along their other axis (data gradients)
    MOE_NEED32(mx->W_gu_tq); MOE_NEED(mx->W_gu_ts); MOE_NEED32(mx->W_down_tq);
    MOE_NEED(mx->W_down_ts);
    MOE_CUDA(launch_mx_quant_cols(t->W_gu, mx->W_gu_tq, mx->W_gu_ts, (int)E, (int)(2 * H),
                                  (int)d, s));
    MOE_CUDA(launch_mx_quant_cols(t->W_down, mx->W_down_tq, mx->W_down_ts, (int)E, (int)d,
                                  (int)H, s));
  }
  if (Hs > 0) {
    MOE_NEED(t->Ws_gu); MOE_NEED(t->Ws_down);
    MOE_NEED32(mx->Ws_gu_q); MOE_NEED(mx->Ws_gu_s); MOE_NEED32(mx->Ws_down_q);
    MOE_NEED(mx->Ws_down_s);
    MOE_CUDA(launch_mx_quant_rows(t->Ws_gu, mx->Ws_gu_q, mx->Ws_gu_s, 2 * Hs, 2 * Hs, (int)d,
                                  (int)(2 * Hs), nullptr, s));
    MOE_CUDA(launch_mx_quant_rows(t->Ws_down, mx->Ws_down_q, mx->Ws_down_s, d, d, (int)Hs,
                                  (int)d, nullptr, s));
  }
  return MOE_OK;
}

#define MOE_MX_ENTRY(name, body)                                                             \
  int name(const moe_config* cfg, const moe_tensors* t, const moe_mx_tensors* mx,            \
           void* workspace, size_t workspace_bytes, void* stream) {                          \
    Call k;                                                                                  \
    int rc = check_cfg(cfg);                                                                 \
    if (rc) return rc;                                                                       \
    if ((rc = check_mx(cfg))) return rc;                                                     \
    if ((rc = begin(cfg, 0, workspace, workspace_bytes, stream, &k))) return rc;             \
    if (!t || !mx) return MOE_ERR_NULL;                                                      \
    body                                                                                     \
  }

MOE_MX_ENTRY(moe_mx_permute, { return do_mx_permute(cfg, t, mx, k, false); })
MOE_MX_ENTRY(moe_mx_expert_gate_up, { return do_mx_gemm(cfg, t, mx, k, true); })
MOE_MX_ENTRY(moe_mx_expert_down, { return do_mx_gemm(cfg, t, mx, k, false); })
MOE_MX_ENTRY(moe_mx_shared_ffn, { return do_mx_shared(cfg, t, mx, k, true); })
MOE_MX_ENTRY(moe_mx_forward, {
  if ((rc = do_router_route(cfg, t, k))) return rc;
  const bool shared = hs_total(*cfg) > 0;
  if ((rc = do_mx_permute(cfg, t, mx, k, shared))) return rc;
  if ((rc = do_mx_gemm(cfg, t, mx, k, true))) return rc;
  if ((rc = do_mx_gemm(cfg, t, mx, k, false))) return rc;
  if ((rc = do_mx_shared(cfg, t, mx, k, false))) return rc;
  return do_combine(cfg, t, k);
})

MOE_MX_ENTRY(moe_mx_forward_train, {
  MOE_NEED(t->x_perm); MOE_NEED(t->h); MOE_NEED32(t->out_perm);
  if ((rc = do_router_route(cfg, t, k))) return rc;
  if ((rc = do_mx_permute(cfg, t, mx, k, false, true))) return rc;
  if ((rc = do_mx_gemm(cfg, t, mx, k, true, true))) return rc;
  if ((rc = do_mx_gemm(cfg, t, mx, k, false))) return rc;
  return do_shared_combine(cfg, t, k);   // the bf16 shared expert, combine in its down GEMM
})

int moe_mx_backward(const moe_config* cfg, const moe_tensors* t, const moe_mx_tensors* mx,
                    const moe_grads* g, void* workspace, size_t workspace_bytes, void* stream) {
  Call k;
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_mx(cfg))) return rc;
  if ((rc = begin(cfg, 1, workspace, workspace_bytes, stream, &k))) return rc;
  if (!t || !mx) return MOE_ERR_NULL;
  return do_backward(cfg, t, g, k, mx);
}

int moe_route_partials(const moe_config* cfg, const moe_tensors* t, double* sums, void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_device())) return rc;
  if (!t) return MOE_ERR_NULL;
  MOE_NEED(t->counts); MOE_NEED(t->p); MOE_NEED(sums);
  MOE_CUDA(launch_route_partials(*cfg, t->counts, t->p, sums, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_route_finalize(const moe_config* cfg, const moe_tensors* t, const double* sums,
                       void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_device())) return rc;
  if (!t) return MOE_ERR_NULL;
  MOE_NEED(sums); MOE_NEED(t->f); MOE_NEED(t->p); MOE_NEED(t->aux);
  MOE_CUDA(launch_route_finalize(*cfg, sums, t->f, t->p, t->aux,
                                 static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_backward(const moe_config* cfg, const moe_tensors* t, const moe_grads* g,
                 void* workspace, size_t workspace_bytes, void* stream) {
  Call k;
  int rc = begin(cfg, 1, workspace, workspace_bytes, stream, &k);
  if (rc) return rc;
  if (!t) return MOE_ERR_NULL;
  return do_backward(cfg, t, g, k);
}

}  // extern "C"
