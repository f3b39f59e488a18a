// The router's backward matrix products on the tensor cores, for expert
// counts where they are compute-bound on the CUDA cores (E a multiple of 32
// beyond the small path): the input-gradient term dL.W_r^T and
// dW_r = x^T.dL.
//
// dL and W_r are fp32.  Each is split into two bf16 pieces, a = a1 + a2
// (a1 = bf16(a), a2 = bf16(a - a1): 16 significant bits), whose products are
// exact in fp32; the products keep the three leading cross terms
// a1 b1 + a1 b2 + a2 b1 and accumulate in fp32 on the tensor cores.  x is
// bf16 already, so dW_r needs only the two pieces of dL.  (The logits
// themselves stay on the CUDA cores in IEEE fp32: routing decisions are
// taken on them, and tensor-core accumulation is measurably looser than fp32
// fused multiply-adds.)
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

__device__ __forceinline__ void split2(float w, bf16& p0, bf16& p1) {
  p0 = __float2bfloat16_rn(w);
  p1 = __float2bfloat16_rn(w - __bfloat162float(p0));
}

// W_r [d][E] -> wr2 [d][3E] (dx B operand, K-major): [c][e] = w1, [c][E+e] = w2,
// [c][2E+e] = w1, matching the A operand [a1 | a1 | a2].
__global__ void split_wr_kernel(const float* __restrict__ Wr, bf16* __restrict__ wr2, int d,
                                int E) {
  const int n = d * E;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int c = i / E, e = i - c * E;
    bf16 p0, p1;
    split2(Wr[i], p0, p1);
    bf16* r = wr2 + (size_t)c * 3 * E;
    r[e] = p0;
    r[E + e] = p1;
    r[2 * E + e] = p0;
  }
}

// dL [T][E] ->
//   dl3 [T][3E]     (dx A operand):   [t][e] = a1, [t][E+e] = a1, [t][2E+e] = a2
//   dl2 [2*Tp][E]   (dW_r B operand): rows [0,T) = a1, rows [Tp, Tp+T) = a2, other rows 0
// and the split-K row groups goff[g] = min(g*chunk, 2*Tp), g = 0..G.
__global__ void split_dl_kernel(const float* __restrict__ dL, bf16* __restrict__ dl3,
                                bf16* __restrict__ dl2, int T, int Tp, int E,
                                int* __restrict__ goff, int G, int chunk) {
  if (blockIdx.x == 0)
    for (int g = threadIdx.x; g <= G; g += blockDim.x) goff[g] = min(g * chunk, 2 * Tp);
  const long long n = (long long)Tp * E;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / E), e = (int)(i - (long long)t * E);
    bf16 a1 = __float2bfloat16_rn(0.f), a2 = a1;
    if (t < T) {
      split2(dL[i], a1, a2);
      bf16* r = dl3 + (size_t)t * 3 * E;
      r[e] = a1;
      r[E + e] = a1;
      r[2 * E + e] = a2;
    }
    dl2[(size_t)t * E + e] = a1;
    dl2[(size_t)(Tp + t) * E + e] = a2;
  }
}

}  // namespace

bool router_tc_path(const moe_config& c) {
  return !router_small_path(c) && c.E % 32 == 0;
}

void router_tc_sizes(const moe_config& c, int* Tp, int* G, int* chunk) {
  const int tp = (c.T + 127) / 128 * 128;
  const int tiles_per_group = ((c.d + 127) / 128) * ((c.E + 255) / 256);
  int g = 152 / tiles_per_group;
  if (g < 1) g = 1;
  if (g > 64) g = 64;
  int ch = ((2 * tp + g - 1) / g + 127) / 128 * 128;
  *Tp = tp;
  *chunk = ch;
  *G = (2 * tp + ch - 1) / ch;
}

// dxr[T][d] = dL . W_r^T  and  dW_r[d][E] = x^T . dL  (split-K over row groups,
// partials summed in group order).
cudaError_t launch_router_bwd_tc(const moe_config& c, const void* x, const float* dL,
                                 const float* Wr, float* dxr, float* dWr, void* wr2, void* dl3,
                                 void* dl2, int* goff, float* part, int* status,
                                 cudaStream_t s) {
  int Tp, G, chunk;
  router_tc_sizes(c, &Tp, &G, &chunk);
  const int n = c.d * c.E;
  split_wr_kernel<<<(n + 255) / 256, 256, 0, s>>>(Wr, static_cast<bf16*>(wr2), c.d, c.E);
  const long long m = (long long)Tp * c.E;
  int blocks = (int)((m + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  split_dl_kernel<<<blocks, 256, 0, s>>>(dL, static_cast<bf16*>(dl3), static_cast<bf16*>(dl2),
                                         c.T, Tp, c.E, goff, G, chunk);
  GemmCall gx{};
  gx.kind = GK_DOWN;
  gx.E = 1;
  gx.rows = c.T;
  gx.A = dl3;
  gx.lda = 3 * c.E;
  gx.B = wr2;
  gx.K = 3 * c.E;
  gx.N = c.d;
  gx.out0 = dxr;
  gx.ld0 = c.d;
  gx.out_f32 = 1;
  gx.status = status;
  cudaError_t err = launch_gemm(gx, s);
  if (err != cudaSuccess) return err;
  GemmCall gw{};
  gw.kind = GK_DW;
  gw.row_offsets = goff;
  gw.E = G;
  gw.rows = 2 * Tp;
  gw.a_rows = c.T;
  gw.a_mod = Tp;
  gw.A = x;
  gw.lda = c.d;
  gw.Mdw = c.d;
  gw.B = dl2;
  gw.N = c.E;
  gw.out0 = part;
  gw.ld0 = c.E;
  gw.out_f32 = 1;
  gw.status = status;
  err = launch_gemm(gw, s);
  if (err != cudaSuccess) return err;
  return launch_sum_splits(part, dWr, n, G, s);
}

}  // namespace moe
